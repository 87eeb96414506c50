/*
 * ORACLE for com.microsoft.PagedAttention over packed variable-length batches.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it. It shares no code with the CUDA implementation.
 *
 * It is the plain definition of the operator, written out with fp64 accumulation:
 *
 *   1. Cache write (com.microsoft.PagedAttention README, "Description" and the
 *      `slot_mapping` row of "Inputs"): every new token's K and V rows are copied into
 *      the cache slot `slot_mapping[i]`, or, when slot_mapping is omitted, into the slot
 *      of its logical position past_seqlens[b] + j, i.e. block_table[b][p / block_size]
 *      * block_size + p % block_size. A slot of -1 suppresses the write.
 *   2. Attention ("Description": the step's K/V are scattered into the cache, then
 *      attended with that history; "block_table remains required because it defines
 *      the read path"): query row j of sequence b and head h attends, causally, the
 *      keys t = 0 .. past_b + j of its sequence, all read from the updated cache
 *      through block_table, with KV head g = h / (num_heads / kv_num_heads):
 *        s_t = scale * <q, k_t>,  scale = attribute, or 1/sqrt(head_size) if it is 0
 *              ("Attributes", `scale`)
 *        o   = sum_t exp(s_t - m) v_t / sum_t exp(s_t - m),  m = max_t s_t
 *        lse = m + ln(sum_t exp(s_t - m))   (natural log, scale included)
 *      then o is rounded once to the 16-bit type (the "downcast at the final write"
 *      of the WS2 CP-Aware Attention Contract, "Reduction Semantics").
 *
 * Readings where the pages leave a step open: bottom-right causal alignment (row j
 * sees keys up to past_b + j, past being the committed length before the call: "Add
 * Qwen3.8 packed hybrid PagedAttention export for ORT GenAI Engine", "Shared inputs"
 * table); GQA groups are contiguous (WS2 CP-Aware Attention Contract, "Qwen3-8B TP=2
 * CP=2 Example": each rank keeps 16 of 32 query heads with 4 of 8 KV heads); packed
 * rows are [Q (nh*hs) | K (kvh*hs) | V (kvh*hs)], head-major inside each part
 * (com.microsoft.PagedAttention README, "Inputs", `query`).
 *
 * Caller errors that the pages leave undefined (a slot out of range, two tokens
 * writing one slot, a block_table entry out of range for an active page) are reported
 * as negative return codes instead of being computed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
  ORACLE_OK = 0,
  ORACLE_BAD_SHAPE = -1,
  ORACLE_BAD_CUM = -2,
  ORACLE_BAD_SLOT = -3,
  ORACLE_DUPLICATE_SLOT = -4,
  ORACLE_BAD_BLOCK = -5,
  ORACLE_NO_MEMORY = -6,
  ORACLE_TOO_LONG = -7,
};

/* ---- 16-bit float formats ------------------------------------------------------- */

static uint64_t dbits(double x) { uint64_t u; memcpy(&u, &x, 8); return u; }

/* IEEE 754 binary16 -> double (exact) */
double oracle_f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1, e = (h >> 10) & 0x1F, m = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)m, -24);                       /* subnormal: m * 2^-24 */
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m | 0x400), e - 25);                 /* 1.m * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16 (the top half of an IEEE binary32) -> double (exact) */
double oracle_bf16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1, e = (h >> 7) & 0xFF, m = h & 0x7F;
  double v;
  if (e == 0) v = ldexp((double)m, -133);                      /* subnormal: m * 2^-133 */
  else if (e == 255) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m | 0x80), e - 134);                 /* 1.m * 2^(e-127) */
  return sign ? -v : v;
}

/* Round a double to a format with `mbits` stored significand bits and exponent bias
 * `bias` (normal exponents 1 .. 2*bias), round to nearest, ties to even, directly from
 * the 53-bit significand (one rounding). */
static uint16_t round_to_small_float(double x, int mbits, int bias, int ebits) {
  uint64_t u = dbits(x);
  uint16_t sign = (uint16_t)((u >> 63) << 15);
  uint16_t inf = (uint16_t)(((1u << ebits) - 1u) << mbits);
  int ef = (int)((u >> 52) & 0x7FF);
  uint64_t frac = u & ((1ULL << 52) - 1);
  if (ef == 0x7FF) return frac ? (uint16_t)(sign | inf | (1u << (mbits - 1))) : (uint16_t)(sign | inf);
  if (ef == 0) return sign; /* double subnormals are far below either format's range */
  int e = ef - 1023;
  if (e > bias) return (uint16_t)(sign | inf);
  uint64_t sig = frac | (1ULL << 52);
  int min_e = 1 - bias;
  int shift = 52 - mbits + (e < min_e ? (min_e - e) : 0);
  if (shift > 60) return sign;
  uint64_t kept = sig >> shift, rem = sig & ((1ULL << shift) - 1), half = 1ULL << (shift - 1);
  if (rem > half || (rem == half && (kept & 1))) kept += 1;
  uint32_t h;
  if (e >= min_e) h = ((uint32_t)(e + bias) << mbits) + (uint32_t)(kept - (1ULL << mbits));
  else h = (uint32_t)kept; /* subnormal, possibly rounded up into the smallest normal */
  if (h >= inf) h = inf;
  return (uint16_t)(sign | h);
}

uint16_t oracle_double_to_f16(double x) { return round_to_small_float(x, 10, 15, 5); }
uint16_t oracle_double_to_bf16(double x) { return round_to_small_float(x, 7, 127, 8); }

/* value table for all 65536 bit patterns of the element type (0 = fp16, 1 = bf16) */
static double* make_table(int dtype) {
  double* t = (double*)malloc(65536 * sizeof(double));
  if (!t) return NULL;
  for (int i = 0; i < 65536; ++i)
    t[i] = dtype == 1 ? oracle_bf16_to_double((uint16_t)i) : oracle_f16_to_double((uint16_t)i);
  return t;
}

/* ---- input checks shared by both steps ----------------------------------------- */

static int check_batch(int32_t N, int32_t B, int32_t nh, int32_t kvh, int32_t hs,
                       int32_t num_blocks, int32_t bs, int32_t max_blocks,
                       const int32_t* cum, const int32_t* past) {
  if (N < 0 || B < 0 || nh <= 0 || kvh <= 0 || hs <= 0 || nh % kvh || num_blocks < 0 || bs <= 0 ||
      max_blocks < 0)
    return ORACLE_BAD_SHAPE;
  if (cum[0] != 0 || cum[B] != N) return ORACLE_BAD_CUM;
  for (int b = 0; b < B; ++b) {
    if (cum[b + 1] < cum[b] || past[b] < 0) return ORACLE_BAD_CUM;
    int64_t kv = (int64_t)past[b] + (cum[b + 1] - cum[b]);
    if ((kv + bs - 1) / bs > max_blocks) return ORACLE_TOO_LONG;
  }
  return ORACLE_OK;
}

/* ---- step 1: cache write -------------------------------------------------------- */

/* The cache slot of every new token (-1: write suppressed), checked: a slot outside the
 * cache, two tokens writing one slot, or a block_table entry outside the pool for a
 * derived slot are errors. */
static int resolve_slots(int32_t B, int32_t num_blocks, int32_t bs, int32_t max_blocks, const int32_t* cum,
                         const int32_t* past, const int32_t* block_table, const int32_t* slot_mapping,
                         int64_t* slots) {
  const int64_t nslots = (int64_t)num_blocks * bs;
  unsigned char* used = (unsigned char*)calloc(nslots > 0 ? (size_t)nslots : 1, 1);
  if (!used) return ORACLE_NO_MEMORY;
  for (int b = 0; b < B; ++b) {
    for (int32_t i = cum[b]; i < cum[b + 1]; ++i) {
      int64_t slot;
      if (slot_mapping) {
        slot = slot_mapping[i];
      } else {
        int64_t p = (int64_t)past[b] + (i - cum[b]);          /* logical position */
        int64_t blk = block_table[(int64_t)b * max_blocks + p / bs];
        if (blk < 0 || blk >= num_blocks) { free(used); return ORACLE_BAD_BLOCK; }
        slot = blk * bs + p % bs;
      }
      slots[i] = slot;
      if (slot == -1) continue;                                 /* write suppressed */
      if (slot < 0 || slot >= nslots) { free(used); return ORACLE_BAD_SLOT; }
      if (used[slot]) { free(used); return ORACLE_DUPLICATE_SLOT; }
      used[slot] = 1;
    }
  }
  free(used);
  return ORACLE_OK;
}

int oracle_scatter(int32_t N, int32_t B, int32_t nh, int32_t kvh, int32_t hs, int32_t num_blocks,
                   int32_t bs, int32_t max_blocks, const uint16_t* query, const uint16_t* key,
                   const uint16_t* value, uint16_t* key_cache, uint16_t* value_cache,
                   const int32_t* cum, const int32_t* past, const int32_t* block_table,
                   const int32_t* slot_mapping) {
  int rc = check_batch(N, B, nh, kvh, hs, num_blocks, bs, max_blocks, cum, past);
  if (rc) return rc;
  const int64_t row = (int64_t)kvh * hs;              /* one token's K (or V) row */
  const int packed = key == NULL;
  const int64_t qw = packed ? (int64_t)(nh + 2 * kvh) * hs : (int64_t)nh * hs;
  int64_t* slots = (int64_t*)malloc((size_t)(N > 0 ? N : 1) * sizeof(int64_t));
  if (!slots) return ORACLE_NO_MEMORY;
  rc = resolve_slots(B, num_blocks, bs, max_blocks, cum, past, block_table, slot_mapping, slots);
  for (int64_t i = 0; i < N && !rc; ++i) {
    const int64_t slot = slots[i];
    if (slot == -1) continue;
    const uint16_t* k_src = packed ? query + i * qw + (int64_t)nh * hs : key + i * row;
    const uint16_t* v_src = packed ? query + i * qw + (int64_t)(nh + kvh) * hs : value + i * row;
    /* cache[slot / bs][slot % bs][:][:] is the contiguous row at flat slot index */
    memcpy(key_cache + slot * row, k_src, (size_t)row * 2);
    memcpy(value_cache + slot * row, v_src, (size_t)row * 2);
  }
  free(slots);
  return rc;
}

/* ---- INT8 / INT4 per-channel KV cache -------------------------------------------------
 * An extension: the Mobius issue ("Add Qwen3.8 packed hybrid PagedAttention export for ORT
 * GenAI Engine", its scope list) asks for an INT8/INT4 per-channel paged KV cache with
 * calibrated scale loading and gives no format. Reading: the caches hold integer codes;
 * K and V each come with a caller-given fp32 scale per (KV head, channel), fixed by
 * calibration; symmetric, no zero point. A value x of T is stored as
 *   code = min(max(rint(fl32(x) / s), -Q), Q),   Q = 127 (INT8) or 7 (INT4),
 * the fp32 quotient correctly rounded, rint rounding half to even (a NaN quotient gives
 * -Q: max(NaN, -Q) is -Q), and attention reads the value code * s, formed in fp64.
 * INT8 codes are bytes, two's complement; INT4 codes are packed two per byte, channel 2i
 * in the low nibble and 2i + 1 in the high nibble, two's complement. Slots, -1, the read
 * path and the attention are the operator's, on those values.
 */
static int quant_code(float x, float s, int qmax) {
  float r = rintf(x / s);
  r = fmaxf(r, (float)-qmax);
  r = fminf(r, (float)qmax);
  return (int)r;
}

/* n rows of kvh * hs values of type T (row i at x + i * x_stride) to code rows: INT8
 * (kind 1) kvh * hs bytes, INT4 (kind 2) kvh * hs / 2 bytes per row. */
int oracle_quantize_rows(int dtype, int kind, int64_t n, int32_t kvh, int32_t hs, const uint16_t* x,
                         int64_t x_stride, const float* scale, uint8_t* codes) {
  if (n < 0 || kvh <= 0 || hs <= 0 || (kind != 1 && kind != 2) || (kind == 2 && hs % 2)) return ORACLE_BAD_SHAPE;
  double* tab = make_table(dtype);
  if (!tab) return ORACLE_NO_MEMORY;
  const int qmax = kind == 1 ? 127 : 7;
  const int64_t rb = kind == 1 ? (int64_t)kvh * hs : (int64_t)kvh * hs / 2;  /* bytes per code row */
  memset(codes, 0, (size_t)(n * rb));
  for (int64_t i = 0; i < n; ++i)
    for (int32_t g = 0; g < kvh; ++g)
      for (int32_t d = 0; d < hs; ++d) {
        const float v = (float)tab[x[i * x_stride + (int64_t)g * hs + d]];  /* exact: T is inside fp32 */
        const int code = quant_code(v, scale[(int64_t)g * hs + d], qmax);
        if (kind == 1) {
          codes[i * rb + (int64_t)g * hs + d] = (uint8_t)(int8_t)code;
        } else {
          uint8_t* byte = codes + i * rb + ((int64_t)g * hs + d) / 2;
          *byte |= (uint8_t)((code & 0x0F) << ((d & 1) ? 4 : 0));
        }
      }
  free(tab);
  return ORACLE_OK;
}

/* The cache write for code caches: the code rows (row_bytes each, token i's K at
 * k_codes + i * row_bytes) copied to their slots. */
int oracle_scatter_codes(int32_t N, int32_t B, int32_t num_blocks, int32_t bs, int32_t max_blocks,
                         int64_t row_bytes, const uint8_t* k_codes, const uint8_t* v_codes, uint8_t* key_cache,
                         uint8_t* value_cache, const int32_t* cum, const int32_t* past, const int32_t* block_table,
                         const int32_t* slot_mapping) {
  if (N < 0 || B < 0 || num_blocks < 0 || bs <= 0 || max_blocks < 0 || row_bytes <= 0) return ORACLE_BAD_SHAPE;
  if (cum[0] != 0 || cum[B] != N) return ORACLE_BAD_CUM;
  for (int b = 0; b < B; ++b) {
    if (cum[b + 1] < cum[b] || past[b] < 0) return ORACLE_BAD_CUM;
    if (((int64_t)past[b] + (cum[b + 1] - cum[b]) + bs - 1) / bs > max_blocks) return ORACLE_TOO_LONG;
  }
  int64_t* slots = (int64_t*)malloc((size_t)(N > 0 ? N : 1) * sizeof(int64_t));
  if (!slots) return ORACLE_NO_MEMORY;
  int rc = resolve_slots(B, num_blocks, bs, max_blocks, cum, past, block_table, slot_mapping, slots);
  for (int64_t i = 0; i < N && !rc; ++i) {
    if (slots[i] == -1) continue;
    memcpy(key_cache + slots[i] * row_bytes, k_codes + i * row_bytes, (size_t)row_bytes);
    memcpy(value_cache + slots[i] * row_bytes, v_codes + i * row_bytes, (size_t)row_bytes);
  }
  free(slots);
  return rc;
}

/* ---- step 2: attention for one (token, head) ----------------------------------- */

/* Where attention reads K or V: a cache of 16-bit values of type T (value table tab), or a
 * cache of integer codes with a per-(KV head, channel) fp32 scale (the quantized caches
 * below; kind 1 = INT8, 2 = INT4). */
typedef struct {
  int kind;
  const uint16_t* bits;  /* kind 0 */
  const double* tab;
  const uint8_t* codes;  /* kinds 1, 2 */
  const float* scale;    /* (kvh, hs) */
} KvView;

/* the INT4 code of channel d in a row of packed codes: channel 2i in the low nibble of
 * byte i, 2i+1 in the high nibble, two's complement */
static int int4_code(const uint8_t* row, int32_t d) {
  int nib = (d & 1) ? row[d / 2] >> 4 : row[d / 2] & 0x0F;
  return nib >= 8 ? nib - 16 : nib;
}

/* the value attention reads for channel d of KV head g in flat cache row `row` */
static double kv_value(const KvView* v, int64_t row, int32_t g, int32_t kvh, int32_t hs, int32_t d) {
  if (v->kind == 0) return v->tab[v->bits[(row * kvh + g) * hs + d]];
  const double s = (double)v->scale[(int64_t)g * hs + d];
  if (v->kind == 1) return (double)(int8_t)v->codes[(row * kvh + g) * hs + d] * s;
  return (double)int4_code(v->codes + (row * kvh + g) * (hs / 2), d) * s;
}

/* Attention of packed query row i (sequence b, position j in it) for head h. rows[t] is
 * the flat cache row of logical key t. Writes hs outputs and the lse. scores is
 * scratch of at least past_b + j + 1 doubles. */
static void attend_one(const double* tab, const uint16_t* query, int64_t qw, int32_t i, int32_t h,
                       int32_t g, int32_t kvh, int32_t hs, int64_t limit, const int64_t* rows,
                       const KvView* kv_k, const KvView* kv_v, double scale, double* scores, double* out,
                       double* lse) {
  const uint16_t* q = query + (int64_t)i * qw + (int64_t)h * hs;
  double m = -INFINITY;
  for (int64_t t = 0; t <= limit; ++t) {
    double dot = 0.0;
    for (int d = 0; d < hs; ++d) dot += tab[q[d]] * kv_value(kv_k, rows[t], g, kvh, hs, d);
    scores[t] = scale * dot;
    if (scores[t] > m) m = scores[t];
  }
  double den = 0.0;
  for (int d = 0; d < hs; ++d) out[d] = 0.0;
  for (int64_t t = 0; t <= limit; ++t) {
    double w = exp(scores[t] - m);
    den += w;
    for (int d = 0; d < hs; ++d) out[d] += w * kv_value(kv_v, rows[t], g, kvh, hs, d);
  }
  for (int d = 0; d < hs; ++d) out[d] /= den;
  *lse = m + log(den);
}

/* flat cache rows of the logical keys 0 .. L-1 of sequence b, through block_table */
static int gather_rows(int32_t b, int64_t L, int32_t bs, int32_t max_blocks, int32_t num_blocks,
                       const int32_t* block_table, int64_t* rows) {
  for (int64_t t = 0; t < L; ++t) {
    int64_t blk = block_table[(int64_t)b * max_blocks + t / bs];
    if (blk < 0 || blk >= num_blocks) return ORACLE_BAD_BLOCK;
    rows[t] = blk * bs + t % bs;
  }
  return ORACLE_OK;
}

static double resolve_scale(float scale, int32_t hs) {
  return scale == 0.0f ? 1.0 / sqrt((double)hs) : (double)scale;
}

/* Attention for every packed row and head, K and V read through the views. out: N x nh x
 * hs doubles; lse: N x nh; out_bits (optional): N x nh x hs 16-bit results rounded once.
 * The caches are the ones after the cache write. nthreads <= 0: the OpenMP default. */
static int attention_all(int dtype, int32_t B, int32_t nh, int32_t kvh, int32_t hs,
                         int32_t num_blocks, int32_t bs, int32_t max_blocks, int32_t query_width,
                         const uint16_t* query, const double* tab, const KvView* kv_k, const KvView* kv_v,
                         const int32_t* cum, const int32_t* past, const int32_t* block_table, float scale,
                         double* out, double* lse, uint16_t* out_bits, int nthreads) {
  const int32_t G = nh / kvh;
  const double sc = resolve_scale(scale, hs);
  int err = ORACLE_OK;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int32_t b = 0; b < B; ++b) {
    for (int32_t h = 0; h < nh; ++h) {
      int32_t q_len = cum[b + 1] - cum[b];
      if (q_len == 0) continue;
      int64_t L = (int64_t)past[b] + q_len;
      int64_t* rows = (int64_t*)malloc((size_t)L * sizeof(int64_t));
      double* scores = (double*)malloc((size_t)L * sizeof(double));
      if (!rows || !scores) {
#pragma omp atomic write
        err = ORACLE_NO_MEMORY;
      } else if (gather_rows(b, L, bs, max_blocks, num_blocks, block_table, rows) != ORACLE_OK) {
#pragma omp atomic write
        err = ORACLE_BAD_BLOCK;
      } else {
        for (int32_t j = 0; j < q_len; ++j) {
          int32_t i = cum[b] + j;
          double* o = out + ((int64_t)i * nh + h) * hs;
          attend_one(tab, query, query_width, i, h, h / G, kvh, hs, (int64_t)past[b] + j, rows, kv_k, kv_v, sc,
                     scores, o, lse + (int64_t)i * nh + h);
          if (out_bits)
            for (int d = 0; d < hs; ++d)
              out_bits[((int64_t)i * nh + h) * hs + d] =
                  dtype == 1 ? oracle_double_to_bf16(o[d]) : oracle_double_to_f16(o[d]);
        }
      }
      free(rows);
      free(scores);
    }
  }
  return err;
}

/* The same attention for a list of (token, head) pairs only: out n_sel x hs, lse n_sel.
 * Lets large workloads be checked on sampled outputs. */
static int attention_sel(int32_t N, int32_t nh, int32_t kvh, int32_t hs, int32_t num_blocks,
                         int32_t bs, int32_t max_blocks, int32_t query_width, const uint16_t* query,
                         const double* tab, const KvView* kv_k, const KvView* kv_v, const int32_t* cum,
                         const int32_t* past, const int32_t* block_table, float scale, int32_t n_sel,
                         const int32_t* sel_token, const int32_t* sel_head, double* out, double* lse, int nthreads) {
  for (int32_t s = 0; s < n_sel; ++s)
    if (sel_token[s] < 0 || sel_token[s] >= N || sel_head[s] < 0 || sel_head[s] >= nh) return ORACLE_BAD_SHAPE;
  const int32_t G = nh / kvh;
  const double sc = resolve_scale(scale, hs);
  int err = ORACLE_OK;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t s = 0; s < n_sel; ++s) {
    int32_t i = sel_token[s], h = sel_head[s];
    int32_t b = 0;
    while (cum[b + 1] <= i) ++b;                    /* the sequence that owns row i */
    int32_t j = i - cum[b];
    int64_t L = (int64_t)past[b] + j + 1;           /* keys this row can see */
    int64_t* rows = (int64_t*)malloc((size_t)L * sizeof(int64_t));
    double* scores = (double*)malloc((size_t)L * sizeof(double));
    if (!rows || !scores) {
#pragma omp atomic write
      err = ORACLE_NO_MEMORY;
    } else if (gather_rows(b, L, bs, max_blocks, num_blocks, block_table, rows) != ORACLE_OK) {
#pragma omp atomic write
      err = ORACLE_BAD_BLOCK;
    } else {
      attend_one(tab, query, query_width, i, h, h / G, kvh, hs, L - 1, rows, kv_k, kv_v, sc, scores,
                 out + (int64_t)s * hs, lse + s);
    }
    free(rows);
    free(scores);
  }
  return err;
}

/* Attention over 16-bit caches of type T (see attention_all). */
int oracle_attention(int dtype, int32_t N, int32_t B, int32_t nh, int32_t kvh, int32_t hs,
                     int32_t num_blocks, int32_t bs, int32_t max_blocks, int32_t query_width,
                     const uint16_t* query, const uint16_t* key_cache, const uint16_t* value_cache,
                     const int32_t* cum, const int32_t* past, const int32_t* block_table, float scale,
                     double* out, double* lse, uint16_t* out_bits, int nthreads) {
  int rc = check_batch(N, B, nh, kvh, hs, num_blocks, bs, max_blocks, cum, past);
  if (rc) return rc;
  double* tab = make_table(dtype);
  if (!tab) return ORACLE_NO_MEMORY;
  const KvView vk = {0, key_cache, tab, NULL, NULL}, vv = {0, value_cache, tab, NULL, NULL};
  rc = attention_all(dtype, B, nh, kvh, hs, num_blocks, bs, max_blocks, query_width, query, tab, &vk, &vv, cum,
                     past, block_table, scale, out, lse, out_bits, nthreads);
  free(tab);
  return rc;
}

int oracle_attention_rows(int dtype, int32_t N, int32_t B, int32_t nh, int32_t kvh, int32_t hs,
                          int32_t num_blocks, int32_t bs, int32_t max_blocks, int32_t query_width,
                          const uint16_t* query, const uint16_t* key_cache,
                          const uint16_t* value_cache, const int32_t* cum, const int32_t* past,
                          const int32_t* block_table, float scale, int32_t n_sel,
                          const int32_t* sel_token, const int32_t* sel_head, double* out,
                          double* lse, int nthreads) {
  int rc = check_batch(N, B, nh, kvh, hs, num_blocks, bs, max_blocks, cum, past);
  if (rc) return rc;
  double* tab = make_table(dtype);
  if (!tab) return ORACLE_NO_MEMORY;
  const KvView vk = {0, key_cache, tab, NULL, NULL}, vv = {0, value_cache, tab, NULL, NULL};
  rc = attention_sel(N, nh, kvh, hs, num_blocks, bs, max_blocks, query_width, query, tab, &vk, &vv, cum, past,
                     block_table, scale, n_sel, sel_token, sel_head, out, lse, nthreads);
  free(tab);
  return rc;
}

/* Attention over code caches (kind 1 INT8, 2 INT4) with their fp32 scales (kvh, hs). */
int oracle_attention_q(int dtype, int kind, int32_t N, int32_t B, int32_t nh, int32_t kvh, int32_t hs,
                       int32_t num_blocks, int32_t bs, int32_t max_blocks, int32_t query_width, const uint16_t* query,
                       const uint8_t* key_codes, const uint8_t* value_codes, const float* k_scale,
                       const float* v_scale, const int32_t* cum, const int32_t* past, const int32_t* block_table,
                       float scale, double* out, double* lse, uint16_t* out_bits, int nthreads) {
  if ((kind != 1 && kind != 2) || (kind == 2 && hs % 2)) return ORACLE_BAD_SHAPE;
  int rc = check_batch(N, B, nh, kvh, hs, num_blocks, bs, max_blocks, cum, past);
  if (rc) return rc;
  double* tab = make_table(dtype);
  if (!tab) return ORACLE_NO_MEMORY;
  const KvView vk = {kind, NULL, NULL, key_codes, k_scale}, vv = {kind, NULL, NULL, value_codes, v_scale};
  rc = attention_all(dtype, B, nh, kvh, hs, num_blocks, bs, max_blocks, query_width, query, tab, &vk, &vv, cum, past,
                     block_table, scale, out, lse, out_bits, nthreads);
  free(tab);
  return rc;
}

int oracle_attention_rows_q(int dtype, int kind, int32_t N, int32_t B, int32_t nh, int32_t kvh, int32_t hs,
                            int32_t num_blocks, int32_t bs, int32_t max_blocks, int32_t query_width,
                            const uint16_t* query, const uint8_t* key_codes, const uint8_t* value_codes,
                            const float* k_scale, const float* v_scale, const int32_t* cum, const int32_t* past,
                            const int32_t* block_table, float scale, int32_t n_sel, const int32_t* sel_token,
                            const int32_t* sel_head, double* out, double* lse, int nthreads) {
  if ((kind != 1 && kind != 2) || (kind == 2 && hs % 2)) return ORACLE_BAD_SHAPE;
  int rc = check_batch(N, B, nh, kvh, hs, num_blocks, bs, max_blocks, cum, past);
  if (rc) return rc;
  double* tab = make_table(dtype);
  if (!tab) return ORACLE_NO_MEMORY;
  const KvView vk = {kind, NULL, NULL, key_codes, k_scale}, vv = {kind, NULL, NULL, value_codes, v_scale};
  rc = attention_sel(N, nh, kvh, hs, num_blocks, bs, max_blocks, query_width, query, tab, &vk, &vv, cum, past,
                     block_table, scale, n_sel, sel_token, sel_head, out, lse, nthreads);
  free(tab);
  return rc;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---- Q/K preparation before the cache write ----------------------------------------
 * Not part of the operator statement: the RMSNorm of each query and key head vector
 * followed by the rotary position embedding, which the Qwen3.8 export issue ("Add Qwen3.8
 * packed hybrid PagedAttention export for ORT GenAI Engine") applies before
 * PagedAttention and which the README ("Description") lists among what the package does
 * not do. For every row i (sequence b, j = i - cum[b], position p = past_b + j) and every
 * head vector x of head_size values:
 *   RMSNorm, when a weight w is given:  x_c <- x_c / sqrt(mean_c x_c^2 + eps) * w_c
 *   rotary embedding, when rotary_dim d > 0, pairing component u with u + d/2
 *   ("rotate half"): for u < d/2
 *     a_u = fl32(fl32(p) * fl32(base^(-2u/d)))
 *     (x_u, x_{u+d/2}) <- (x_u cos a_u - x_{u+d/2} sin a_u, x_{u+d/2} cos a_u + x_u sin a_u)
 *   components from d on are unchanged.
 * Everything is fp64 except the angle a_u: the fp32 product of the position and the
 * fp32 frequency, the way fp32 frameworks form the rotary table (at positions near 1e5
 * the exact angle differs from it by ~1e-2 rad, far more than the rounding of the
 * result). The values are returned unrounded: out_q (N, nh, hs), out_k (N, kvh, hs).
 */
static void prep_vector(const double* x, double* y, int32_t hs, const double* w, double eps, int32_t d,
                        const double* ca, const double* sa) {
  double r = 1.0;
  if (w) {
    double ss = 0.0;
    for (int32_t c = 0; c < hs; ++c) ss += x[c] * x[c];
    r = 1.0 / sqrt(ss / hs + eps);
  }
  for (int32_t c = 0; c < hs; ++c) y[c] = w ? x[c] * r * w[c] : x[c];
  for (int32_t u = 0; u < d / 2; ++u) {
    const double a = y[u], b = y[u + d / 2];
    y[u] = a * ca[u] - b * sa[u];
    y[u + d / 2] = b * ca[u] + a * sa[u];
  }
}

int oracle_qk_prep(int dtype, int32_t N, int32_t B, int32_t nh, int32_t kvh, int32_t hs, int64_t q_width,
                   const uint16_t* query, const uint16_t* key, const int32_t* cum, const int32_t* past,
                   const uint16_t* q_weight, const uint16_t* k_weight, double eps, int32_t rotary_dim, double base,
                   double* out_q, double* out_k) {
  if (N < 0 || B <= 0 || nh <= 0 || kvh <= 0 || hs <= 0 || rotary_dim < 0 || rotary_dim > hs || rotary_dim % 2)
    return ORACLE_BAD_SHAPE;
  if (cum[0] != 0 || cum[B] != N) return ORACLE_BAD_CUM;
  double* tab = make_table(dtype);
  double* wq = malloc(sizeof(double) * hs);
  double* wk = malloc(sizeof(double) * hs);
  if (!tab || !wq || !wk) { free(tab); free(wq); free(wk); return ORACLE_NO_MEMORY; }
  for (int32_t c = 0; c < hs; ++c) {
    if (q_weight) wq[c] = tab[q_weight[c]];
    if (k_weight) wk[c] = tab[k_weight[c]];
  }
  int err = ORACLE_OK;
  for (int32_t b = 0; b < B && !err; ++b) {
    if (cum[b + 1] < cum[b]) err = ORACLE_BAD_CUM;
  }
  if (!err) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int32_t i = 0; i < N; ++i) {
      int32_t lo = 0, hi = B - 1;  /* the last b with cum[b] <= i */
      while (lo < hi) {
        const int32_t mid = (lo + hi + 1) / 2;
        if (cum[mid] <= i) lo = mid; else hi = mid - 1;
      }
      const int64_t pos = (int64_t)past[lo] + (i - cum[lo]);
      double ca[512], sa[512], x[1024];
      for (int32_t u = 0; u < rotary_dim / 2; ++u) {
        const float freq = (float)pow(base, -2.0 * u / rotary_dim);
        const float ang = (float)pos * freq;
        ca[u] = cos((double)ang);
        sa[u] = sin((double)ang);
      }
      const uint16_t* qrow = query + (int64_t)i * q_width;
      const uint16_t* krow = key ? key + (int64_t)i * kvh * hs : qrow + (int64_t)nh * hs;
      for (int32_t h = 0; h < nh; ++h) {
        for (int32_t c = 0; c < hs; ++c) x[c] = tab[qrow[(int64_t)h * hs + c]];
        prep_vector(x, out_q + ((int64_t)i * nh + h) * hs, hs, q_weight ? wq : NULL, eps, rotary_dim, ca, sa);
      }
      for (int32_t g = 0; g < kvh; ++g) {
        for (int32_t c = 0; c < hs; ++c) x[c] = tab[krow[(int64_t)g * hs + c]];
        prep_vector(x, out_k + ((int64_t)i * kvh + g) * hs, hs, k_weight ? wk : NULL, eps, rotary_dim, ca, sa);
      }
    }
  }
  free(tab);
  free(wq);
  free(wk);
  return err;
}

/* n values rounded once to fp16 (dtype 0) or bf16 (dtype 1), round to nearest even */
void oracle_round_array(int dtype, const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = dtype ? oracle_double_to_bf16(x[i]) : oracle_double_to_f16(x[i]);
}

/* ---- output gate --------------------------------------------------------------------------
 * Not part of the operator statement: Qwen3.5's full-attention layers multiply the
 * attention output elementwise by a sigmoid gate ("Add Qwen3.8 packed hybrid PagedAttention
 * export for ORT GenAI Engine": the layer's output is gated by a sigmoid). For every output
 * element, gated = out / (1 + exp(-gate)) in fp64, then rounded once to T. n values. */
int oracle_apply_gate(int dtype, int64_t n, const double* out, const uint16_t* gate, double* gated,
                      uint16_t* bits) {
  double* tab = make_table(dtype);
  if (!tab) return ORACLE_NO_MEMORY;
  for (int64_t i = 0; i < n; ++i) {
    gated[i] = out[i] / (1.0 + exp(-tab[gate[i]]));
    bits[i] = dtype ? oracle_double_to_bf16(gated[i]) : oracle_double_to_f16(gated[i]);
  }
  free(tab);
  return ORACLE_OK;
}
