// Split-KV decode attention and the deterministic (out, lse) merge.
//
// Decode-class sequences have q_len * G <= 16 query rows per KV head, so one work item
// (sequence b, KV head g, key range) holds all of them in a single 16-row MMA tile:
// row r = j * G + hq is query row j of the sequence for query head g * G + hq. The
// operation is memory bound (every K and V element of the history is read once), so the
// kernel is built around streaming pages:
//   - one producer warp brings 64-key K and V tiles of the item into a 3-stage shared
//     memory ring with TMA (a 3-D tensor map over (head_size, kv_heads, slots): one box
//     per page segment, located through block_table; 128-byte swizzle so ldmatrix reads
//     are bank-conflict free);
//   - four consumer warps each take 16 keys of every tile: S = Q K^T and O += P V on the
//     warp-level tensor cores (mma.sync m16n8k16, fp32 accumulation), with an online
//     softmax in registers (row max over the quad by shuffles, base-2 exponentials; for
//     bf16 the weights P enter P V as a bf16 hi + lo pair, two products);
//   - at the end of the item the four warps' (m, l, O) are combined in a fixed order in
//     shared memory (at head_size 256 in two buffers, warps 0 + 2 and 1 + 3, which the
//     writer adds; an item of at most four rows in one round, the four warps' rows side by
//     side, added by the writer in warp order). An item that is its whole unit writes the
//     output row rounded once to T; otherwise the unit's pieces are merged in key order:
//     the (out, lse) reduction of the WS2 CP-Aware Attention Contract, "Reduction
//     Semantics" (fp32, fixed order, downcast at the final write). On the balanced cut the
//     first piece's CTA merges, from its own combine buffer and the others' normalised fp32
//     partial rows and natural-log lse, once their arrival count says they are written;
//     with forced split lengths the last piece to finish merges.
// Integer caches: the codes become fp16 in registers as the tiles are read (three CTAs per
// SM below head_size 256); items of at most 8 rows take the "narrow" form, keys and
// channels as the MMA rows and the query rows as its columns (half the MMAs).
// CTA c processes the items [cta_begin[c], cta_begin[c+1]) that the planner cut so that
// the CTAs finish together (each item counting a fixed cost of a few tiles beside its keys);
// a decode-only batch with the host's bound cuts its own share (the self-planned form).
#include "common.cuh"

namespace pa {

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// combined max and denominator of one row over the four warps' (m, l) (base 2)
__device__ __forceinline__ void row_stats(const float* mw, const float* lw, int row, float& M, float& L) {
  M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, mw[w * kDecRows + row]);
  L = 0.f;
#pragma unroll
  for (int w = 0; w < kDecWarps; ++w) {
    const float m = mw[w * kDecRows + row];
    if (m != -INFINITY) L += lw[w * kDecRows + row] * fast_exp2(m - M);
  }
}

// the record of item it (all zeros from it_end on)
__device__ __forceinline__ DecodeItem load_item(const Args& a, int it, int it_end) {
  if (it >= it_end) return DecodeItem{};
  const int4* p = reinterpret_cast<const int4*>(a.items + it);
  const int4 x = p[0], y = p[1], z = p[2];
  DecodeItem d;
  d.b = x.x; d.g = x.y; d.key_begin = x.z; d.key_end = x.w;
  d.unit_first = y.x; d.n_split = y.y; d.c0 = y.z; d.q_len = y.w;
  d.past = z.x; d.pad[0] = d.pad[1] = d.pad[2] = 0;
  return d;
}

// ---- decode-only batches planned by the decode kernel itself ----
// With derived slots, at most self_max_b(HS) sequences and a host bound proving every sequence
// decode-class, no plan and no cache-write kernel run: each CTA reads the batch description
// into shared memory (cum[0..B], past[0..B), and T[0..B], the first virtual tile of each
// sequence's units), cuts the same balanced partition as the planner (unit (b, g) spans
// V + n_b tiles, V standing for an item's fixed cost, then its n_b key tiles; CTA c owns the
// tiles [floor(c W / P), floor((c + 1) W / P))) and generates its items in order. The new
// K/V rows of a tile are written by the CTA that loads the tile, just before the load.
// meta: [0] R0, [1] R1 (this CTA's tiles), [2] W, [3] first candidate sequence, [4] its
// first candidate head, [5] nonzero for a refused batch, [7] W / P ([6] unused).
struct SelfView {
  int* cum;
  int* past;
  int64_t* T;
  int64_t* meta;
};

template <int HS>
__device__ __forceinline__ SelfView self_view(uint8_t* base) {
  constexpr int MB = self_max_b(HS);
  SelfView v;
  v.T = reinterpret_cast<int64_t*>(base);                // MB + 1
  v.meta = v.T + (MB + 1);                                // 6 (8 reserved)
  v.cum = reinterpret_cast<int*>(v.meta + 8);             // MB + 1
  v.past = v.cum + (MB + 1);                              // MB
  return v;
}

// the CTA whose tile range holds virtual tile t: the largest c with floor(c W / P) <= t, i.e.
// floor(((t + 1) P - 1) / W), below P <= 1024: a float estimate set right by integer steps
__device__ __forceinline__ int self_cta_of(int64_t t, int64_t W, int64_t P) {
  const int64_t n = (t + 1) * P - 1;
  int64_t q = (int64_t)((float)n / (float)W);
  while (q > 0 && q * W > n) --q;
  while ((q + 1) * W <= n) ++q;
  return (int)min(P - 1, q);
}

// floor(c W / P) = c floor(W / P) + floor(c (W mod P) / P), with wq = floor(W / P) given
// (c (W mod P) < P^2 <= 2^20 stays in 32 bits)
__device__ __forceinline__ int64_t self_start(int64_t c, int64_t W, int64_t P, int64_t wq) {
  return c * wq + (int64_t)((uint32_t)c * (uint32_t)(W - wq * P) / (uint32_t)P);
}

// The items of a CTA of a self-planned batch in key order, each with the slot of its partial
// result: 2c for the CTA's first item, 2c + 1 for its other split item (a unit cut across
// CTAs c0 .. c1 leaves its pieces in the slots unit_first, then 2c for the CTAs after c0).
// (The planner's items carry their list index as the slot.)
template <int HS>
struct SelfGen {
  int b, g;  // the next candidate unit (the rest is read from the shared batch view)

  __device__ explicit SelfGen(const SelfView& v) : b((int)v.meta[3]), g((int)v.meta[4]) {}

  __device__ bool next(const Args& a, const SelfView& v, DecodeItem& d, int& slot) {
    const int V = dec_item_cost_tiles(HS, a.kvq);
    const int64_t P = gridDim.x;
    const int* cum = v.cum;
    const int* past = v.past;
    const int64_t* T = v.T;
    const int64_t R0 = v.meta[0], R1 = v.meta[1], W = v.meta[2], wq = v.meta[7];
    while (b < a.B) {
      const int bb = b, gg = g;
      const int q = cum[bb + 1] - cum[bb];
      if (q < 1) {
        ++b;
        g = 0;
        continue;
      }
      const int ps = past[bb], kv = ps + q;
      const int64_t n = ceil_div((int64_t)kv, kDecTile);
      const int64_t span0 = T[bb] + (int64_t)gg * (n + V), ks = span0 + V, ke = ks + n;
      if (ks >= R1) {  // later units start later still
        b = a.B;
        return false;
      }
      if (++g == a.kvh) {
        g = 0;
        ++b;
      }
      if (ke <= R0) continue;
      const int c0 = self_cta_of(ks, W, P), c1 = self_cta_of(ke - 1, W, P);
      d.b = bb;
      d.g = gg;
      d.key_begin = (int)((max(ks, R0) - ks) * kDecTile);
      d.key_end = (int)min((min(ke, R1) - ks) * kDecTile, (int64_t)kv);
      d.unit_first = 2 * c0 + (self_start(c0, W, P, wq) >= span0 ? 0 : 1);
      d.n_split = c1 - c0 + 1;
      d.c0 = cum[bb];
      d.q_len = q;
      d.past = ps;
      d.pad[0] = d.pad[1] = d.pad[2] = 0;
      slot = 2 * (int)blockIdx.x + (R0 >= span0 ? 0 : 1);
      return true;
    }
    return false;
  }
};

// Reads and checks the batch, lays out the units and finds this CTA's range (all threads;
// only the batch description is read, which the previous kernels of the stream never write)
template <int HS>
__device__ void self_plan_prologue(const Args& a, const SelfView& v) {
  const int tid = threadIdx.x, B = a.B;
  const int V = dec_item_cost_tiles(HS, a.kvq);
  for (int b = tid; b <= B; b += blockDim.x) v.cum[b] = a.cum[b];
  for (int b = tid; b < B; b += blockDim.x) v.past[b] = a.past[b];
  __syncthreads();
  if (tid < 32) {  // one warp: each lane sums the spans of self_max_b / 32 sequences, then a scan
    constexpr int PER = self_max_b(HS) / 32;
    int64_t span[PER], sum = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int b = tid * PER + i;
      span[i] = 0;
      if (b < B) {
        const int64_t q = (int64_t)v.cum[b + 1] - v.cum[b], past = v.past[b], kv = past + q;
        if (q < 0 || past < 0 || kv > (int64_t)a.max_blocks * a.bs || (a.max_query_len > 0 && q > a.max_query_len))
          bad = true;
        else if (q >= 1)
          span[i] = (ceil_div(kv, kDecTile) + V) * a.kvh;
      }
      sum += span[i];
    }
    int64_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (tid >= o) incl += y;
    }
    int64_t run = incl - sum;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int b = tid * PER + i;
      if (b < B) v.T[b] = run;
      run += span[i];
    }
    bad = __any_sync(0xffffffffu, bad) || v.cum[0] != 0 || v.cum[B] != a.N;
    if (tid == 31) v.T[B] = incl;
    if (tid == 0) v.meta[5] = bad;
  }
  __syncthreads();
  if (tid == 0) {
    const int64_t W = v.T[B], P = gridDim.x, c = blockIdx.x;
    const int64_t wq = W / P;
    const int64_t R0 = W > 0 ? self_start(c, W, P, wq) : 0, R1 = W > 0 ? self_start(c + 1, W, P, wq) : 0;
    int lo = 0, hi = B - 1;  // the last b with T[b] <= R0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (v.T[mid] <= R0) lo = mid; else hi = mid - 1;
    }
    int g0 = 0;
    const int64_t q = (int64_t)v.cum[lo + 1] - v.cum[lo];
    if (q >= 1) {
      const int64_t n = ceil_div((int64_t)v.past[lo] + q, kDecTile);
      g0 = (int)min((R0 - v.T[lo]) / (n + V), (int64_t)a.kvh - 1);
    }
    v.meta[0] = R0;
    v.meta[1] = R1;
    v.meta[2] = W;
    v.meta[3] = lo;
    v.meta[4] = g0;
    v.meta[7] = wq;
  }
  __syncthreads();
}

// (integer caches) The bias of a query row's scores, in natural-log units. INT8 keys enter
// Q K^T as the fp16 integers code + 1152, INT4 keys as the fp16 subnormals (code + 8) 2^-24
// (the row constant takes the 2^-24 back), which adds 1152 (or 8) sum_c Q'_c to every score
// of the row: the softmax, the four warps' combine and the split merge only compare scores
// and lse of one row and do not see it; the exported lse has it taken off. Eight threads per
// row (t & 7), each summing HS / 8 values of the scaled query row; all 32 lanes take part.
template <int HS, int KQ>
__device__ __forceinline__ float key_row_bias(const Args& a, int tok, int head, int t, bool valid) {
  float s = 0.f;
  int e = 0;
  if (valid) {
    const int64_t row = (int64_t)tok * a.nh + head;
    const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.query) + row * HS +
                                                    (t & 7) * (HS / 8));
#pragma unroll
    for (int i = 0; i < HS / 64; ++i) {
      const uint4 w = __ldg(q + i);
      const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        s += __half2float(__ushort_as_half((unsigned short)(x[j] & 0xFFFFu))) +
             __half2float(__ushort_as_half((unsigned short)(x[j] >> 16)));
    }
    e = __ldg(a.qexp + row);
  }
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  s += __shfl_xor_sync(0xffffffffu, s, 4);
  return (KQ == 1 ? 1152.f : 8.f) * s * ldexpf(a.scale_log2, e) * 0.69314718055994531f;
}

// A V code from the normalised P V of integer caches: the conversion's offset taken off
// (INT8: code + 1152; INT4: (code + 8) 2^-24)
template <int KQ>
__device__ __forceinline__ float v_code_value(float x) {
  if constexpr (KQ == 1) return x - 1152.f;
  else if constexpr (KQ == 2) return x * 0x1p24f - 8.f;
  else return x;
}

// the partial-result slot of piece s2 of an item's unit
template <bool SELF>
__device__ __forceinline__ int piece_slot(const DecodeItem& d, int s2) {
  return !SELF ? d.unit_first + s2 : s2 == 0 ? d.unit_first : 2 * ((d.unit_first >> 1) + s2);
}

// This call's K and V rows among the keys [k0, k0 + 64) of an item of a self-planned batch,
// copied from the inputs into the caches (head item.g) by the producer warp before it loads
// the tile: each new key of head g is read only by the CTA whose range holds its tile. An
// out-of-range block is skipped (the tile load reads it as zeros and flags it).
template <int HS>
__device__ __forceinline__ void write_new_rows(const Args& a, const DecodeItem& item, int k0, int lane) {
  const int kv_len = item.past + item.q_len;
  const int n0 = max(k0, max(item.key_begin, item.past));
  const int n1 = min(k0 + kDecTile, min(item.key_end, kv_len));
  if (n1 <= n0) return;
  constexpr int CH = HS / 8;             // 16-byte chunks of one head's row
  const int total = (n1 - n0) * 2 * CH;  // K and V chunks
  const int* bt = a.block_table + (int64_t)item.b * a.max_blocks;
  for (int i0 = 0; i0 < total; i0 += 4 * 32) {  // four chunks per lane in flight
    uint4 v[4];
    uint4* dst[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = i0 + lane + 32 * r;
      dst[r] = nullptr;
      if (i < total) {
        const int rr = i / (2 * CH), rem = i % (2 * CH), which = rem / CH, ch = rem % CH;
        const int key = n0 + rr;
        const int blk = bt[key / a.bs];
        if (blk >= 0 && blk < a.num_blocks) {
          const int64_t tok = item.c0 + (key - item.past);
          const uint16_t* src =
              a.packed ? reinterpret_cast<const uint16_t*>(a.query) + tok * a.q_stride + (which ? a.v_offset : a.k_offset)
                       : reinterpret_cast<const uint16_t*>(which ? a.value : a.key) + tok * a.kv_row;
          v[r] = __ldg(reinterpret_cast<const uint4*>(src + item.g * HS) + ch);
          dst[r] = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(which ? a.value_cache : a.key_cache) +
                                            ((int64_t)blk * a.bs + key % a.bs) * a.kv_row + item.g * HS) + ch;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
      if (dst[r]) *dst[r] = v[r];
  }
  fence_proxy_async_global();  // the rows, seen by the tile's TMA load
  __syncwarp();
}

// Q fragments of an item (A operand, row-major 16 x HS, row r = j * G + hq), straight from
// global memory; rows past the item's q_len * G are zeros
template <int HS>
__device__ __forceinline__ void load_q(const Args& a, const DecodeItem& item, int r0, int r1, int tq,
                                       uint32_t (&qa)[HS / 16][4]) {
  const int n_rows = item.q_len * a.G;
  const uint16_t* q = reinterpret_cast<const uint16_t*>(a.query);
  const uint16_t* p0 = nullptr;
  const uint16_t* p1 = nullptr;
  if (r0 < n_rows)
    p0 = q + (int64_t)(item.c0 + r0 / a.G) * a.q_stride + (int64_t)(item.g * a.G + r0 % a.G) * HS + tq * 2;
  if (r1 < n_rows)
    p1 = q + (int64_t)(item.c0 + r1 / a.G) * a.q_stride + (int64_t)(item.g * a.G + r1 % a.G) * HS + tq * 2;
#pragma unroll
  for (int ks = 0; ks < HS / 16; ++ks) {
    qa[ks][0] = p0 ? __ldg(reinterpret_cast<const uint32_t*>(p0 + ks * 16)) : 0u;
    qa[ks][2] = p0 ? __ldg(reinterpret_cast<const uint32_t*>(p0 + ks * 16 + 8)) : 0u;
    qa[ks][1] = p1 ? __ldg(reinterpret_cast<const uint32_t*>(p1 + ks * 16)) : 0u;
    qa[ks][3] = p1 ? __ldg(reinterpret_cast<const uint32_t*>(p1 + ks * 16 + 8)) : 0u;
  }
}

// ---- integer caches ------------------------------------------------------------------------
// Tiles of code rows (P bytes per row in a box, 64 rows per box; 128-byte swizzle for
// P = 128, 64-byte swizzle for P = 64): the shared address of byte b of row r.
template <int P>
__device__ __forceinline__ uint32_t code_addr(uint32_t base, int r, int b) {
  const int box = b / P, wb = b % P, c = wb >> 4;
  const int cs = P == 128 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3));
  return base + box * (kDecTile * P) + r * P + (cs << 4) + (wb & 15);
}
// R bytes (16 or 8) of shared memory as R / 4 words
template <int R>
__device__ __forceinline__ void lds_run(uint32_t addr, uint32_t (&w)[R / 4]) {
  if constexpr (R == 16)
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
  else
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "r"(addr));
}

// The channel order of the MMA operands on integer caches (Q K^T sums over channels and
// P V keeps each channel's column apart, so any fixed assignment works when Q and the
// output follow it), chosen so that each thread reads its codes of a key row as one run of
// 16 (or 8) bytes, conflict-free in the swizzled tiles at head_size 128:
//  - Q K^T: thread tq owns channels [HS/4 tq, HS/4 (tq + 1)) of a key row. INT8: k-step ks
//    takes the 32-bit word ks of them, channels HS/4 tq + 4ks + {0, 1} as b0 (k = 2tq,
//    2tq+1) and + {2, 3} as b1 (k = 2tq+8, 2tq+9). INT4: word i holds channels
//    HS/4 tq + 8i .. + 7 for the k-steps 2i (channels +0/+4 as b0, +1/+5 as b1) and 2i + 1
//    (+2/+6, +3/+7).
//  - P V: n-tile d column n is channel out_channel(d, n); thread gq (column gq of every
//    n-tile) reads G consecutive INT8 channels per G n-tiles (one 128-byte box each), or
//    its HS/8 consecutive INT4 channels.
template <int HS, int KQ>
__device__ __forceinline__ int out_channel(int d, int n) {
  if constexpr (KQ == 1) {
    constexpr int G = HS / 8 < 16 ? HS / 8 : 16;
    return (d / G) * (8 * G) + G * n + d % G;
  } else {
    return (HS / 8) * n + d;
  }
}

// Q' fragments (the scaled query rows, fp16, in the channel order above) of an item and the
// softmax constants of its two rows: scale * log2(e) * 2^E (E the row's exponent). Without
// LOAD_Q only the constants.
template <int HS, int KQ, bool LOAD_Q = true>
__device__ __forceinline__ void load_q_int(const Args& a, const DecodeItem& item, int r0, int r1, int tq,
                                           uint32_t (&qa)[HS / 16][4], float& c0, float& c1) {
  const int n_rows = item.q_len * a.G;
  const uint16_t* q = reinterpret_cast<const uint16_t*>(a.query);
  const uint16_t* p[2] = {nullptr, nullptr};
  int ex[2] = {0, 0};
  const int rr[2] = {r0, r1};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (rr[i] < n_rows) {
      const int64_t row = (int64_t)(item.c0 + rr[i] / a.G) * a.nh + item.g * a.G + rr[i] % a.G;
      p[i] = q + row * HS;
      ex[i] = __ldg(a.qexp + row);
    }
  }
  constexpr int kSub = KQ == 2 ? 24 : 0;  // (INT4 keys as subnormals: 2^-24 per code unit)
  c0 = ldexpf(a.scale_log2, ex[0] + kSub);
  c1 = ldexpf(a.scale_log2, ex[1] + kSub);
  if constexpr (LOAD_Q) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if constexpr (KQ == 1) {
#pragma unroll
        for (int ks = 0; ks < HS / 16; ++ks) {
          const uint2 v =
              p[i] ? __ldg(reinterpret_cast<const uint2*>(p[i] + (HS / 4) * tq + 4 * ks)) : make_uint2(0, 0);
          qa[ks][i] = v.x;
          qa[ks][2 + i] = v.y;
        }
      } else {
#pragma unroll
        for (int k2 = 0; k2 < HS / 32; ++k2) {
          const uint4 v =
              p[i] ? __ldg(reinterpret_cast<const uint4*>(p[i] + (HS / 4) * tq + 8 * k2)) : make_uint4(0, 0, 0, 0);
          qa[2 * k2][i] = prmt(v.x, v.z, 0x5410u);
          qa[2 * k2][2 + i] = prmt(v.x, v.z, 0x7632u);
          qa[2 * k2 + 1][i] = prmt(v.y, v.w, 0x5410u);
          qa[2 * k2 + 1][2 + i] = prmt(v.y, v.w, 0x7632u);
        }
      }
    }
  }
}

// Items of at most 8 query rows on integer caches ("narrow"): S^T = K Q'^T and
// O^T += V^T P^T, keys and channels as the MMA rows (M = 16), the query rows as its columns
// (N = 8), half the MMAs of the row-major form. Q' is the B operand: k-step ks of row gq is
// the pair of words of q_frags_int's channel order (INT8: channels HS/4 tq + 4 ks .. + 3;
// INT4: the two pairs its prmt forms). Also the softmax constants of the thread's rows ra, rb.
template <int HS, int KQ>
__device__ __forceinline__ void load_q_narrow(const Args& a, const DecodeItem& item, int gq, int ra, int rb,
                                              int tq, uint32_t (&qb)[HS / 16][2], float& c0, float& c1) {
  const int n_rows = item.q_len * a.G;
  const uint16_t* q = reinterpret_cast<const uint16_t*>(a.query);
  auto qrow = [&](int r) { return (int64_t)(item.c0 + r / a.G) * a.nh + item.g * a.G + r % a.G; };
  constexpr int kSub = KQ == 2 ? 24 : 0;  // (INT4 keys as subnormals: 2^-24 per code unit)
  c0 = ldexpf(a.scale_log2, (ra < n_rows ? __ldg(a.qexp + qrow(ra)) : 0) + kSub);
  c1 = ldexpf(a.scale_log2, (rb < n_rows ? __ldg(a.qexp + qrow(rb)) : 0) + kSub);
  const uint16_t* p = gq < n_rows ? q + qrow(gq) * HS : nullptr;
  if constexpr (KQ == 1) {
#pragma unroll
    for (int ks = 0; ks < HS / 16; ++ks) {
      const uint2 v = p ? __ldg(reinterpret_cast<const uint2*>(p + (HS / 4) * tq + 4 * ks)) : make_uint2(0, 0);
      qb[ks][0] = v.x;
      qb[ks][1] = v.y;
    }
  } else {
#pragma unroll
    for (int k2 = 0; k2 < HS / 32; ++k2) {
      const uint4 v =
          p ? __ldg(reinterpret_cast<const uint4*>(p + (HS / 4) * tq + 8 * k2)) : make_uint4(0, 0, 0, 0);
      qb[2 * k2][0] = prmt(v.x, v.z, 0x5410u);
      qb[2 * k2][1] = prmt(v.x, v.z, 0x7632u);
      qb[2 * k2 + 1][0] = prmt(v.y, v.w, 0x5410u);
      qb[2 * k2 + 1][1] = prmt(v.y, v.w, 0x7632u);
    }
  }
}

template <int HS, bool BF16, int KQ, bool SELF, bool NARROW>
__global__ void __launch_bounds__(160, dec_ctas_per_sm(HS, KQ))
    decode_kernel(const Args a, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const int seg_rows) {
  using L = DecSmem<HS, KQ, SELF>;
  static_assert(!NARROW || KQ != 0, "the narrow form is built for integer caches");
  constexpr int NKS = HS / 16;  // k-steps of Q K^T
  constexpr int P = L::kBoxBytes;
  constexpr int ND = HS / 8;    // n-tiles of P V
  constexpr int kCombStride = L::kCombStride;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  float* comb = reinterpret_cast<float*>(smem + L::kComb);
  uint4* qsm = reinterpret_cast<uint4*>(smem + L::kQ);  // (integer caches at three CTAs per SM)
  float* mw = reinterpret_cast<float*>(smem + L::kMw);
  float* lw = reinterpret_cast<float*>(smem + L::kLw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* empty = full + L::kStages;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);
  volatile int* s_last = reinterpret_cast<volatile int*>(smem + L::kAbort + 4);
  uint32_t* err = &a.hdr->error;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecWarps);
    }
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // the work lists and caches written by the earlier kernels of this call. Launched after
  // this call's prefill kernel, which starts its dependents only once its own wait for
  // those kernels has returned, the kernel runs beside the prefill (on the SMs the planner
  // took from it) and waits for it only before exiting, so that the next call still finds
  // both finished.
  const bool beside_prefill = a.dec_after_prefill != 0;
  // a self-planned batch: the partition is cut before the wait (the kernel before this one
  // releases it only once all earlier work of the stream is done, and only the batch
  // description is read); the wait is then for the reset of the merge counters
  constexpr bool self = SELF;
  const SelfView sv = self_view<HS>(smem + L::kSelf);
  if constexpr (SELF) self_plan_prologue<HS>(a, sv);
  if (!beside_prefill) pdl_wait();
  pdl_launch_dependents();
  if (self ? sv.meta[5] != 0 : !a.hdr->valid) {  // a refused batch: nothing is written
    if (self && blockIdx.x == 0 && threadIdx.x == 0) {
      atomicOr(err, PA_DEVERR_BAD_BATCH);
      a.hdr->valid = 0;
    }
    if (beside_prefill) pdl_wait();
    return;
  }
  // the planner's items [it_begin, it_end), or (self-planned) the generator's until it ends
  const int it_begin = self ? 0 : a.cta_begin[blockIdx.x];
  const int it_end = self ? 0 : a.cta_begin[blockIdx.x + 1];

  if (warp == kDecWarps) {
    // ================= producer warp: TMA page loads =================
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    const int nseg = kDecTile / seg_rows;
    const int oob = a.num_blocks * a.bs;  // a row coordinate past the end: TMA fills zeros
    uint32_t cnt = 0;
    SelfGen<HS> gen(sv);  // (self-planned batches)
    int next_slot = 0;
    DecodeItem next;
    bool more;
    if constexpr (SELF) more = gen.next(a, sv, next, next_slot);
    else more = it_begin < it_end, next = load_item(a, it_begin, it_end);
    for (int it = it_begin; more; ++it) {
      const DecodeItem item = next;  // loaded one item ahead
      if constexpr (SELF) {
        more = gen.next(a, sv, next, next_slot);
      } else {
        more = it + 1 < it_end;
        next = load_item(a, it + 1, it_end);
      }
      {
        // this item's query rows into L2: the producer runs a ring's depth of tiles ahead
        // of the consumers, so their Q loads at the item's start find the rows there
        // (q_len tokens x G heads x HS contiguous values each)
        constexpr int kLine = 128;
        const int lines = a.G * HS * 2 / kLine;
        const char* q0 = reinterpret_cast<const char*>(a.query) +
                         ((int64_t)item.c0 * a.q_stride + (int64_t)item.g * a.G * HS) * 2;
        for (int i = lane; i < item.q_len * lines; i += 32)
          prefetch_l2(q0 + (int64_t)(i / lines) * a.q_stride * 2 + (i % lines) * kLine);
      }
      const int kv_len = item.past + item.q_len;
      const int* bt = a.block_table + (int64_t)item.b * a.max_blocks;
      for (int k0 = item.key_begin; k0 < item.key_end; k0 += kDecTile, ++cnt) {
        const int s = cnt % L::kStages;
        const uint32_t ph = (cnt / L::kStages) & 1;
        if constexpr (SELF && KQ == 0) {
          if (a.self_write_rows) write_new_rows<HS>(a, item, k0, lane);
        }
        if (lane == 0) {
          mbar_wait(&empty[s], ph ^ 1, abort, err);
          mbar_arrive_expect_tx(&full[s], L::kStageBytes);
        }
        __syncwarp();
        if (lane < nseg) {
          if constexpr (SELF && KQ == 0) {
            if (a.self_write_rows) fence_proxy_async_global();  // (the rows written above, before the load)
          }
          const int key = k0 + lane * seg_rows;
          int z = oob;
          if (key < kv_len) {
            const int blk = bt[key / a.bs];
            if (blk >= 0 && blk < a.num_blocks) z = blk * a.bs + key % a.bs;
            else atomicOr(err, PA_DEVERR_BAD_BLOCK);
          }
          uint8_t* kdst = smem + s * L::kStageBytes + lane * seg_rows * P;
          constexpr int kBoxX = KQ == 0 ? P / 2 : P;  // box width in map elements
#pragma unroll
          for (int h = 0; h < L::kBoxes; ++h) {
            tma_load_3d(kdst + h * kDecTile * P, &tmK, &full[s], h * kBoxX, item.g, z);
            tma_load_3d(kdst + L::kTileBytes + h * kDecTile * P, &tmV, &full[s], h * kBoxX, item.g, z);
          }
        }
        __syncwarp();
      }
    }
    return;
  }

  // ================= consumer warps =================
  const int w = warp;
  const int tq = lane & 3, gq = lane >> 2;  // quad position, row within the 8-row group
  const int r0 = gq, r1 = gq + 8;           // the two rows this thread holds in MMA fragments
  int stage = 0;  // ring slot and phase of the next tile
  uint32_t phase = 0;
  // integer caches: this thread's byte offsets inside a stage's K tile (its runs of key row
  // 16w + gq; row + 8 has the same swizzle, 8 rows further) and V tile (its runs of key rows
  // 16w + 2tq and 16w + 2tq + 1; rows + 8 likewise)
  constexpr int KRUN = KQ == 1 ? HS / 4 : HS / 8;             // bytes of a K run
  constexpr int VG = KQ == 1 ? (HS / 8 < 16 ? HS / 8 : 16) : HS / 16;  // bytes of a V run
  constexpr int NVR = KQ == 1 ? (HS / 8) / VG : 1;           // V runs per key row
  uint32_t koff[KQ == 0 ? 1 : KRUN / 16], voff[2][NVR];
  if constexpr (KQ != 0) {
#pragma unroll
    for (int j = 0; j < KRUN / 16; ++j) koff[j] = code_addr<P>(0, 16 * w + gq, KRUN * tq + 16 * j);
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int D = 0; D < NVR; ++D)
        voff[e][D] = code_addr<P>(0, 16 * w + 2 * tq + e, KQ == 1 ? D * 8 * VG + VG * gq : VG * gq);
  }
  SelfGen<HS> gen(sv);  // (self-planned batches)
  int next_slot = 0;
  DecodeItem next;
  bool more;
  if constexpr (SELF) more = gen.next(a, sv, next, next_slot);
  else more = it_begin < it_end, next = load_item(a, it_begin, it_end);
  for (int it_i = it_begin; more; ++it_i) {
    const DecodeItem item = next;  // loaded one item ahead
    const int it = SELF ? next_slot : it_i;  // the slot of this item's partial result
    if constexpr (SELF) {
      more = gen.next(a, sv, next, next_slot);
    } else {
      more = it_i + 1 < it_end;
      next = load_item(a, it_i + 1, it_end);
    }
    const int c0 = item.c0, q_len = item.q_len, past = item.past;
    const int n_rows = q_len * a.G;
    uint32_t qa[NKS][4];
    uint32_t qb[NARROW ? NKS : 1][2];  // (narrow items)
    float cr0 = a.scale_log2, cr1 = a.scale_log2;  // the two rows' softmax constants
    // the thread's two rows: r0, r1 (row-major form), or 2tq, 2tq + 1 (narrow: columns of S^T)
    const int ra = NARROW ? 2 * tq : r0, rb = NARROW ? 2 * tq + 1 : r1;
    if constexpr (KQ == 0) {
      load_q<HS>(a, item, r0, r1, tq, qa);
    } else if constexpr (NARROW) {
      load_q_narrow<HS, KQ>(a, item, gq, ra, rb, tq, qb, cr0, cr1);
    } else if constexpr (L::kQSmem) {
      // the four warps' fragments are the same: warp 0 loads them into shared memory (the
      // last item's were read before the barrier that closed its key loop)
      if (w == 0) {
        load_q_int<HS, KQ>(a, item, r0, r1, tq, qa, cr0, cr1);
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) qsm[ks * 32 + lane] = make_uint4(qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
      } else {
        load_q_int<HS, KQ, false>(a, item, r0, r1, tq, qa, cr0, cr1);
      }
      consumer_bar();
    } else {
      load_q_int<HS, KQ>(a, item, r0, r1, tq, qa, cr0, cr1);
    }
    // k-step ks of Q' (integer caches)
    auto qfrag = [&](int ks, uint32_t (&f)[4]) {
      if constexpr (L::kQSmem) {
        const uint4 v = qsm[ks * 32 + lane];
        f[0] = v.x, f[1] = v.y, f[2] = v.z, f[3] = v.w;
      } else if constexpr (!NARROW) {
        f[0] = qa[ks][0], f[1] = qa[ks][1], f[2] = qa[ks][2], f[3] = qa[ks][3];
      }
    };
    // causal limits (inclusive) of the two rows; padding rows borrow the last row's
    const int lim0 = past + min(ra / a.G, q_len - 1);
    const int lim1 = past + min(rb / a.G, q_len - 1);

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    constexpr int NO = NARROW ? ND / 2 : ND;  // accumulator tiles: O (16 x 8) or O^T (16 x 8)
    float o[NO][4];
#pragma unroll
    for (int d = 0; d < NO; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;

    for (int k0 = item.key_begin; k0 < item.key_end; k0 += kDecTile) {
      const int s = stage;
      mbar_wait(&full[s], phase, abort, err);
      const int kw = k0 + 16 * w;  // first key of this warp's 16
      if (kw < item.key_end) {
        const uint32_t kb = smem_u32(smem + s * L::kStageBytes);
        const uint32_t vb = kb + L::kTileBytes;
        if constexpr (NARROW) {
          // ---- S^T (16 keys x 8 rows) = K Q'^T: this thread's keys kw + gq, kw + gq + 8 and
          // rows ra, rb; even and odd k-steps in two accumulator chains ----
          float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (KQ == 1) {
#pragma unroll
            for (int j = 0; j < NKS / 4; ++j) {
              uint32_t u[4], v[4];
              lds_run<16>(kb + koff[j], u);          // key row 16w + gq
              lds_run<16>(kb + koff[j] + 8 * P, v);  // key row 16w + gq + 8
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t A[4];
                s8x4_to_f16_biased(u[i], A[0], A[2]);
                s8x4_to_f16_biased(v[i], A[1], A[3]);
                mma16816<false>((i & 1) ? sb : sa, A, qb[4 * j + i][0], qb[4 * j + i][1]);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < NKS / 8; ++j) {
              uint32_t u[4], v[4];
              lds_run<16>(kb + koff[j], u);
              lds_run<16>(kb + koff[j] + 8 * P, v);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int k2 = 4 * j + i;
                uint32_t uu[4], vv[4];
                s4x8_to_f16_sub(u[i], uu);
                s4x8_to_f16_sub(v[i], vv);
                const uint32_t A0[4] = {uu[0], vv[0], uu[1], vv[1]}, A1[4] = {uu[2], vv[2], uu[3], vv[3]};
                mma16816<false>(sa, A0, qb[2 * k2][0], qb[2 * k2][1]);
                mma16816<false>(sb, A1, qb[2 * k2 + 1][0], qb[2 * k2 + 1][1]);
              }
            }
          }
          // ---- online softmax (base 2): x[e] is key kw + gq + 8 (e >> 1), row (e & 1 ? rb : ra) ----
          const bool ragged = (k0 + kDecTile > item.key_end) || (k0 + kDecTile - 1 > past);
          float x[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float v = (sa[e] + sb[e]) * ((e & 1) ? cr1 : cr0);
            if (ragged) {
              const int key = kw + gq + 8 * (e >> 1);
              if (key >= item.key_end || key > ((e & 1) ? lim1 : lim0)) v = -INFINITY;
            }
            x[e] = v;
          }
#ifdef PA_COVERAGE
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = kw + gq + 8 * (e >> 1), r = (e & 1) ? rb : ra;
            const bool in = !(ragged && (key >= item.key_end || key > ((e & 1) ? lim1 : lim0)));
            if (in && r < n_rows) cov_count(a, c0 + r / a.G, item.g * a.G + r % a.G, key);
          }
#endif
          // the rows' maxima over the warp's 16 keys: the lanes of one tq hold them
          float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
          }
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
          const float ms0 = mn0 == -INFINITY ? 0.f : mn0;  // a row with no key yet stays empty
          const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
          const float al0 = fast_exp2(m0 - ms0), al1 = fast_exp2(m1 - ms1);
          m0 = mn0;
          m1 = mn1;
          // P^T of keys gq and gq + 8, each an fp16 pair (row ra, row rb)
          const uint32_t h0 = pack2<false>(fast_exp2(x[0] - ms0), fast_exp2(x[1] - ms1));
          const uint32_t h1 = pack2<false>(fast_exp2(x[2] - ms0), fast_exp2(x[3] - ms1));
          // the row sums add the fp16 weights the MMA multiplies (see the integer-cache note below)
          const float2 q0 = __half22float2(*reinterpret_cast<const __half2*>(&h0));
          const float2 q1 = __half22float2(*reinterpret_cast<const __half2*>(&h1));
          l0 = l0 * al0 + (q0.x + q1.x);
          l1 = l1 * al1 + (q0.y + q1.y);
          if (!__all_sync(0xffffffffu, al0 == 1.f && al1 == 1.f)) {  // (no row's max grew: O stays)
#pragma unroll
            for (int d = 0; d < NO; ++d) {
              o[d][0] *= al0;
              o[d][1] *= al1;
              o[d][2] *= al0;
              o[d][3] *= al1;
            }
          }
          // ---- O^T (16 channels x 8 rows per tile) += V^T P^T: the B operand is P (rows x
          // keys), the two 8 x 8 blocks of P^T transposed; the A operand pairs the channel
          // columns d, d + 1 of the row-major form (rows gq and gq + 8 of O^T tile d / 2) ----
          const uint32_t pb0 = movmatrix_trans(h0), pb1 = movmatrix_trans(h1);
          if constexpr (KQ == 1) {
            constexpr int G = VG;
#pragma unroll
            for (int D = 0; D < ND / G; ++D) {
              uint32_t w0[G / 4], w1[G / 4], w8[G / 4], w9[G / 4];
              lds_run<G>(vb + voff[0][D], w0);
              lds_run<G>(vb + voff[1][D], w1);
              lds_run<G>(vb + voff[0][D] + 8 * P, w8);
              lds_run<G>(vb + voff[1][D] + 8 * P, w9);
#pragma unroll
              for (int i = 0; i < G / 4; ++i) {
                uint32_t lo[4], hi[4];
                s8_key_pairs_biased(w0[i], w1[i], lo);
                s8_key_pairs_biased(w8[i], w9[i], hi);
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                  const uint32_t A[4] = {lo[e], lo[e + 1], hi[e], hi[e + 1]};
                  mma16816<false>(o[(D * G + 4 * i + e) / 2], A, pb0, pb1);
                }
              }
            }
          } else {
            constexpr int R = VG;
            uint32_t w0[R / 4], w1[R / 4], w8[R / 4], w9[R / 4];
            lds_run<R>(vb + voff[0][0], w0);
            lds_run<R>(vb + voff[1][0], w1);
            lds_run<R>(vb + voff[0][0] + 8 * P, w8);
            lds_run<R>(vb + voff[1][0] + 8 * P, w9);
#pragma unroll
            for (int i = 0; i < R / 4; ++i) {
              uint32_t lo[8], hi[8];
              s4_key_pairs_sub(w0[i], w1[i], lo);
              s4_key_pairs_sub(w8[i], w9[i], hi);
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                const uint32_t A[4] = {lo[e], lo[e + 1], hi[e], hi[e + 1]};
                mma16816<false>(o[(8 * i + e) / 2], A, pb0, pb1);
              }
            }
          }
        } else {
          // ---- S (16 x 16) = Q K^T ----
          float sc[2][4];
  #pragma unroll
          for (int n = 0; n < 2; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
          if constexpr (KQ == 0) {
            const int mi = lane >> 3, rr = lane & 7;
            const int kr = 16 * w + (mi >> 1) * 8 + rr;  // key row inside the tile
  #pragma unroll
            for (int ks = 0; ks < NKS; ++ks) {
              const int c = 2 * ks + (mi & 1);             // 16-byte chunk along head_size
              const uint32_t addr = kb + (c >> 3) * (kDecTile * 128) + kr * 128 + (((c & 7) ^ (kr & 7)) << 4);
              uint32_t b0, b1, b2, b3;
              ldsm_x4(addr, b0, b1, b2, b3);
              mma16816<BF16>(sc[0], qa[ks], b0, b1);
              mma16816<BF16>(sc[1], qa[ks], b2, b3);
            }
          } else if constexpr (KQ == 1) {
  #pragma unroll
            for (int j = 0; j < NKS / 4; ++j) {  // 16 bytes of each row: 4 k-steps
              uint32_t u[4], v[4];
              lds_run<16>(kb + koff[j], u);           // key row 16w + gq
              lds_run<16>(kb + koff[j] + 8 * P, v);   // key row 16w + gq + 8
  #pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t b0, b1, b2, b3, f[4];
                s8x4_to_f16_biased(u[i], b0, b1);
                s8x4_to_f16_biased(v[i], b2, b3);
                qfrag(4 * j + i, f);
                mma16816<false>(sc[0], f, b0, b1);
                mma16816<false>(sc[1], f, b2, b3);
              }
            }
          } else {
  #pragma unroll
            for (int j = 0; j < NKS / 8; ++j) {  // 16 bytes of each row: 8 k-steps
              uint32_t u[4], v[4];
              lds_run<16>(kb + koff[j], u);
              lds_run<16>(kb + koff[j] + 8 * P, v);
  #pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int k2 = 4 * j + i;
                uint32_t uu[4], vv[4], f0[4], f1[4];
                s4x8_to_f16_sub(u[i], uu);
                s4x8_to_f16_sub(v[i], vv);
                qfrag(2 * k2, f0);
                qfrag(2 * k2 + 1, f1);
                mma16816<false>(sc[0], f0, uu[0], uu[1]);
                mma16816<false>(sc[0], f1, uu[2], uu[3]);
                mma16816<false>(sc[1], f0, vv[0], vv[1]);
                mma16816<false>(sc[1], f1, vv[2], vv[3]);
              }
            }
          }
          // ---- online softmax (base 2) ----
          const bool ragged = (k0 + kDecTile > item.key_end) || (k0 + kDecTile - 1 > past);
          float x[2][4];
  #pragma unroll
          for (int n = 0; n < 2; ++n) {
  #pragma unroll
            for (int e = 0; e < 4; ++e) {
              float v = sc[n][e] * (e < 2 ? cr0 : cr1);
              if (ragged) {
                const int key = kw + n * 8 + tq * 2 + (e & 1);
                const int lim = e < 2 ? lim0 : lim1;
                if (key >= item.key_end || key > lim) v = -INFINITY;
              }
              x[n][e] = v;
            }
          }
  #ifdef PA_COVERAGE
  #pragma unroll
          for (int n = 0; n < 2; ++n)
  #pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = kw + n * 8 + tq * 2 + (e & 1), r = e < 2 ? r0 : r1;
              const bool in = !(ragged && (key >= item.key_end || key > (e < 2 ? lim0 : lim1)));
              if (in && r < n_rows) cov_count(a, c0 + r / a.G, item.g * a.G + r % a.G, key);
            }
  #endif
          float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
          float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
          const float ms0 = mn0 == -INFINITY ? 0.f : mn0;  // a row with no key yet stays empty
          const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
          const float al0 = fast_exp2(m0 - ms0), al1 = fast_exp2(m1 - ms1);
          m0 = mn0;
          m1 = mn1;
          float p[2][4];
  #pragma unroll
          for (int n = 0; n < 2; ++n) {
            p[n][0] = fast_exp2(x[n][0] - ms0);
            p[n][1] = fast_exp2(x[n][1] - ms0);
            p[n][2] = fast_exp2(x[n][2] - ms1);
            p[n][3] = fast_exp2(x[n][3] - ms1);
          }
          // P as the MMA A fragment; bf16 carries it as hi + lo (two products), fp16 as one
          uint32_t pa[4], pl[4];
          if constexpr (BF16 && KQ == 0) {
            split_bf16x2(p[0][0], p[0][1], pa[0], pl[0]);
            split_bf16x2(p[0][2], p[0][3], pa[1], pl[1]);
            split_bf16x2(p[1][0], p[1][1], pa[2], pl[2]);
            split_bf16x2(p[1][2], p[1][3], pa[3], pl[3]);
          } else {
            pa[0] = pack2<false>(p[0][0], p[0][1]);
            pa[1] = pack2<false>(p[0][2], p[0][3]);
            pa[2] = pack2<false>(p[1][0], p[1][1]);
            pa[3] = pack2<false>(p[1][2], p[1][3]);
          }
          if constexpr (KQ != 0) {
            // integer caches: the V codes enter P V with the conversion's offset (INT8 code +
            // 1152; INT4 (code + 8) 2^-24), which the output takes off after dividing by the row
            // sum; that sum must then add exactly the fp16 weights the MMA multiplies
            const float2 q0 = __half22float2(*reinterpret_cast<const __half2*>(&pa[0]));
            const float2 q1 = __half22float2(*reinterpret_cast<const __half2*>(&pa[1]));
            const float2 q2 = __half22float2(*reinterpret_cast<const __half2*>(&pa[2]));
            const float2 q3 = __half22float2(*reinterpret_cast<const __half2*>(&pa[3]));
            l0 = l0 * al0 + ((q0.x + q0.y) + (q2.x + q2.y));
            l1 = l1 * al1 + ((q1.x + q1.y) + (q3.x + q3.y));
          } else {
            l0 = l0 * al0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
            l1 = l1 * al1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
          }
          if (!__all_sync(0xffffffffu, al0 == 1.f && al1 == 1.f)) {  // (no row's max grew: O stays)
  #pragma unroll
            for (int d = 0; d < ND; ++d) {
              o[d][0] *= al0;
              o[d][1] *= al0;
              o[d][2] *= al1;
              o[d][3] *= al1;
            }
          }
          // ---- O (16 x HS) += P (16 x 16) V (16 x HS) ----
          // keys this thread contributes in the transposed V fragments: kw + 2tq + {0,1}, +8
          if constexpr (KQ == 1) {
            // (codes are finite: keys past the item contribute 0 * code = 0)
            // this thread's keys: ka = 16w + 2tq, ka + 1 (b0), ka + 8, ka + 9 (b1)
            constexpr int G = VG;  // channels (bytes) of a run
  #pragma unroll
            for (int D = 0; D < ND / G; ++D) {
              uint32_t w0[G / 4], w1[G / 4], w8[G / 4], w9[G / 4];
              lds_run<G>(vb + voff[0][D], w0);
              lds_run<G>(vb + voff[1][D], w1);
              lds_run<G>(vb + voff[0][D] + 8 * P, w8);
              lds_run<G>(vb + voff[1][D] + 8 * P, w9);
  #pragma unroll
              for (int i = 0; i < G / 4; ++i) {
                uint32_t lo[4], hi[4];
                s8_key_pairs_biased(w0[i], w1[i], lo);
                s8_key_pairs_biased(w8[i], w9[i], hi);
  #pragma unroll
                for (int e = 0; e < 4; ++e) mma16816<false>(o[D * G + 4 * i + e], pa, lo[e], hi[e]);
              }
            }
          } else if constexpr (KQ == 2) {
            constexpr int R = VG;  // bytes of the thread's HS / 8 channels in a key row
            uint32_t w0[R / 4], w1[R / 4], w8[R / 4], w9[R / 4];
            lds_run<R>(vb + voff[0][0], w0);
            lds_run<R>(vb + voff[1][0], w1);
            lds_run<R>(vb + voff[0][0] + 8 * P, w8);
            lds_run<R>(vb + voff[1][0] + 8 * P, w9);
  #pragma unroll
            for (int i = 0; i < R / 4; ++i) {
              uint32_t lo[8], hi[8];
              s4_key_pairs_sub(w0[i], w1[i], lo);
              s4_key_pairs_sub(w8[i], w9[i], hi);
  #pragma unroll
              for (int e = 0; e < 8; ++e) mma16816<false>(o[8 * i + e], pa, lo[e], hi[e]);
            }
          } else {
            const int mi = lane >> 3, rr = lane & 7;
            const int kr = 16 * w + (mi & 1) * 8 + rr;
            // keys past the item may be unwritten cache slots: on the item's last tile their V
            // is cleared, so that no NaN reaches 0 * V (the other tiles skip the masking)
            auto pv = [&](uint32_t mlo, uint32_t mhi) {
  #pragma unroll
              for (int dp = 0; dp < ND / 2; ++dp) {
                const int c = 2 * dp + (mi >> 1);
                const uint32_t addr = vb + (c >> 3) * (kDecTile * 128) + kr * 128 + (((c & 7) ^ (kr & 7)) << 4);
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(addr, v0, v1, v2, v3);
                v0 &= mlo;
                v2 &= mlo;
                v1 &= mhi;
                v3 &= mhi;
                mma16816<BF16>(o[2 * dp], pa, v0, v1);
                mma16816<BF16>(o[2 * dp + 1], pa, v2, v3);
                if constexpr (BF16) {
                  mma16816<BF16>(o[2 * dp], pl, v0, v1);
                  mma16816<BF16>(o[2 * dp + 1], pl, v2, v3);
                }
              }
            };
            const int ka = kw + tq * 2, kb2 = ka + 8;
            const uint32_t mlo = (ka < item.key_end ? 0x0000ffffu : 0u) | (ka + 1 < item.key_end ? 0xffff0000u : 0u);
            const uint32_t mhi = (kb2 < item.key_end ? 0x0000ffffu : 0u) | (kb2 + 1 < item.key_end ? 0xffff0000u : 0u);
            if (HS == 256 || k0 + kDecTile > item.key_end) pv(mlo, mhi);  // (one copy of the loop at 256)
            else pv(0xffffffffu, 0xffffffffu);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++stage == L::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }

    // ---- combine the four warps' partial states in a fixed order ----
    constexpr int kCompactRows = kDecRows / kDecWarps;
    bool compact = false;  // (row-major form, items of at most kCompactRows rows)
    if constexpr (NARROW) {
      // the rows' sums over the warp's keys (the lanes of one tq), then the row states
      l0 += __shfl_xor_sync(0xffffffffu, l0, 4);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 8);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 16);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 4);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 8);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 16);
      if (gq == 0) {
        mw[w * kDecRows + ra] = m0;
        mw[w * kDecRows + rb] = m1;
        lw[w * kDecRows + ra] = l0;
        lw[w * kDecRows + rb] = l1;
      }
      consumer_bar();
      float M0, L0, M1, L1;
      row_stats(mw, lw, ra, M0, L0);
      row_stats(mw, lw, rb, M1, L1);
      const float f0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - M0);
      const float f1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M1);
      // warps 0 and 1 write rows 0 .. 7 and 8 .. 15 of the buffer, then warps 2 and 3 add
      // theirs; the write below adds the two halves (the order, and so the rounding, fixed)
      float* cw = comb + (w & 1) * 8 * kCombStride;
#pragma unroll 1
      for (int rr = 0; rr < 2; ++rr) {
        if ((w >> 1) == rr) {
          float* pa0 = cw + ra * kCombStride;
          float* pa1 = cw + rb * kCombStride;
#pragma unroll
          for (int d = 0; d < NO; ++d) {
            const int ch0 = out_channel<HS, KQ>(2 * d, gq), ch1 = out_channel<HS, KQ>(2 * d + 1, gq);
            if (rr == 0) {
              pa0[ch0] = o[d][0] * f0;
              pa1[ch0] = o[d][1] * f1;
              pa0[ch1] = o[d][2] * f0;
              pa1[ch1] = o[d][3] * f1;
            } else {
              pa0[ch0] += o[d][0] * f0;
              pa1[ch0] += o[d][1] * f1;
              pa0[ch1] += o[d][2] * f0;
              pa1[ch1] += o[d][3] * f1;
            }
          }
        }
        consumer_bar();
      }
    } else {
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      if (tq == 0) {
        mw[w * kDecRows + r0] = m0;
        mw[w * kDecRows + r1] = m1;
        lw[w * kDecRows + r0] = l0;
        lw[w * kDecRows + r1] = l1;
      }
      consumer_bar();
      float M0, L0, M1, L1;
      row_stats(mw, lw, r0, M0, L0);
      row_stats(mw, lw, r1, M1, L1);
      const float f0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - M0);
      const float f1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M1);
      // An item of at most kDecRows / kDecWarps rows (one decode token of up to four heads): the
      // four warps' rows fit the buffer side by side, warp w's at rows 4w .. 4w + 3, so they
      // are written in one round and the write below adds them in warp order (the order, and
      // so the rounding, of the rounds).
      compact = L::kCombBufs == 1 && n_rows <= kCompactRows;
      if (compact) {
        if (gq < kCompactRows) {
          if constexpr (KQ == 0) {
            float* cw = comb + (w * kCompactRows + r0) * kCombStride + tq * 2;
  #pragma unroll
            for (int d = 0; d < ND; ++d)
              *reinterpret_cast<float2*>(cw + d * 8) = make_float2(o[d][0] * f0, o[d][1] * f0);
          } else {  // integer caches: the columns' channels in natural order
            float* cw = comb + (w * kCompactRows + r0) * kCombStride;
  #pragma unroll
            for (int d = 0; d < ND; ++d) {
              cw[out_channel<HS, KQ>(d, 2 * tq)] = o[d][0] * f0;
              cw[out_channel<HS, KQ>(d, 2 * tq + 1)] = o[d][1] * f0;
            }
          }
        }
        consumer_bar();
      } else {
        // round rr: warps rr * B .. rr * B + B - 1 write (first round) or add their partials
        // into buffers 0 .. B - 1; buffer b ends up holding warps b, b + B, ... in that order
        constexpr int B = L::kCombBufs;
        float* cw = comb + (w % B) * (kDecRows * kCombStride);
  #pragma unroll 1
        for (int rr = 0; rr < kDecWarps / B; ++rr) {
          if (w / B == rr) {
  #pragma unroll
            for (int d = 0; d < ND; ++d) {
              if constexpr (KQ == 0) {
                float2* c0p = reinterpret_cast<float2*>(cw + r0 * kCombStride + d * 8 + tq * 2);
                float2* c1p = reinterpret_cast<float2*>(cw + r1 * kCombStride + d * 8 + tq * 2);
                const float2 a0 = make_float2(o[d][0] * f0, o[d][1] * f0), a1 = make_float2(o[d][2] * f1, o[d][3] * f1);
                if (rr == 0) {
                  *c0p = a0;
                  *c1p = a1;
                } else {
                  const float2 b0 = *c0p, b1 = *c1p;
                  *c0p = make_float2(b0.x + a0.x, b0.y + a0.y);
                  *c1p = make_float2(b1.x + a1.x, b1.y + a1.y);
                }
              } else {  // integer caches: the columns' channels in natural order
                const int ch0 = out_channel<HS, KQ>(d, 2 * tq), ch1 = out_channel<HS, KQ>(d, 2 * tq + 1);
                float* c0p = cw + r0 * kCombStride;
                float* c1p = cw + r1 * kCombStride;
                if (rr == 0) {
                  c0p[ch0] = o[d][0] * f0;
                  c0p[ch1] = o[d][1] * f0;
                  c1p[ch0] = o[d][2] * f1;
                  c1p[ch1] = o[d][3] * f1;
                } else {
                  c0p[ch0] += o[d][0] * f0;
                  c0p[ch1] += o[d][1] * f0;
                  c1p[ch0] += o[d][2] * f1;
                  c1p[ch1] += o[d][3] * f1;
                }
              }
            }
          }
          consumer_bar();
        }
      }
    }
    // ---- write: thread t owns row t / 8, HS / 8 consecutive columns ----
    {
      const int t = threadIdx.x;  // 0..127
      const int row = t >> 3;
      constexpr int CW = HS / 8;
      const int col = (t & 7) * CW;
      const bool mine = row < n_rows;
      const int tok = c0 + row / a.G;
      const int head = item.g * a.G + row % a.G;
      uint16_t* dst = reinterpret_cast<uint16_t*>(a.output) + ((int64_t)tok * a.nh + head) * HS + col;
      float M = 0.f, Lr = 0.f;
      if (mine) row_stats(mw, lw, row, M, Lr);
      const float inv = Lr > 0.f ? 1.f / Lr : 0.f;
      const float* src = comb + row * kCombStride + col;
      // the combined (unnormalised) O of this thread's row and column v: the warps'
      // partials added in warp order
      auto cval = [&](int v) {
        float x = src[v];
        if constexpr (NARROW) return x + src[8 * kCombStride + v];
        if (compact) {  // (row < kCompactRows)
#pragma unroll
          for (int ww = 1; ww < kDecWarps; ++ww) x += src[ww * kCompactRows * kCombStride + v];
          return x;
        }
#pragma unroll
        for (int bb = 1; bb < L::kCombBufs; ++bb) x += src[bb * (kDecRows * kCombStride) + v];
        return x;
      };
      float lbias = 0.f;  // (integer caches) the row's key bias, taken off the exported lse
      if constexpr (KQ != 0) {
        if (a.lse) lbias = key_row_bias<HS, KQ>(a, tok, head, t, mine);
      }
      if (item.n_split == 1) {
        if (mine && a.lse && (t & 7) == 0)  // natural log; M is the base-2 max of s * scale
          a.lse[(int64_t)tok * a.nh + head] =
              Lr > 0.f ? (M + fast_log2(Lr)) * 0.69314718055994531f - lbias : -INFINITY;
        if (mine) {
#pragma unroll
          for (int v = 0; v < CW; v += 8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = cval(v + e) * inv;
            if constexpr (KQ != 0) {  // integer caches: the V scales of the output channels
#pragma unroll
              for (int e = 0; e < 8; ++e)  // (the V codes' offset off) then the V scales
                x[e] = v_code_value<KQ>(x[e]) * __ldg(a.v_scale + item.g * HS + col + v + e);
            }
            if (a.gate)  // output gate: times sigmoid(gate), elementwise
              apply_gate8<BF16>(a.gate + ((int64_t)tok * a.nh + head) * HS + col + v, x);
            uint4 pk;
            pk.x = pack2<BF16>(x[0], x[1]);
            pk.y = pack2<BF16>(x[2], x[3]);
            pk.z = pack2<BF16>(x[4], x[5]);
            pk.w = pack2<BF16>(x[6], x[7]);
            *reinterpret_cast<uint4*>(dst + v) = pk;
          }
        }
      } else {
        // A unit the balanced partition cuts has its pieces in different CTAs: the first
        // piece (keys from 0) is the last item of its CTA, the others are the first items of
        // the next CTAs (or a later CTA's whole range). The first piece's CTA merges, once the
        // others have arrived (by then they usually have: they were done early), from its own
        // combine buffer and their partials; the others publish their partials and move on.
        // With forced split lengths a CTA may hold several pieces of one unit: there the last
        // piece to finish merges.
        const bool balanced = a.forced_split <= 0;
        const bool merger = balanced && item.key_begin == 0;
        int* done = &a.unit_done[item.b * a.kvh + item.g];
        const float own_lse = Lr > 0.f ? (M + fast_log2(Lr)) * 0.69314718055994531f : -INFINITY;
        if (!merger) {
          if (mine) {
            float* pdst = a.part_o + ((int64_t)it * kDecRows + row) * HS + col;
#pragma unroll
            for (int v = 0; v < CW; v += 4)
              *reinterpret_cast<float4*>(pdst + v) =
                  make_float4(cval(v) * inv, cval(v + 1) * inv, cval(v + 2) * inv, cval(v + 3) * inv);
            if ((t & 7) == 0) a.part_lse[(int64_t)it * kDecRows + row] = own_lse;
          }
          consumer_bar();  // every consumer thread's partial is written
          if (t == 0) {
            // at gpu scope after the barrier: the release publishes the CTA's partial
            // (cumulative over the writes the barrier ordered before it); with forced splits
            // the acquire also orders the merge's reads of the other items' partials
            if (balanced) red_add_release_gpu(done, 1);
            else *s_last = atom_add_acq_rel_gpu(done, 1) == item.n_split - 1;
          }
          if (!balanced) consumer_bar();
        } else {
          // (acquire at gpu scope, then the barrier: the reads below follow the arrivals)
          if (t == 0) *s_last = wait_count_acquire_gpu(done, item.n_split - 1, abort, err);
          consumer_bar();
        }
        if ((merger || !balanced) && *s_last && mine) {
          // merge the unit's pieces in key order with a running max: the merger's own piece
          // from its combine buffer, then the partials two per step (both pieces' lse and rows
          // loaded together, one L2 round trip per step: this merge usually ends the CTA's work)
          float Mx = -INFINITY;
          float acc[CW];
          float den = 0.f;
#pragma unroll
          for (int v = 0; v < CW; ++v) acc[v] = 0.f;
          if (merger && own_lse != -INFINITY) {
            Mx = own_lse;
            den = 1.f;
#pragma unroll
            for (int v = 0; v < CW; ++v) acc[v] = cval(v) * inv;
          }
          for (int s2 = merger ? 1 : 0; s2 < item.n_split; s2 += 2) {
            const bool two = s2 + 1 < item.n_split;
            const int64_t pa = (int64_t)piece_slot<SELF>(item, s2) * kDecRows + row;
            const int64_t pb = two ? (int64_t)piece_slot<SELF>(item, s2 + 1) * kDecRows + row : pa;
            const float la = __ldcg(a.part_lse + pa);
            const float lb = two ? __ldcg(a.part_lse + pb) : -INFINITY;
            const float4* psa = reinterpret_cast<const float4*>(a.part_o + pa * HS + col);
            const float4* psb = reinterpret_cast<const float4*>(a.part_o + pb * HS + col);
            float4 xa[CW / 4], xb[CW / 4];
#pragma unroll
            for (int v = 0; v < CW / 4; ++v) {
              xa[v] = __ldcg(psa + v);
              xb[v] = __ldcg(psb + v);  // (piece a again when there is no second piece: weight 0)
            }
            const float Mn = fmaxf(Mx, fmaxf(la, lb));
            if (Mn == -INFINITY) continue;  // no key so far
            const float sc = Mx == -INFINITY ? 0.f : fast_exp2((Mx - Mn) * 1.4426950408889634f);
            const float wa = la == -INFINITY ? 0.f : fast_exp2((la - Mn) * 1.4426950408889634f);
            const float wb = lb == -INFINITY ? 0.f : fast_exp2((lb - Mn) * 1.4426950408889634f);
            den = (den * sc + wa) + wb;
#pragma unroll
            for (int v = 0; v < CW / 4; ++v) {
              acc[4 * v + 0] = (acc[4 * v + 0] * sc + wa * xa[v].x) + wb * xb[v].x;
              acc[4 * v + 1] = (acc[4 * v + 1] * sc + wa * xa[v].y) + wb * xb[v].y;
              acc[4 * v + 2] = (acc[4 * v + 2] * sc + wa * xa[v].z) + wb * xb[v].z;
              acc[4 * v + 3] = (acc[4 * v + 3] * sc + wa * xa[v].w) + wb * xb[v].w;
            }
            Mx = Mn;
          }
          const float dinv = 1.f / den;
          if (a.lse && (t & 7) == 0) a.lse[(int64_t)tok * a.nh + head] = Mx + fast_log2(den) * 0.69314718055994531f - lbias;
#pragma unroll
          for (int v = 0; v < CW; v += 8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = acc[v + e] * dinv;
            if constexpr (KQ != 0) {
#pragma unroll
              for (int e = 0; e < 8; ++e)  // (the V codes' offset off) then the V scales
                x[e] = v_code_value<KQ>(x[e]) * __ldg(a.v_scale + item.g * HS + col + v + e);
            }
            if (a.gate) apply_gate8<BF16>(a.gate + ((int64_t)tok * a.nh + head) * HS + col + v, x);
            uint4 pk;
            pk.x = pack2<BF16>(x[0], x[1]);
            pk.y = pack2<BF16>(x[2], x[3]);
            pk.z = pack2<BF16>(x[4], x[5]);
            pk.w = pack2<BF16>(x[6], x[7]);
            *reinterpret_cast<uint4*>(dst + v) = pk;
          }
        }
      }
    }
    consumer_bar();  // comb, mw, lw are reused by the next item
  }
  if (beside_prefill) pdl_wait();
}

// Ahead of a self-planned decode-only call (one CTA): the header reset for this call (the
// error word describes the most recent call) and the merge counters of the batch's
// (sequence, KV head) units zeroed. Its dependents start once the previous call's kernels
// are done, so the decode kernel can cut its partition from the batch description while
// this kernel runs.
__global__ void __launch_bounds__(256) decode_prep_kernel(const Args a) {
  // the batch description into L2 while the previous call finishes (hints only): the decode
  // kernel's prologue reads it next
  for (int i = threadIdx.x * 32; i <= a.B; i += blockDim.x * 32) {
    prefetch_l2(a.cum + i);
    if (i < a.B) prefetch_l2(a.past + i);
  }
  pdl_wait();  // the previous call's kernels may still use this workspace
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    WsHeader* hdr = a.hdr;
    hdr->error = 0;
    hdr->valid = 1;  // (the decode kernel clears it for a refused batch)
    hdr->n_decode_items = 0;
    hdr->n_prefill_tiles = 0;
    hdr->dec_ctas = a.dec_ctas;
    hdr->v_mirror = 0;
    hdr->v_mirror_bad = 0;
    hdr->mirror_rows = 0;
    hdr->pre_ctas = 0;
  }
  for (int u = threadIdx.x; u < a.B * a.kvh; u += blockDim.x) a.unit_done[u] = 0;
}

// ---- host launchers (kernels are launched from the translation unit that defines them) ----
cudaError_t launch_decode_prep(const Args& a, cudaStream_t s) {
  return launch_pdl(decode_prep_kernel, dim3(1), dim3(256), 0, s, a);
}

template <int HS, bool BF16, int KQ, bool SELF = false, bool NARROW = false>
static cudaError_t launch_decode_t(const Args& a, const CUtensorMap& tk, const CUtensorMap& tv, int seg,
                                   cudaStream_t s) {
  if constexpr (!SELF) {  // self-planned decode-only batches: their own instantiation
    if (a.self_plan) return launch_decode_t<HS, BF16, KQ, true, NARROW>(a, tk, tv, seg, s);
  }
  if constexpr (KQ != 0 && !NARROW) {  // items of at most 8 rows on integer caches
    if (a.dec_narrow) return launch_decode_t<HS, BF16, KQ, SELF, true>(a, tk, tv, seg, s);
  }
  constexpr int smem = DecSmem<HS, KQ, SELF>::kBytes;
  cudaError_t e =
      cudaFuncSetAttribute(decode_kernel<HS, BF16, KQ, SELF, NARROW>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_kernel<HS, BF16, KQ, SELF, NARROW>, dim3(a.dec_ctas), dim3(160), smem, s, a, tk, tv, seg);
}

template <int KQ>
static cudaError_t launch_decode_kq(const Args& a, bool bf16, const CUtensorMap& tk, const CUtensorMap& tv, int seg,
                                    cudaStream_t s) {
  if (a.hs == 256)
    return bf16 ? launch_decode_t<256, true, KQ>(a, tk, tv, seg, s) : launch_decode_t<256, false, KQ>(a, tk, tv, seg, s);
  if constexpr (KQ != 2) {  // (INT4 needs head_size 128 or 256)
    if (a.hs == 64)
      return bf16 ? launch_decode_t<64, true, KQ>(a, tk, tv, seg, s) : launch_decode_t<64, false, KQ>(a, tk, tv, seg, s);
  }
  return bf16 ? launch_decode_t<128, true, KQ>(a, tk, tv, seg, s) : launch_decode_t<128, false, KQ>(a, tk, tv, seg, s);
}

cudaError_t launch_decode(const Args& a, bool bf16, const CUtensorMap& tk, const CUtensorMap& tv, int seg,
                          cudaStream_t s) {
  if (a.kvq == 1) return launch_decode_kq<1>(a, bf16, tk, tv, seg, s);
  if (a.kvq == 2) return launch_decode_kq<2>(a, bf16, tk, tv, seg, s);
  return launch_decode_kq<0>(a, bf16, tk, tv, seg, s);
}

}  // namespace pa
