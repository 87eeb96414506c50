// Shared definitions of the GB300 PagedAttention kernels: workspace layout, work-item
// records, and inline-PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor), tcgen05
// (TMEM allocation, MMA, loads/stores) and the warp-level ldmatrix / mma.sync used by
// the decode kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedattn.h"

namespace pa {

// ---- tiling constants ---------------------------------------------------------------
constexpr int kDecTile = 64;          // keys per decode pipeline stage
constexpr int kDecStages = 3;         // decode K/V ring depth
constexpr int kDecWarps = 4;          // decode consumer warps (16 keys of a tile each)
constexpr int kDecRows = 16;          // query rows per decode work item (one m16 MMA tile)
constexpr int kDecCtasPerSm = 2;      // resident decode CTAs per SM (shared-memory bound), head_size <= 128
// head_size 256: a 3-stage ring of 64-key K and V tiles is 192 KB, one CTA per SM. Integer
// caches below 256: three (their tiles are half or a quarter of the bytes, and the codes'
// conversion is latency-bound, so a third CTA's warps hide more of it)
__host__ __device__ constexpr int dec_ctas_per_sm(int hs, int kq = 0) {
  return hs == 256 ? 1 : kq ? 3 : kDecCtasPerSm;
}
// What an item costs a decode CTA beyond streaming its keys (the warps' combine, the write
// of the row or partial, the merge, the refill of the ring at the next item), in 64-key
// tiles streamed in the same time (measured: about 5 us per item against 1.4 us per tile
// at head_size 256 with one CTA per SM; at 128 with two, per-CTA timestamps fitted about
// 4 us per item against 1.2 us per tile, the CTAs with the most items finishing last).
// On integer caches a tile streams in about 1.0 us (the codes' conversion, not HBM, bounds it)
// against an item cost of about 5 us, so an item counts 5 tiles there.
__host__ __device__ constexpr int dec_item_cost_tiles(int /*hs*/, int kq = 0) { return kq ? 5 : 3; }
constexpr int kMaxDecCtas = 1024;     // upper bound of the decode grid
constexpr int kSelfMaxB = 256;        // sequences of a decode-only batch the decode kernel plans itself
// (at head_size 256, whose one CTA per SM holds a 192 KB ring, 64: the batch view fits beside
// the two combine buffers)
__host__ __device__ constexpr int self_max_b(int hs) { return hs == 256 ? 64 : kSelfMaxB; }
constexpr int kEarlyWriteMaxB = 1024; // sequences a bit-copy cache write checks per CTA to run beside the planner
// rates of the planner's model that splits the SMs between the prefill and the decode
// kernel of a call with both kinds of rows (measured on GB300 at head_size 128)
constexpr float kSplitPreFlops = 8.2e12f;   // prefill FLOP/s per SM, 128 x 128 tiles counted whole
constexpr float kSplitDecBytes = 85.0e9f;   // decode K/V bytes/s per SM while HBM is not the limit
constexpr float kSplitHbmBytes = 5.9e12f;   // decode K/V bytes/s of the whole chip
constexpr int kPreTileQ = 128;        // query rows per prefill tile (MMA M)
constexpr int kPreTileK = 128;        // keys per prefill KV tile (MMA N of Q K^T, K of P V)
constexpr int kSortCap = 4096;        // prefill tiles the planner sorts by cost

// ---- workspace records ----------------------------------------------------------------
struct WsHeader {
  uint32_t error;           // PA_DEVERR_* bits
  int32_t valid;            // 1 when the planner accepted the batch
  int32_t n_decode_items;
  int32_t n_prefill_tiles;
  int32_t dec_ctas;         // decode grid the item ranges were cut for
  int32_t v_mirror;         // 1: bf16 prefill reads V from the fp16 copy (planner)
  uint32_t v_mirror_bad;    // set by the copy kernel when a value does not fit fp16
  int32_t mirror_rows;      // rows of the copy in use
  int32_t mirror_seqs;      // sequences copied (entries of mirror_seq)
  int32_t pre_ctas;         // prefill CTAs that take units (0: the whole grid); the others exit
  int32_t pad[54];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte line");

// One (sequence b, KV head g, key range) of a decode-class sequence. The (b, g) pair is a
// "unit" (index b * kv_num_heads + g); a unit cut into several items has each item write
// an fp32 partial, and the last item to finish (counted in unit_done) merges them in key
// order.
struct __align__(16) DecodeItem {
  int32_t b, g, key_begin, key_end;
  int32_t unit_first;   // index of the unit's first item (its items are consecutive)
  int32_t n_split;      // items in the unit; 1 = the item writes the output itself
  int32_t c0;           // cumulative_sequence_length[b]
  int32_t q_len, past;  // the sequence's new rows and history (so the kernel needs no lookups)
  int32_t pad[3];
};

// 128 query rows [j0, j0 + 128) of sequence b (all heads), with the sequence's geometry,
// so the prefill kernel reads one record per unit and no further lookups.
struct __align__(32) PrefillTile {
  int32_t b, j0;
  int32_t c0;           // cumulative_sequence_length[b]: the sequence's first packed row
  int32_t q_len, past;
  int32_t n_kv;         // 128-key tiles the query tile reads (causal)
  int32_t mirror_row0;  // the sequence's first row in the fp16 V copy (when it is used)
  int32_t pad;
};

struct WsLayout {
  size_t header, items, cta_begin, unit_done, tiles, tiles_unsorted, part_o, part_lse, mirror_base, mirror_seq,
      mirror, qprep, qexp, total;
  int32_t max_items, max_tiles;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Upper bounds of the device-built lists, from host-known sizes only.
//  - decode items, balanced partition: the concatenated key tiles of all units are cut
//    into at most kMaxDecCtas contiguous ranges, so items <= kMaxDecCtas + units;
//  - decode items, forced split length S: at most ceil(max_kv / S) per unit;
//  - prefill tiles: sum_b ceil(q_b / 128) <= N / 128 + B.
// mirror_keys: rows of the fp16 copy of V that bf16 prefill reads (0: none); qprep_values:
// 16-bit values of the prepared query rows (0: no Q/K preparation and no integer caches);
// qexp_values: the per-row exponents of the scaled query rows of integer caches (0: none).
__host__ __device__ inline WsLayout ws_layout(int32_t N, int32_t B, int32_t kvh, int32_t hs,
                                               int32_t max_blocks, int32_t bs, int32_t forced_split,
                                               int64_t mirror_keys, int64_t qprep_values,
                                               int64_t qexp_values = 0) {
  WsLayout L;
  const int64_t units = (int64_t)B * kvh;
  int64_t items;
  if (forced_split > 0) items = units * ceil_div((int64_t)max_blocks * bs, forced_split);
  else items = kMaxDecCtas + units;
  int64_t tiles = ceil_div(N, kPreTileQ) + (B < N ? B : N);
  L.max_items = (int32_t)items;
  L.max_tiles = (int32_t)tiles;
  size_t off = 0;
  L.header = off; off += sizeof(WsHeader);
  L.items = off; off = align_up(off + sizeof(DecodeItem) * (size_t)items, 256);
  L.cta_begin = off; off = align_up(off + sizeof(int32_t) * (kMaxDecCtas + 1), 256);
  L.unit_done = off; off = align_up(off + sizeof(int32_t) * (size_t)units, 256);
  L.tiles = off; off = align_up(off + sizeof(PrefillTile) * (size_t)tiles, 256);
  L.tiles_unsorted = off; off = align_up(off + sizeof(PrefillTile) * (size_t)tiles, 256);
  L.part_o = off; off = align_up(off + sizeof(float) * (size_t)items * kDecRows * hs, 256);
  L.part_lse = off; off = align_up(off + sizeof(float) * (size_t)items * kDecRows, 256);
  L.mirror_base = off; off = align_up(off + sizeof(int32_t) * ((size_t)B + 1), 256);
  L.mirror_seq = off; off = align_up(off + 2 * sizeof(int32_t) * ((size_t)B + 1), 256);
  L.mirror = off; off = align_up(off + (size_t)mirror_keys * kvh * hs * 2, 256);
  L.qprep = off; off = align_up(off + (size_t)qprep_values * 2, 256);
  L.qexp = off; off = align_up(off + (size_t)qexp_values * 4, 256);
  L.total = off;
  return L;
}

// ---- arguments shared by the kernels ----------------------------------------------------
struct Args {
  const void* query;
  const void* key;
  const void* value;
  void* key_cache;
  void* value_cache;
  const int32_t* cum;
  const int32_t* past;
  const int32_t* block_table;
  const int32_t* slot_mapping;
  void* output;
  float* lse;             // (N, nh) natural-log lse of each output row, or null
  const uint16_t* gate;   // (N, nh * hs) output gate (output *= sigmoid(gate)), or null
  // Q/K preparation in the cache-write stage (prep != 0): RMSNorm weights (or null), the
  // rotary dimension, its fp32 frequency table, and the prepared query rows (N, nh, hs)
  int32_t prep;
  int32_t bf16;           // T is bf16 (else fp16)
  int32_t rotary_dim;
  float norm_eps;
  const uint16_t* q_norm_w;
  const uint16_t* k_norm_w;
  uint16_t* qprep;
  // Integer caches (kvq = 1 INT8, 2 INT4; 0: caches of T): the fp32 (kvh, hs) scales, and
  // per query row (token, head) the exponent E of its scaled copy: the attention kernels
  // read Q' = fp16(q * k_scale * 2^-E) from qprep and multiply the scores by 2^E
  int32_t kvq;
  const float* k_scale;
  const float* v_scale;
  int32_t* qexp;
  float inv_freq[128];   // rotary inverse frequencies, one per rotated pair (rotary_dim / 2 <= 128)
  int32_t N, B, nh, kvh, G, hs, num_blocks, bs, max_blocks;
  int32_t q_stride;       // elements per query row
  int32_t kv_row;         // kvh * hs
  int32_t k_offset;       // element offset of K inside a query row (packed) or 0
  int32_t v_offset;
  int32_t packed;
  int32_t forced_split;   // > 0: decode units cut into items of this many keys
  int32_t route;
  int32_t max_query_len;  // > 0: host bound on every q_len (checked by the planner)
  int32_t dec_ctas;       // decode grid size
  int32_t sms;            // SMs of the device
  // A whole call that launches both attention kernels may run them at the same time: the
  // planner gives the decode work d SMs (decode_sms > 0 fixes d) and the prefill kernel the
  // other SMs; the decode kernel, launched after the prefill kernel, then does not wait for
  // it to finish before starting (dec_after_prefill), only before exiting.
  int32_t split_sms;
  int32_t decode_sms;
  int32_t dec_after_prefill;
  // decode-only batch with derived slots and at most kSelfMaxB sequences: no plan and no
  // cache-write kernel; each decode CTA cuts its own share of the balanced partition from
  // the batch description and writes the new K/V rows of the tiles it loads
  int32_t self_plan;
  int32_t self_write_rows;  // self-planned and the decode kernel writes this call's K/V rows
  int32_t dec_narrow;       // integer caches, every decode item at most 8 query rows (host bound)
  int32_t cw_early;         // bit-copy cache write launched right after this call's planner:
                            // it copies the rows while the planner runs (checking the batch
                            // itself) and waits for the plan only before the fp16 V copy
                            // (else the cache-write kernel writes them, checking the batch itself)
  int32_t out_v8;         // output 32-byte aligned (prefill stores 32-byte chunks)
  float scale_log2;       // scale * log2(e)
  WsHeader* hdr;
  DecodeItem* items;
  int32_t* cta_begin;     // decode CTA c owns items [cta_begin[c], cta_begin[c + 1])
  int32_t* unit_done;     // per unit: items finished (for the fused merge)
  PrefillTile* tiles;
  PrefillTile* tiles_unsorted;
  float* part_o;
  float* part_lse;
  int32_t* mirror_base;   // per prefill-class sequence b: its first row in the V copy
  int2* mirror_seq;       // k-th copied sequence: (b, first row), in row order
  uint16_t* mirror;       // fp16 copy of the V history of the prefill-class sequences (bf16)
  int32_t mirror_keys;    // rows the copy holds (0: no copy)
  int32_t max_items, max_tiles;
  // coverage counters (a library built with PA_COVERAGE; null otherwise): see cov_count
  int32_t* cov;
  int32_t cov_keys;
};

// Coverage counting, compiled only into the debug library built with PA_COVERAGE: every
// (query row, head, key) that an attention kernel lets into its softmax adds one to
// cov[(row * nh + head) * cov_keys + key] (keys from cov_keys on to the overflow counter
// cov[N * nh * cov_keys]), so that a test can check that the work partition and the
// kernels' loop bounds and masks take every key of every row's causal range exactly once.
#ifdef PA_COVERAGE
__device__ __forceinline__ void cov_count(const Args& a, int64_t row, int h, int key) {
  if (!a.cov) return;
  const int64_t i = key < a.cov_keys ? (row * a.nh + h) * (int64_t)a.cov_keys + key
                                     : (int64_t)a.N * a.nh * a.cov_keys;
  atomicAdd(a.cov + i, 1);
}
#endif

// ---- shared-memory layouts (bytes) of the attention kernels --------------------------
// Decode: a ring of K+V tiles, the warp-combine buffer, per-warp (m, l), barriers.
// The consumer warps combine their partial states in kCombBufs shared-memory buffers: warp
// w adds into buffer w % kCombBufs, the buffers' warps in turn, and the writer sums the
// buffers in order. At head_size 256 (one CTA per SM) there is room for two buffers next to
// the 3-stage ring (two rounds instead of four); below, two CTAs share an SM and one buffer
// takes the four warps in turn.
//
// Integer caches (KQ = 1 INT8, 2 INT4) have rows of HS or HS / 2 bytes, so a stage is half or
// a quarter of the 16-bit one and the ring is that much deeper (the same bytes in flight).
// A row is TMA'd in boxes of kBoxBytes (at most 128) with the matching swizzle.
template <int HS, int KQ = 0, bool SELF = false>
struct DecSmem {
  static constexpr int kRowBytes = KQ == 0 ? HS * 2 : KQ == 1 ? HS : HS / 2;
  static constexpr int kBoxBytes = kRowBytes < 128 ? kRowBytes : 128;
  static constexpr int kBoxes = kRowBytes / kBoxBytes;
  // (the self-planned 256-wide INT4 kernel, whose ring is deepest, gives its second buffer's
  // room to the batch view)
  static constexpr int kCombBufs = HS == 256 && !(SELF && KQ == 2) ? 2 : 1;
  static constexpr int kHalves = HS / 64;
  static constexpr int kTileBytes = kDecTile * kRowBytes;   // one K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  // ring depth: kDecStages stages on fp16 caches; integer caches fill the same 192 KB at
  // head_size 256 (one CTA per SM) and 48 KB below (three CTAs per SM)
  static constexpr int kStages =
      KQ == 0 ? kDecStages : (HS == 256 ? 3 * 65536 : 3 * 16384) / kStageBytes;
  // floats; the pad spreads rows over banks (2 for the self-planned 256-wide kernel, whose
  // batch view takes the last bytes of shared memory)
  static constexpr int kCombStride = HS + (HS == 256 && SELF ? 2 : 4);
  static constexpr int kComb = kStages * kStageBytes;        // float [kCombBufs][16][kCombStride]
  static constexpr int kMw = kComb + kCombBufs * kDecRows * kCombStride * 4;  // float [4][16]
  static constexpr int kLw = kMw + kDecWarps * kDecRows * 4; // float [4][16]
  static constexpr int kBars = kLw + kDecWarps * kDecRows * 4;
  static constexpr int kAbort = kBars + 2 * kStages * 8;
  // self-planned batches: int64 T[MB + 1], int64 meta[8], int cum[MB + 1], int past[MB],
  // MB = self_max_b(HS)
  static constexpr int kSelf = (kAbort + 16 + 15) / 16 * 16;
  static constexpr int kSelfBytes =
      !SELF ? 0 : ((self_max_b(HS) + 1 + 8) * 8 + (2 * self_max_b(HS) + 1) * 4 + 15) / 16 * 16;
  // integer caches at three CTAs per SM: the item's Q' fragments in shared memory
  // (uint4 [HS / 16][32], k-step by lane), not in registers
  static constexpr bool kQSmem = KQ != 0 && HS <= 128;
  static constexpr int kQ = kSelf + kSelfBytes;
  static constexpr int kQBytes = kQSmem ? HS / 16 * 32 * 16 : 0;
  static constexpr int kBytes = kQ + kQBytes + 1024;   // + alignment slack
};
static_assert(DecSmem<256>::kBytes <= 232448 && 2 * (DecSmem<128>::kBytes + 1024) <= 233472 &&
                  DecSmem<256, 1>::kBytes <= 232448 && DecSmem<256, 2>::kBytes <= 232448 &&
                  3 * (DecSmem<128, 1>::kBytes + 1024) <= 233472 && 3 * (DecSmem<128, 2>::kBytes + 1024) <= 233472 &&
                  2 * (DecSmem<128, 0, true>::kBytes + 1024) <= 233472 &&
                  3 * (DecSmem<128, 1, true>::kBytes + 1024) <= 233472 &&
                  3 * (DecSmem<128, 2, true>::kBytes + 1024) <= 233472 &&
                  3 * (DecSmem<64, 1, true>::kBytes + 1024) <= 233472 && DecSmem<256, 0, true>::kBytes <= 232448 &&
                  DecSmem<256, 1, true>::kBytes <= 232448 && DecSmem<256, 2, true>::kBytes <= 232448,
              "decode shared memory");

// Prefill: Q tile, two K and two V tiles, barriers, the TMEM address slot.
template <int HS>
struct PreSmem {
  static constexpr int kQBytes = kPreTileQ * HS * 2;  // one query tile (one head)
  static constexpr int kKVBytes = kPreTileK * HS * 2;
  static constexpr int kHalfBytes = kPreTileK * 128;  // one 64-column slab of a tile
  static constexpr int kQ = 0;                        // Q of head A, then Q of head B
  static constexpr int kK0 = kQ + 2 * kQBytes;
  static constexpr int kV0 = kK0 + 2 * kKVBytes;
  static constexpr int kBars = kV0 + 2 * kKVBytes;
  // q_full, q_empty, k_full[2], k_empty[2], v_full[2], v_empty[2], and per head (A, B):
  // s_full, p_full, o_done, o_free; integer caches: kc_full[2], vc_full[2] (code rows landed)
  static constexpr int kNumBars = 22;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kPreCtas = kAbort + 4;  // CTAs of the grid that take units
  // row-max exchange between the two warps that share a TMEM lane quarter:
  // float [tile parity][head][row][column half]
  static constexpr int kXmax = kAbort + 12;
  // row-sum exchange at the end of a unit: float [head][row][column half]
  static constexpr int kXsum = kXmax + 2 * 2 * kPreTileQ * 2 * 4;
  static constexpr int kBytes = kXsum + 2 * kPreTileQ * 2 * 4 + 1024;
};

// ---- programmatic dependent launch ---------------------------------------------------------
// Every kernel (but the prefill kernels on integer caches, see launch_prefill_t) is launched
// so that it may start while its predecessor in the stream is still finishing: its launch
// and prologue (barrier set-up, TMEM allocation) overlap the predecessor's tail. Each kernel
// calls pdl_wait() on every path before it first touches memory that an earlier kernel
// reads or writes; that wait returns once the predecessor has
// completed and its writes are visible, and since the predecessor waited for its own
// predecessor, completion is transitive along the stream. pdl_launch_dependents() lets the
// next kernel launch (its CTAs then sit in their own pdl_wait until this grid completes).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// A launch that may start before the previous kernel of the stream finishes (programmatic
// dependent launch): its blocks wait (griddepcontrol.wait) for that kernel's results. With
// pdl false an ordinary launch: the kernel starts once the previous one has finished.
template <typename... KArgs, typename... Actual>
inline cudaError_t launch_pdl_if(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, Actual&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Actual&&>(args)...);
}
template <typename... KArgs, typename... Actual>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Actual&&... args) {
  return launch_pdl_if(true, kernel, grid, block, smem, s, static_cast<Actual&&>(args)...);
}

// ---- the prefill kernels' persistent unit order ----
// Unit k of this CTA. Units are dealt out in rounds of gridDim.x, alternately in CTA order
// and in reverse; with the units sorted by decreasing cost this pairs a CTA's expensive
// units with cheap ones, and the per-CTA totals come out close to those of the greedy
// longest-first assignment (a plain round robin gives the first CTAs the most work in
// every round). Strictly increasing in k, so a CTA's loop ends at its first unit past the
// end.
__device__ __forceinline__ int snake_unit(int k, int g) {
  return k * g + ((k & 1) ? g - 1 - (int)blockIdx.x : (int)blockIdx.x);
}

// CTAs of a prefill grid that take units: the planner's share when it split the SMs
// between the prefill and the decode kernels of one call, else the whole grid
__device__ __forceinline__ int prefill_ctas(const Args& a) {
  const int p = a.split_sms ? a.hdr->pre_ctas : 0;
  return p > 0 && p < (int)gridDim.x ? p : (int)gridDim.x;
}

// the record of unit u (all zeros past the end)
__device__ __forceinline__ PrefillTile load_tile(const Args& a, int u, int n_units, int units_per_tile) {
  if (u >= n_units) return PrefillTile{};
  return a.tiles[u / units_per_tile];
}

// TMEM column (relative to S) of P for the 16 keys of block kk of a 128-key tile: the P of
// keys [32c, 32c + 32) replaces the S columns of those keys, hi pairs in the first 16
// columns and lo pairs (bf16) in the last 16.
__device__ __forceinline__ uint32_t p_col(int kk) { return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8); }

// ---- host launchers, one per kernel family (defined next to their kernels) -----------------
cudaError_t launch_plan(const Args& a, cudaStream_t s);
cudaError_t launch_cache_write(const Args& a, int sms, cudaStream_t s);
cudaError_t launch_decode_prep(const Args& a, cudaStream_t s);
cudaError_t launch_v_mirror(const Args& a, int grid, cudaStream_t s);
cudaError_t launch_prefill(const Args& a, bool bf16, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& tvm, int seg, int grid, cudaStream_t s);
cudaError_t launch_prefill256(const Args& a, bool bf16, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, const CUtensorMap& tvm, int seg, int grid, cudaStream_t s);
cudaError_t launch_decode(const Args& a, bool bf16, const CUtensorMap& tk, const CUtensorMap& tv, int seg,
                          cudaStream_t s);

// ---- small device helpers -----------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float fast_exp2(float x) {  // MUFU.EX2 (ex2.approx, flush-to-zero)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {  // lo -> bits 0..15
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// Two bf16 values (bits 0..15 and 16..31) as two fp16 values in the same positions:
// exact for magnitudes in [2^-14, 65504]; below that fp16 keeps fewer bits (absolute error
// at most 2^-25); from 65520 up the result is inf, and NaN stays NaN.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
  uint32_t h;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi), "f"(lo));
  return h;
}

// per-half unsigned maximum of two 16-bit pairs
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// p as two bf16 values hi + lo with hi = bf16(p), lo = bf16(p - hi): their sum carries
// about 16 significant bits, so P V computed as hi V + lo V keeps the softmax weights'
// rounding error near 2^-17 instead of bf16's 2^-9.
__device__ __forceinline__ void split_bf16x2(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// ---- packed fp32 pairs (two lanes of arithmetic per instruction) ----
__device__ __forceinline__ uint64_t f2_make(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// 32 bytes (8 words) to global memory in one store; dst 32-byte aligned
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// atomic add with acquire-release semantics at GPU scope; returns the old value
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void red_add_release_gpu(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// x[0..7] times sigmoid of the 8 gate values (T) at g (16-byte aligned): x / (1 + e^-gate)
template <bool BF16>
__device__ __forceinline__ void apply_gate8(const uint16_t* g, float* x) {
  const uint4 w = __ldg(reinterpret_cast<const uint4*>(g));
  const uint32_t gw[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint32_t b = (gw[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
    const float gf = BF16 ? __uint_as_float(b << 16) : __half2float(__ushort_as_half((unsigned short)b));
    x[e] = x[e] / (1.f + __expf(-gf));
  }
}

// one lane of the (fully active) warp, chosen by the hardware; the rest of the warp skips
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .b32 r;\n .reg .pred p;\n elect.sync r|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred != 0;
}

// ---- mbarrier ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a pipeline wait gives up after ~2 s

// Wait for the phase of parity `parity` to complete, at most ~2 s. On time-out (or when
// another thread of the CTA already gave up, *abort != 0) it sets *abort and the
// PA_DEVERR_TIMEOUT bit and returns false; callers then skip their remaining waits so
// the CTA drains and exits instead of hanging.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        atomicOr(err, PA_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Wait until the counter at p reaches need (acquire at gpu scope), at most ~2 s: on time-out
// (or when another thread of the CTA already gave up, *abort != 0) it sets *abort and the
// PA_DEVERR_TIMEOUT bit and returns false.
__device__ __forceinline__ bool wait_count_acquire_gpu(const int* p, int need, volatile int* abort, uint32_t* err) {
  if (ld_acquire_gpu(p) >= need) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (ld_acquire_gpu(p) >= need) return true;
    if ((it & 15) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        atomicOr(err, PA_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}
// barrier `id` (1..15) among `count` threads (a multiple of 32)
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMA ----------------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// bring a tile into L2 ahead of its load (no shared memory, no barrier)
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y)
               : "memory");
}
// ---- integer cache codes to fp16 pairs (exact: the codes are small integers) ---------------
// A biased code u (INT8: code + 128, INT4: code + 8) placed in the low bits of an fp16 with
// the bit pattern 0x6400 (1024.0) reads 1024 + u; subtracting 1024 + bias leaves the code.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// (a & mask) | 0x64006400 in one instruction
__device__ __forceinline__ uint32_t nib_pair_f16(uint32_t a) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(0x000F000Fu), "r"(0x64006400u));
  return r;
}
constexpr uint32_t kF16Magic = 0x64646464u;   // fp16 high bytes 0x64
constexpr uint32_t kF16Int8Bias = 0x64806480u; // 1152.0 (1024 + 128) in both halves
constexpr uint32_t kF16Int4Bias = 0x64086408u; // 1032.0 (1024 + 8)

// four INT8 codes (bytes 0..3 of w) as fp16 pairs (byte 0, byte 1) and (byte 2, byte 3)
// four INT8 codes (bytes 0..3 of w) as the exact fp16 integers code + 1152, pairs (byte 0,
// byte 1) and (byte 2, byte 3): the bias is left in (a constant per query row once summed
// against the query, which the softmax does not see)
__device__ __forceinline__ void s8x4_to_f16_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;
  lo = prmt(x, kF16Magic, 0x5140u);
  hi = prmt(x, kF16Magic, 0x7362u);
}
// byte i of w0 and byte i of w1 (two keys, one channel) as one fp16 pair, i = 0..3, as the
// exact fp16 integers code + 1152 (the consumer takes the offset off)
__device__ __forceinline__ void s8_key_pairs_biased(uint32_t w0, uint32_t w1, uint32_t (&p)[4]) {
  const uint32_t x0 = w0 ^ 0x80808080u, x1 = w1 ^ 0x80808080u;
  const uint32_t a = prmt(x0, x1, 0x5140u), b = prmt(x0, x1, 0x7362u);  // interleaved by key
  p[0] = prmt(a, kF16Magic, 0x5140u);
  p[1] = prmt(a, kF16Magic, 0x7362u);
  p[2] = prmt(b, kF16Magic, 0x5140u);
  p[3] = prmt(b, kF16Magic, 0x7362u);
}
// eight INT4 codes as fp16 subnormals: (code + 8) 2^-24 (the bits of code + 8 as the fp16
// bits), pairs (0, 4), (1, 5), (2, 6), (3, 7); the decode kernel's form. The offset, 8 units
// of 2^-24 per channel, is of the codes' own size (so fp32 sums keep it to rounding), and
// the kernel takes it off the scores' row constant and the output.
__device__ __forceinline__ void s4x8_to_f16_sub(uint32_t w, uint32_t (&p)[4]) {
  const uint32_t x = w ^ 0x88888888u;
  p[0] = x & 0x000F000Fu;
  p[1] = (x >> 4) & 0x000F000Fu;
  p[2] = (x >> 8) & 0x000F000Fu;
  p[3] = (x >> 12) & 0x000F000Fu;
}
// channel i of w0 and channel i of w1 (two keys) as one fp16 pair of subnormals (code + 8) 2^-24
__device__ __forceinline__ void s4_key_pairs_sub(uint32_t w0, uint32_t w1, uint32_t (&p)[8]) {
  const uint32_t x0 = w0 ^ 0x88888888u, x1 = w1 ^ 0x88888888u;
  const uint32_t a = prmt(x0, x1, 0x6420u);
  const uint32_t b = prmt(x0, x1, 0x7531u);
  p[0] = a & 0x000F000Fu;
  p[1] = (a >> 4) & 0x000F000Fu;
  p[4] = (a >> 8) & 0x000F000Fu;
  p[5] = (a >> 12) & 0x000F000Fu;
  p[2] = b & 0x000F000Fu;
  p[3] = (b >> 4) & 0x000F000Fu;
  p[6] = (b >> 8) & 0x000F000Fu;
  p[7] = (b >> 12) & 0x000F000Fu;
}

// The converter warps' work on one K or V tile of an integer cache: row r's code bytes sit
// at the start of the 128-byte row r of the tile's last slab (128-byte swizzle: 16-byte
// chunk j at position j ^ (r & 7)); they become the row's HS fp16 values at row r of every
// slab, as exact fp16 integers. (Leaving the conversion's offset in V, a constant to take off
// the normalised output, would save an instruction per pair, but the offset multiplies the
// difference between the fp16 weights the MMA sums and the fp32 row sum that normalises them:
// about 1152 * 2^-12 of a code. So V is exact, like K.) Each lane takes one 16-byte code chunk
// (16 INT8 or 32 INT4 channels) of a row in each of UNR rounds, reading all of them before
// writing any, so only a row's own codes are overwritten and only after the whole warp has
// read them. cw: this converter warp (0 or 1). With SUB (the 128-wide kernel's K tiles) the
// codes become the fp16 subnormals (code + 128) 2^-24 (INT4: (code + 8) 2^-24), the bits of
// the biased code as the fp16's bits: no subtraction; the offset adds a constant per query
// row to its scores, which the softmax does not see and the exported lse has taken off.
template <int HS, int KQ, bool SUB = false>
__device__ __forceinline__ void convert_code_tile(uint8_t* tile, int cw, int lane) {
  constexpr int RB = KQ == 1 ? HS : HS / 2;                       // code bytes per row
  constexpr int CH = RB / 16;                                      // code chunks per row
  constexpr int ROWS = 32 / CH;                                    // rows per warp round
  constexpr int CODES = KQ == 1 ? 16 : 32;                         // channels per code chunk
  constexpr int SLAB = (HS / 64 - 1) * kPreTileK * 128;            // the slab the codes land in
  constexpr int UNR = 4;                                           // rounds read before writing
  static_assert(kPreTileK % (2 * ROWS * UNR) == 0, "rounds per tile");
  const int rr = lane / CH, j = lane % CH;
#pragma unroll 1
  for (int r0 = cw * ROWS * UNR; r0 < kPreTileK; r0 += 2 * ROWS * UNR) {
    uint4 c[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = r0 + u * ROWS + rr;
      c[u] = *reinterpret_cast<const uint4*>(tile + SLAB + r * 128 + ((j ^ (r & 7)) << 4));
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = r0 + u * ROWS + rr;
      const uint32_t w[4] = {c[u].x, c[u].y, c[u].z, c[u].w};
      uint32_t f[CODES / 2];  // fp16 pairs of consecutive channels
      if constexpr (KQ == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // channels 4i .. 4i + 3 of the chunk
          const uint32_t x = w[i] ^ 0x80808080u;
          if constexpr (SUB) {
            f[2 * i] = prmt(x, 0u, 0x4140u);
            f[2 * i + 1] = prmt(x, 0u, 0x4342u);
          } else {
            f[2 * i] = hsub2_u32(prmt(x, kF16Magic, 0x5140u), kF16Int8Bias);
            f[2 * i + 1] = hsub2_u32(prmt(x, kF16Magic, 0x7362u), kF16Int8Bias);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // channels 8i .. 8i + 7: byte b holds 2b (low), 2b + 1 (high)
          const uint32_t x = w[i] ^ 0x88888888u, x4 = x >> 4;
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const uint32_t nib = prmt(x, x4, (uint32_t)(b | ((4 + b) << 8)));
            f[4 * i + b] = SUB ? nib & 0x000F000Fu : hsub2_u32(nib_pair_f16(nib), kF16Int4Bias);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < CODES / 8; ++q) {  // 8 channels per 16-byte fp16 chunk
        const int ch = CODES * j + 8 * q;
        const int cc = (ch & 63) >> 3;
        *reinterpret_cast<uint4*>(tile + (ch >> 6) * (kPreTileK * 128) + r * 128 + ((cc ^ (r & 7)) << 4)) =
            make_uint4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
      }
    }
  }
}

// one 128-byte line of global memory into L2 (a hint: no data returned, no fault)
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- warp-level tensor core path (decode) -------------------------------------------------
// the 8 x 8 16-bit matrix held one row pair per thread (thread 4i + j: row i, columns 2j,
// 2j + 1), transposed
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
template <bool BF16>
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// ---- tcgen05 (5th-generation tensor cores, tensor memory) ------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {  // whole warp
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive on `bar` once every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand (the layout TMA writes
// with CU_TENSOR_MAP_SWIZZLE_128B: rows of 128 bytes, 16-byte chunks XOR-permuted by row % 8,
// 8-row atoms of 1024 bytes). lbo / sbo are the byte strides between atoms along the
// leading / strided dimension. Bits: start >> 4 [0,14), lbo >> 4 [16,30), sbo >> 4 [32,46),
// version 1 at bit 46, layout SWIZZLE_128B (2) at [61,64).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma.kind::f16 with fp32 accumulation: D format F32 at
// bit 4, A/B format (0 f16, 1 bf16) at bits 7 / 10, B major-ness (0 K-major, 1 MN-major) at
// bit 16, N >> 3 at bits [17,23), M >> 4 at bits [24,29).
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int M, int N, bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// tcgen05.ld 32x32b.x32: this thread's TMEM lane, 32 consecutive 32-bit columns from taddr;
// the wait is in the same asm so the registers are valid when it returns.
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// tcgen05.ld 32x32b.x64: this thread's TMEM lane, 64 consecutive 32-bit columns from taddr;
// the wait is in the same asm so the registers are valid when it returns.
__device__ __forceinline__ void tmem_ld_x64(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

// tcgen05.st 32x32b.x32: 32 consecutive 32-bit columns of this thread's TMEM lane; waits for completion.
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n"
      "tcgen05.wait::st.sync.aligned;\n"
      :
      : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Four tcgen05.ld 32x32b.x32 (128 consecutive columns of this thread's TMEM lane) and one
// wait, in a single asm so the registers are valid when it returns.
__device__ __forceinline__ void tmem_ld_x128(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%128+0];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%128+32];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95}, [%128+64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128+96];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
}

// tcgen05.st 32x32b.x32 without waiting (the source registers are read at issue); pair with
// tmem_wait_st before the stored columns are handed to another thread.
__device__ __forceinline__ void tmem_st_x32_nowait(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n"
      :
      : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// tcgen05.st 32x32b.x8 of eight registers without waiting (see tmem_st_x32_nowait)
__device__ __forceinline__ void tmem_st_x8_nowait(uint32_t taddr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3,
                                                  uint32_t r4, uint32_t r5, uint32_t r6, uint32_t r7) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"r"(taddr), "r"(r0),
               "r"(r1), "r"(r2), "r"(r3), "r"(r4), "r"(r5), "r"(r6), "r"(r7)
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// three-input max / min (sm_100+)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

}  // namespace pa
