// Prefill / chunked-prefill attention for 256-wide heads on the 5th-generation tensor cores.
//
// Same operation, tile records and unit order as the 128/64-wide kernel; what changes is how
// the tensor memory and shared memory are spent. One head's O (128 rows x 256 fp32 columns)
// takes half of the 512 TMEM columns, so a unit is 128 query rows of ONE head, and the other
// half holds two S buffers used by alternate KV tiles: while the softmax works on tile t in
// one buffer, the tensor core computes S of tile t + 1 into the other, then O += P_t V_t.
// MMA order: S_0, S_1, O += P_0 V_0, S_2, O += P_1 V_1, ..., O += P_{n-1} V_{n-1}.
//
// Shared memory: the query tile (64 KB) stays for the whole unit; K and V stream through a
// ring of four 32 KB chunks, a chunk being 128 keys x 128 of the 256 columns (two 64-column
// slabs, 128-byte swizzle), loaded in the order the MMA consumes them (K_t as two chunks,
// then V_{t-1} as two chunks), each chunk released by the commit of the MMAs that read it.
// Q K^T runs as 16 k-steps over the two K chunks; P V as two N = 128 halves of O, one per V
// chunk.
//
// Roles (384 threads):
//   warp 0      TMA producer: Q (four 64-column boxes), then the K/V chunks page segment by
//               page segment through block_table; segments past the sequence read as zeros.
//   warp 1      TMEM owner and MMA issuer (one elected thread).
//   warps 2..9  softmax: two warps per TMEM lane quarter, each thread half (64 columns) of
//               a query row, exactly as in the 128-wide kernel (masking, partner max exchange,
//               lazy rescale with threshold 2^8, P over S as fp16, or bf16 hi + lo against
//               bf16 V); at the end of the unit each thread normalises and stores its 128 of
//               the row's 256 output columns.
//   warps 10,11 idle (the block is a whole number of warpgroups); with integer caches they
//               turn the code rows of each chunk into fp16 in place, as the converters of the
//               128-wide kernel do (a chunk's 128 channels are 128 INT8 or 64 INT4 code bytes
//               of each key row, landed in the chunk's second slab).
#include "common.cuh"

namespace pa {
namespace {

constexpr int kHS = 256;
constexpr int kThreads = 384;
constexpr int kSoftWarps = 8;
constexpr int kChunks = 4;          // K/V ring depth, in 32 KB chunks
constexpr uint32_t kCols = 512;     // S buffers at columns 0 and 128, O at 256..511
constexpr uint32_t kOCol = 256;

struct Smem {
  static constexpr int kSlab = kPreTileK * 128;    // 128 rows x 64 columns of 16-bit values
  static constexpr int kChunkBytes = 2 * kSlab;    // 128 rows x 128 columns
  static constexpr int kQ = 0;                     // four slabs
  static constexpr int kCh0 = kQ + 4 * kSlab;
  static constexpr int kBars = kCh0 + kChunks * kChunkBytes;
  // q_full, q_empty, ch_full[kChunks], ch_empty[kChunks], s_full[2], p_full, o_done, o_free,
  // integer caches: chc_full[kChunks] (a chunk's code rows landed)
  static constexpr int kNumBars = 2 + 2 * kChunks + 2 + 3 + kChunks;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kPreCtas = kAbort + 4;  // CTAs of the grid that take units
  // row-max exchange between the two warps of a lane quarter: float [tile parity][row][half]
  static constexpr int kXmax = (kPreCtas + 4 + 15) / 16 * 16;
  // row-sum exchange at the end of a unit: float [row][half]
  static constexpr int kXsum = kXmax + 2 * kPreTileQ * 2 * 4;
  static constexpr int kBytes = kXsum + kPreTileQ * 2 * 4 + 1024;  // + alignment slack
};
static_assert(Smem::kBytes <= 232448, "shared memory of one CTA");
static_assert(kPreTileQ == 128 && kPreTileK == 128, "tile shape");

template <bool BF16, int KQ>
__global__ void __launch_bounds__(kThreads, 1)
    prefill256_kernel(const Args a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmVm,
                      const int seg_rows) {
  using L = Smem;
  // the MMA operand type: T, except on integer caches (fp16 scaled queries and fp16 codes);
  // BF16 is the type of the output
  constexpr bool MB = BF16 && KQ == 0;
  constexpr int RB = KQ == 1 ? kHS : kHS / 2;  // code bytes of one KV head's row
  constexpr uint32_t IDESC_QK = idesc_f16(MB, kPreTileQ, kPreTileK, false);
  constexpr uint32_t IDESC_PV = idesc_f16(MB, kPreTileQ, 128, true);
  constexpr uint32_t IDESC_PV16 = idesc_f16(false, kPreTileQ, 128, true);  // fp16 P times the fp16 V copy

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* ch_full = bars + 2;
  uint64_t* ch_empty = bars + 2 + kChunks;
  uint64_t* s_full = bars + 2 + 2 * kChunks;  // [S buffer]
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = s_full + 3;
  uint64_t* o_free = s_full + 4;
  uint64_t* chc_full = s_full + 5;  // [kChunks]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);
  uint32_t* err = &a.hdr->error;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < kChunks; ++i) {
      mbar_init(&ch_full[i], KQ ? 2 : 1);  // (integer caches: the two converter warps)
      mbar_init(&ch_empty[i], 1);
      mbar_init(&chc_full[i], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, 32 * kSoftWarps);
    mbar_init(o_done, 1);
    mbar_init(o_free, 32 * kSoftWarps);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the work list, caches and V copy written by the earlier kernels of this call
  pdl_launch_dependents();

  // bf16: V from the fp16 copy unless the planner found no room for it or the copy met a
  // value fp16 cannot hold (then bf16 V, P as hi + lo)
  const bool v16 = MB && a.hdr->v_mirror && !a.hdr->v_mirror_bad;
  const int units_per_tile = a.nh;  // one head per unit
  // units dealt to the CTAs that take work; the others (the planner gave their SMs to the
  // decode kernel of this call) run no loop and release their TMEM at once
  // (the count is kept in shared memory and read where a unit index is formed: a register
  // held across the kernel pushes the softmax warps over their register budget)
  volatile int* pre_ctas = reinterpret_cast<volatile int*>(smem + L::kPreCtas);
  if (threadIdx.x == 0) *pre_ctas = prefill_ctas(a);
  __syncthreads();
  const int n_units = (int)blockIdx.x < *pre_ctas ? a.hdr->n_prefill_tiles * units_per_tile : 0;
  const int64_t cache_rows = (int64_t)a.num_blocks * a.bs;

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      if (v16) tma_prefetch_desc(&tmVm);
    }
    const int nseg = kPreTileK / seg_rows;
    uint32_t gc = 0, unit_cnt = 0;
    PrefillTile next = load_tile(a, snake_unit(0, *pre_ctas), n_units, units_per_tile);
    PrefillTile next2 = load_tile(a, snake_unit(1, *pre_ctas), n_units, units_per_tile);
    for (int u = snake_unit(0, *pre_ctas); u < n_units; u = snake_unit(++unit_cnt, *pre_ctas)) {
      const PrefillTile tile = next;
      next = next2;
      const int un = snake_unit(unit_cnt + 1, *pre_ctas);
      next2 = load_tile(a, snake_unit(unit_cnt + 2, *pre_ctas), n_units, units_per_tile);
      const int h = u % units_per_tile, g = h / a.G;
      const int kv_len = tile.past + tile.q_len;
      const int n_kv = tile.n_kv;
      const int* bt = a.block_table + (int64_t)tile.b * a.max_blocks;
      if (lane == 0) {
        if (unit_cnt > 0) mbar_wait(q_empty, (unit_cnt - 1) & 1, abort, err);
        mbar_arrive_expect_tx(q_full, 4 * L::kSlab);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh)
          tma_load_2d(smem + L::kQ + hh * L::kSlab, &tmQ, q_full, h * kHS + hh * 64, tile.c0 + tile.j0);
        if (un < n_units) {  // the next unit's Q into L2 now, so its load at the boundary is short
          const int hn = un % units_per_tile;
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) tma_prefetch_l2_2d(&tmQ, hn * kHS + hh * 64, next.c0 + next.j0);
        }
      }
      // the two chunks of K (is_v false) or V of KV tile t
      auto emit = [&](bool is_v, int t) {
        int z = (int)cache_rows;  // past the end: zero fill
        int zv = v16 ? a.mirror_keys : z;
        if (lane < nseg) {
          const int key = t * kPreTileK + lane * seg_rows;
          if (key < kv_len) {
            const int blk = bt[key / a.bs];
            if (blk >= 0 && blk < a.num_blocks) z = blk * a.bs + key % a.bs;
            else if (!v16) atomicOr(err, PA_DEVERR_BAD_BLOCK);  // (the copy kernel flags it otherwise)
            zv = v16 ? tile.mirror_row0 + key : z;
          }
        }
        const CUtensorMap* map = is_v ? (v16 ? &tmVm : &tmV) : &tmK;
        const int row = is_v ? zv : z;
#pragma unroll
        for (int c = 0; c < 2; ++c, ++gc) {
          const int slot = gc % kChunks;
          const uint32_t ph = (gc / kChunks) & 1;
          if constexpr (KQ != 0) {  // the chunk's code rows (128 bytes from its channels' start)
            if (lane == 0) {
              mbar_wait(&ch_empty[slot], ph ^ 1, abort, err);
              mbar_arrive_expect_tx(&chc_full[slot], kPreTileK * 128);
            }
            __syncwarp();
            if (lane < nseg)
              tma_load_2d(smem + L::kCh0 + slot * L::kChunkBytes + L::kSlab + lane * seg_rows * 128, map,
                          &chc_full[slot], g * RB + c * (RB / 2), row);
            __syncwarp();
            continue;
          }
          if (lane == 0) {
            mbar_wait(&ch_empty[slot], ph ^ 1, abort, err);
            mbar_arrive_expect_tx(&ch_full[slot], L::kChunkBytes);
          }
          __syncwarp();
          if (lane < nseg) {
            uint8_t* dst = smem + L::kCh0 + slot * L::kChunkBytes + lane * seg_rows * 128;
            tma_load_3d(dst, map, &ch_full[slot], (2 * c) * 64, g, row);
            tma_load_3d(dst + L::kSlab, map, &ch_full[slot], (2 * c + 1) * 64, g, row);
          }
          __syncwarp();
        }
      };
      for (int t = 0; t < n_kv; ++t) {
        emit(false, t);
        if (t > 0) emit(true, t - 1);
      }
      emit(true, n_kv - 1);
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    // descriptors of the tile bases; an operand's descriptor is its base plus its byte
    // offset >> 4 (the start-address field never carries: shared addresses stay below 2^18)
    const uint64_t qdesc0 = sdesc_sw128(smem_u32(smem + L::kQ), 16, 1024);
    const uint64_t kdesc0 = sdesc_sw128(smem_u32(smem + L::kCh0), 16, 1024);
    const uint64_t vdesc0 = sdesc_sw128(smem_u32(smem + L::kCh0), L::kSlab, 1024);
    constexpr uint32_t kSlab16 = L::kSlab >> 4;
    uint32_t gc = 0, gs = 0, unit_cnt = 0;
    PrefillTile next = load_tile(a, snake_unit(0, *pre_ctas), n_units, units_per_tile);
    for (int u = snake_unit(0, *pre_ctas); u < n_units; u = snake_unit(++unit_cnt, *pre_ctas)) {
      const PrefillTile tile = next;  // loaded one unit ahead
      next = load_tile(a, snake_unit(unit_cnt + 1, *pre_ctas), n_units, units_per_tile);
      const int kv_len = tile.past + tile.q_len;
      const int n_kv = tile.n_kv;
      mbar_wait(q_full, unit_cnt & 1, abort, err);
      tc_fence_after();

      auto issue_qk = [&](int t) {
        const uint32_t gt = gs + t;
        const uint32_t d_tmem = tmem + (gt & 1) * 128u;
#pragma unroll
        for (int c = 0; c < 2; ++c, ++gc) {
          const int slot = gc % kChunks;
          mbar_wait(&ch_full[slot], (gc / kChunks) & 1, abort, err);
          tc_fence_after();
          if (elect_one()) {
            const uint64_t kd = kdesc0 + (uint64_t)((slot * L::kChunkBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              // k-step 8c + kk: Q slab 2c + kk / 4, K slab kk / 4 of the chunk, 32-byte step kk % 4
              const uint64_t qoff = (uint64_t)((2 * c + (kk >> 2)) * kSlab16 + (kk & 3) * 2);
              const uint64_t koff = (uint64_t)((kk >> 2) * kSlab16 + (kk & 3) * 2);
              tc_mma_ss(d_tmem, qdesc0 + qoff, kd + koff, IDESC_QK, (c | kk) ? 1u : 0u);
            }
            tc_commit(&ch_empty[slot]);
            if (c == 1) {
              tc_commit(&s_full[gt & 1]);
              if (t == n_kv - 1) tc_commit(q_empty);
            }
          }
          __syncwarp();
        }
      };
      auto issue_pv = [&](int t) {
        const uint32_t gt = gs + t;
        mbar_wait(p_full, gt & 1, abort, err);
        if (t == 0 && unit_cnt > 0) mbar_wait(o_free, (unit_cnt - 1) & 1, abort, err);
        const uint32_t p_tmem = tmem + (gt & 1) * 128u;
        const uint32_t acc0 = t > 0 ? 1u : 0u;
        const int valid = kv_len - t * kPreTileK;  // keys of this tile inside the sequence
#pragma unroll
        for (int c = 0; c < 2; ++c, ++gc) {
          const int slot = gc % kChunks;
          mbar_wait(&ch_full[slot], (gc / kChunks) & 1, abort, err);
          tc_fence_after();
          if (KQ == 0 && valid < kPreTileK) {  // (codes are finite)
            // keys past the sequence may be unwritten cache rows; P is 0 there but 0 * NaN
            // is not, so clear those V rows (whole 128-byte rows: the swizzle stays inside)
            uint8_t* vchunk = smem + L::kCh0 + slot * L::kChunkBytes;
            const int rows = kPreTileK - valid;
            for (int i = lane; i < rows * 8 * 2; i += 32) {
              const int hh = i / (rows * 8), rem = i % (rows * 8);
              const int r = valid + rem / 8, ch = rem % 8;
              *reinterpret_cast<uint4*>(vchunk + hh * L::kSlab + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
          const uint64_t vd = vdesc0 + (uint64_t)((slot * L::kChunkBytes) >> 4);
          const uint32_t d_tmem = tmem + kOCol + c * 128u;
          if (elect_one()) {
            // 16 keys of V per MMA (8-row atoms 1024 B apart), the chunk's two 64-column
            // slabs kSlab apart along N
            if (MB && !v16) {
#pragma unroll
              for (int kk = 0; kk < kPreTileK / 16; ++kk) {
                const uint64_t vdesc = vd + (uint64_t)(kk * ((16 * 128) >> 4));
                tc_mma_ts(d_tmem, p_tmem + p_col(kk), vdesc, IDESC_PV, kk > 0 ? 1u : acc0);
                tc_mma_ts(d_tmem, p_tmem + p_col(kk) + 16, vdesc, IDESC_PV, 1u);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < kPreTileK / 16; ++kk) {
                const uint64_t vdesc = vd + (uint64_t)(kk * ((16 * 128) >> 4));
                tc_mma_ts(d_tmem, p_tmem + p_col(kk), vdesc, BF16 ? IDESC_PV16 : IDESC_PV, kk > 0 ? 1u : acc0);
              }
            }
            tc_commit(&ch_empty[slot]);
            if (c == 1) tc_commit(o_done);
          }
          __syncwarp();
        }
      };

      for (int t = 0; t < n_kv; ++t) {
        issue_qk(t);
        if (t > 0) issue_pv(t - 1);
      }
      issue_pv(n_kv - 1);
      gs += n_kv;
    }
  } else if (warp < 2 + kSoftWarps) {
    // ======================= softmax =======================
    constexpr int COLS = kPreTileK / 2;  // score columns per thread
    constexpr int OCOLS = kHS / 2;       // output columns per thread
    const int sw = warp - 2;
    const int hsel = (sw >> 2) & 1;      // column half
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t o_tmem = tmem + lane_off + kOCol + hsel * OCOLS;
    float* xmax = reinterpret_cast<float*>(smem + L::kXmax);
    float* xsum = reinterpret_cast<float*>(smem + L::kXsum);
    const int pair_bar = 2 + quarter;  // named barrier of the two warps of this lane quarter
    uint32_t gs = 0;
    PrefillTile next = load_tile(a, snake_unit(0, *pre_ctas), n_units, units_per_tile);
    for (int k = 0, u = snake_unit(0, *pre_ctas); u < n_units; u = snake_unit(++k, *pre_ctas)) {
      const PrefillTile tile = next;  // loaded during the previous unit's epilogue
      const int h = u % units_per_tile;
      const int c0 = tile.c0, q_len = tile.q_len, past = tile.past;
      const int kv_len = past + q_len;
      const int n_kv = tile.n_kv;
      const int lim = min(past + tile.j0 + row, kv_len - 1);  // last key this row sees
      const int lim_tile0 = past + tile.j0;                   // the smallest limit of the unit
      // the softmax constant scale * log2(e); integer caches: times 2^E, the exponent the
      // cache-write stage took out of this row's scaled query (rows past the sequence: 1)
      float c = a.scale_log2;
      if constexpr (KQ != 0)
        if (tile.j0 + row < q_len) c = ldexpf(c, __ldg(a.qexp + (int64_t)(c0 + tile.j0 + row) * a.nh + h));
      float m_used = -INFINITY, l = 0.f;
      for (int t = 0; t < n_kv; ++t) {
        const uint32_t gt = gs + t;
        mbar_wait(&s_full[gt & 1], (gt >> 1) & 1, abort, err);
        tc_fence_after();
        const uint32_t s_base = tmem + lane_off + (gt & 1) * 128u;
        const int key0 = t * kPreTileK + hsel * COLS;  // first key of this thread's columns
        const bool masked = (t * kPreTileK + kPreTileK - 1 > lim_tile0) || (t * kPreTileK + kPreTileK > kv_len);
        uint32_t r[COLS];
        tmem_ld_x64(s_base + hsel * COLS, r);
        // keys past this row's limit become -inf for s * c (so both the max and exp2 ignore them)
        const float sentinel = c > 0.f ? -INFINITY : INFINITY;
        if (masked) {
#pragma unroll
          for (int e = 0; e < COLS; ++e)
            if (key0 + e > lim) r[e] = __float_as_uint(sentinel);
        }
#ifdef PA_COVERAGE
        if (tile.j0 + row < q_len)
          for (int e = 0; e < COLS; ++e)
            if (!(masked && key0 + e > lim)) cov_count(a, c0 + tile.j0 + row, h, key0 + e);
#endif
        // ---- the row's max of s * c, on raw s (max, or min for c < 0), four chains ----
        float mc[4] = {sentinel, sentinel, sentinel, sentinel};
        if (c > 0.f) {
#pragma unroll
          for (int e = 0; e < COLS; e += 8)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              mc[q] = fmax3(mc[q], __uint_as_float(r[e + 2 * q]), __uint_as_float(r[e + 2 * q + 1]));
        } else {
#pragma unroll
          for (int e = 0; e < COLS; e += 8)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              mc[q] = fmin3(mc[q], __uint_as_float(r[e + 2 * q]), __uint_as_float(r[e + 2 * q + 1]));
        }
        const float mr = c > 0.f ? fmax3(fmaxf(mc[0], mc[1]), mc[2], mc[3]) : fmin3(fminf(mc[0], mc[1]), mc[2], mc[3]);
        float* xm = xmax + (gt & 1) * (kPreTileQ * 2) + row * 2;
        xm[hsel] = mr * c;
        named_bar_sync(pair_bar, 64);
        const float m_tile = fmaxf(xm[0], xm[1]);
        const float m_new = fmaxf(m_used, m_tile);
        const bool any_grow = __any_sync(0xffffffffu, m_new > m_used + 8.0f);  // first tile: m_used = -inf
        float alpha = 1.f;
        if (any_grow) {
          alpha = fast_exp2(m_used - m_new);  // 0 on the first tile; 1 where m_new == m_used
          m_used = m_new;
          l *= alpha;
        }
        // ---- P = exp2(s * c - m) over S, 16 keys at a time ----
        const float neg_m = -m_used;
        if constexpr (MB) {
          float lc[2] = {0.f, 0.f};
          if (!v16) {
#pragma unroll
            for (int g2 = 0; g2 < COLS / 16; ++g2) {
              uint32_t* q = r + g2 * 16;
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float p0 = fast_exp2(fmaf(__uint_as_float(q[2 * e]), c, neg_m));
                const float p1 = fast_exp2(fmaf(__uint_as_float(q[2 * e + 1]), c, neg_m));
                lc[0] += p0;
                lc[1] += p1;
                split_bf16x2(p0, p1, q[2 * e], q[2 * e + 1]);
              }
              const int kk = hsel * (COLS / 16) + g2;  // 16-key block of the tile
              tmem_st_x8_nowait(s_base + p_col(kk), q[0], q[2], q[4], q[6], q[8], q[10], q[12], q[14]);
              tmem_st_x8_nowait(s_base + p_col(kk) + 16, q[1], q[3], q[5], q[7], q[9], q[11], q[13], q[15]);
            }
          } else {
#pragma unroll
            for (int g2 = 0; g2 < COLS / 16; ++g2) {
              uint32_t* q = r + g2 * 16;
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float p0 = fast_exp2(fmaf(__uint_as_float(q[2 * e]), c, neg_m));
                const float p1 = fast_exp2(fmaf(__uint_as_float(q[2 * e + 1]), c, neg_m));
                lc[0] += p0;
                lc[1] += p1;
                q[2 * e] = pack2<false>(p0, p1);
              }
              const int kk = hsel * (COLS / 16) + g2;
              tmem_st_x8_nowait(s_base + p_col(kk), q[0], q[2], q[4], q[6], q[8], q[10], q[12], q[14]);
            }
          }
          l += lc[0] + lc[1];
        } else {
          const uint64_t c2 = f2_make(c, c), nm2 = f2_make(neg_m, neg_m);
          uint64_t lsum[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
#pragma unroll
          for (int g2 = 0; g2 < COLS / 16; ++g2) {
            uint32_t* q = r + g2 * 16;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              float x0, x1;
              f2_split(f2_fma(f2_make(__uint_as_float(q[2 * e]), __uint_as_float(q[2 * e + 1])), c2, nm2), x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              lsum[e & 1] = f2_add(lsum[e & 1], f2_make(p0, p1));
              q[2 * e] = pack2<false>(p0, p1);
            }
            const int kk = hsel * (COLS / 16) + g2;
            tmem_st_x8_nowait(s_base + p_col(kk), q[0], q[2], q[4], q[6], q[8], q[10], q[12], q[14]);
          }
          float a0, a1, b0, b1;
          f2_split(lsum[0], a0, a1);
          f2_split(lsum[1], b0, b1);
          l += (a0 + b0) + (a1 + b1);
        }
        tmem_wait_st();
        if (t > 0) {
          // O holds P_0..P_{t-2} V; wait for P_{t-1} V before rescaling it
          mbar_wait(o_done, (gt - 1) & 1, abort, err);
          if (any_grow) {
            tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < OCOLS; cc += 32) {
              uint32_t ov[32];
              tmem_ld_x32(o_tmem + cc, ov);
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
              tmem_st_x32(o_tmem + cc, ov);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(p_full);
      }
      // ---- epilogue: wait for the last P V, normalise, store the valid rows ----
      next = load_tile(a, snake_unit(k + 1, *pre_ctas), n_units, units_per_tile);
      mbar_wait(o_done, (gs + n_kv - 1) & 1, abort, err);
      tc_fence_after();
      {
        float* xs = xsum + row * 2;
        xs[hsel] = l;
        named_bar_sync(pair_bar, 64);
        const float l_row = xs[0] + xs[1];
        const float inv = 1.f / l_row;
        const bool store = tile.j0 + row < q_len;
        const int64_t orow = (int64_t)(c0 + tile.j0 + row) * a.nh + h;
        if (a.lse && store && hsel == 0)  // natural log; m_used is the base-2 max of s * scale
          a.lse[orow] = (m_used + fast_log2(l_row)) * 0.69314718055994531f;
        // this thread's 128 output columns, packed to 16-bit pairs, then O is released
        uint32_t pk[OCOLS / 2];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t ov[64];
          tmem_ld_x64(o_tmem + half * 64, ov);
          if constexpr (KQ != 0) {
            // integer caches: O holds sum p code over the V codes; the row's output is O / l
            // times the V scale of each channel (then the gate), 8 at a time
            const float4* vs =
                reinterpret_cast<const float4*>(a.v_scale + (h / a.G) * kHS + hsel * OCOLS + half * 64);
#pragma unroll
            for (int v = 0; v < 64; v += 8) {
              const float4 s0 = __ldg(vs + v / 4), s1 = __ldg(vs + v / 4 + 1);
              const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
              float x[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(ov[v + e]) * inv * sv[e];
              if (store && a.gate) apply_gate8<BF16>(a.gate + orow * kHS + hsel * OCOLS + half * 64 + v, x);
#pragma unroll
              for (int e = 0; e < 8; e += 2) pk[half * 32 + (v + e) / 2] = pack2<BF16>(x[e], x[e + 1]);
            }
            continue;
          }
          if (store && a.gate) {  // output gate: times sigmoid(gate), elementwise
            const uint16_t* gsrc = a.gate + orow * kHS + hsel * OCOLS + half * 64;
#pragma unroll
            for (int v = 0; v < 64; v += 8) apply_gate8<BF16>(gsrc + v, reinterpret_cast<float*>(ov + v));
          }
#pragma unroll
          for (int v = 0; v < 32; ++v)
            pk[half * 32 + v] = pack2<BF16>(__uint_as_float(ov[2 * v]) * inv, __uint_as_float(ov[2 * v + 1]) * inv);
        }
        tc_fence_before();
        mbar_arrive(o_free);
        if (store) {
          uint16_t* dst = reinterpret_cast<uint16_t*>(a.output) + orow * kHS + hsel * OCOLS;
          if (a.out_v8) {
#pragma unroll
            for (int v = 0; v < OCOLS / 2; v += 8) st_global_v8(dst + 2 * v, &pk[v]);
          } else {
#pragma unroll
            for (int v = 0; v < OCOLS / 2; v += 4)
              *reinterpret_cast<uint4*>(dst + 2 * v) = make_uint4(pk[v], pk[v + 1], pk[v + 2], pk[v + 3]);
          }
        }
      }
      gs += n_kv;
    }
  }

  if constexpr (KQ != 0) {
    if (warp >= 2 + kSoftWarps) {
      // ======================= converters: warps 10, 11 (integer caches) =======================
      // the chunks in the producer's order: 4 per KV tile (K_t's two, V_{t-1}'s two, ...)
      const int cw = warp - (2 + kSoftWarps);
      uint32_t gc = 0, unit_cnt = 0;
      for (int u = snake_unit(0, *pre_ctas); u < n_units; u = snake_unit(++unit_cnt, *pre_ctas)) {
        const int chunks = 4 * load_tile(a, u, n_units, units_per_tile).n_kv;
        for (int i = 0; i < chunks; ++i, ++gc) {
          const int slot = gc % kChunks;
          mbar_wait(&chc_full[slot], (gc / kChunks) & 1, abort, err);
          convert_code_tile<128, KQ>(smem + L::kCh0 + slot * L::kChunkBytes, cw, lane);
          fence_proxy_async_smem();  // (the MMA reads the chunk through the async proxy)
          __syncwarp();
          if (lane == 0) mbar_arrive(&ch_full[slot]);
        }
      }
    }
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

template <bool BF16, int KQ>
cudaError_t launch_t(const Args& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const CUtensorMap& tvm, int seg, int grid, cudaStream_t s) {
  constexpr int smem = Smem::kBytes;
  cudaError_t e =
      cudaFuncSetAttribute(prefill256_kernel<BF16, KQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // (integer caches: after the quantizing cache write has finished, as the 128-wide kernel)
  return launch_pdl_if(KQ == 0, prefill256_kernel<BF16, KQ>, dim3(grid), dim3(kThreads), smem, s, a, tq, tk, tv,
                       tvm, seg);
}

template <int KQ>
cudaError_t launch_kq(const Args& a, bool bf16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tvm, int seg, int grid, cudaStream_t s) {
  return bf16 ? launch_t<true, KQ>(a, tq, tk, tv, tvm, seg, grid, s)
              : launch_t<false, KQ>(a, tq, tk, tv, tvm, seg, grid, s);
}

}  // namespace

cudaError_t launch_prefill256(const Args& a, bool bf16, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, const CUtensorMap& tvm, int seg, int grid, cudaStream_t s) {
  if (a.kvq == 1) return launch_kq<1>(a, bf16, tq, tk, tv, tvm, seg, grid, s);
  if (a.kvq == 2) return launch_kq<2>(a, bf16, tq, tk, tv, tvm, seg, grid, s);
  return launch_kq<0>(a, bf16, tq, tk, tv, tvm, seg, grid, s);
}

}  // namespace pa
