// Prefill / chunked-prefill attention on the 5th-generation tensor cores.
//
// Work unit: 128 query rows [j0, j0 + 128) of one sequence for two query heads A, B of
// the same KV head (grouped-query heads share K and V, so both heads consume every K/V
// tile the CTA loads; with an odd group size a unit is one head). Rows never straddle
// sequences; rows past the sequence end are computed and not stored. The unit walks the
// 128-key KV tiles 0 .. ceil((past + last row + 1) / 128) - 1 of its sequence
// (bottom-right causal: row j sees keys 0 .. past + j) with the online softmax of
// FlashAttention.
//
// Roles (640 threads, persistent over the planner's tile list, longest tiles first):
//   warp 0      TMA producer: the two Q tiles once per unit (2-D map over the query rows),
//               then K and V tiles into a 2-deep ring, each tile gathered page segment by
//               page segment through block_table (3-D map over (head_size, kv_heads,
//               slots), 128-byte swizzle). Segments past the sequence read as zeros.
//   warp 1      TMEM owner and MMA issuer (one thread), in the order
//                 S_A = Q_A K_t^T, O_B += P_B V_{t-1}, S_B = Q_B K_t^T, O_A += P_A V_t, ...
//               so the tensor core works on one head while the other head's softmax runs.
//               Q K^T takes both operands from shared memory; P V takes P from TMEM
//               (where the softmax wrote it over S) and V from shared memory; fp32
//               accumulators in TMEM.
//   warps 2..9  softmax of head A, warps 10..17 softmax of head B: two warps per TMEM lane
//               quarter, so each thread owns half (64 columns) of query row (TMEM lane) i.
//               Per tile: one 64-column TMEM load, keys past the row's causal limit replaced
//               by -inf, the partial row max (three-input max on four independent chains)
//               exchanged with the partner warp through shared memory, the running max
//               update (O is rescaled only when the
//               max grew by more than 2^8, exact because the final division uses the same
//               stale max), then P = exp2(s * scale * log2 e - m) written over S as 16-bit
//               pairs: for bf16 as a hi part bf16(p) and a lo part bf16(p - hi), multiplied
//               by V separately, so the weights keep ~16 significant bits instead of 8.
//               At the end of the unit the partner threads add their row sums and each
//               normalises and stores its half of the row of O.
//   warps 18,19 idle (the block is a whole number of warpgroups); with integer caches they
//               are the converters below.
// TMEM: S_A at column 0, S_B at 128, O_A at 256, O_B at 384 (512 columns allocated).
//
// Integer caches (KQ = 1 INT8, 2 INT4): the tensor cores multiply fp16 values, so the codes
// are turned into fp16 in shared memory. The producer's TMA lands each tile's code rows in
// the last 64-column slab of the tile's fp16 buffer, one 128-byte row per key (the KV head's
// code bytes, then the next head's, unused); warps 18 and 19 rewrite every row in place as
// the exact fp16 integers of its codes (a warp reads whole rows before writing any of them)
// and release the tile to the MMA. Q K^T then multiplies the query rows the cache-write
// stage scaled by the K scales (fp16, with a power-of-two exponent per row that the row's
// softmax constant takes back) by the codes; P V multiplies fp16 P by the V codes, and the
// epilogue applies the V scales per channel. The scores and output are those of the
// operator on the values code * scale.
#include "common.cuh"

namespace pa {

constexpr uint32_t kTmemCols = 512;
// warp 0 TMA, warp 1 MMA, warps 2..9 softmax of head A, 10..17 of head B, 18..19 idle (the
// block is a whole number of warpgroups, the unit registers are allocated in)
constexpr int kPreThreads = 640;
constexpr int kSoftWarpsPerHead = 8;  // two warps per TMEM lane quarter, 64 score columns each

__device__ __forceinline__ uint32_t s_col(int x) { return x ? 128u : 0u; }
__device__ __forceinline__ uint32_t o_col(int x) { return x ? 384u : 256u; }

template <int HS, bool BF16, int KQ>
__global__ void __launch_bounds__(kPreThreads, 1)
    prefill_kernel(const Args a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmVm,
                   const int seg_rows) {
  using L = PreSmem<HS>;
  constexpr int HALVES = HS / 64;
  constexpr int KSTEPS = HS / 16;  // k-steps of Q K^T
  // the MMA operand type: T, except on integer caches (fp16 scaled queries and fp16 codes);
  // BF16 is the type of the output
  constexpr bool MB = BF16 && KQ == 0;
  constexpr uint32_t IDESC_QK = idesc_f16(MB, kPreTileQ, kPreTileK, false);
  constexpr uint32_t IDESC_PV = idesc_f16(MB, kPreTileQ, HS, true);
  constexpr uint32_t IDESC_PV16 = idesc_f16(false, kPreTileQ, HS, true);  // fp16 P times fp16 V (copy or codes)
  constexpr int RB = KQ == 1 ? HS : HS / 2;  // code bytes of one KV head's row

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = bars + 4;
  uint64_t* v_full = bars + 6;
  uint64_t* v_empty = bars + 8;
  uint64_t* s_full = bars + 10;  // [head]
  uint64_t* p_full = bars + 12;
  uint64_t* o_done = bars + 14;
  uint64_t* o_free = bars + 16;
  uint64_t* kc_full = bars + 18;  // integer caches: a tile's code rows landed
  uint64_t* vc_full = bars + 20;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);
  uint32_t* err = &a.hdr->error;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], KQ ? 2 : 1);  // (integer caches: the two converter warps)
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], KQ ? 2 : 1);
      mbar_init(&kc_full[i], 1);
      mbar_init(&vc_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 32 * kSoftWarpsPerHead);
      mbar_init(&o_done[i], 1);
      mbar_init(&o_free[i], 32 * kSoftWarpsPerHead);
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the work list, caches and V copy written by the earlier kernels of this call
  pdl_launch_dependents();

  const bool pair = (a.G & 1) == 0;  // two query heads of one KV head per unit
  // bf16: V from the fp16 copy (one fp16 P V product per 16 keys), unless the planner found
  // no room for it or the copy met a value fp16 cannot hold (then bf16 V, P as hi + lo)
  const bool v16 = MB && a.hdr->v_mirror && !a.hdr->v_mirror_bad;
  const int hpu = pair ? 2 : 1;
  const int units_per_tile = a.nh / hpu;
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
    uint32_t gs = 0, unit_cnt = 0;
    // records of the current and the next two units, each loaded two units ahead of use
    PrefillTile next = load_tile(a, snake_unit(0, *pre_ctas), n_units, units_per_tile);
    PrefillTile next2 = load_tile(a, snake_unit(1, *pre_ctas), n_units, units_per_tile);
    for (int u = snake_unit(0, *pre_ctas); u < n_units; u = snake_unit(++unit_cnt, *pre_ctas)) {
      const PrefillTile tile = next;
      next = next2;
      const int un = snake_unit(unit_cnt + 1, *pre_ctas);
      next2 = load_tile(a, snake_unit(unit_cnt + 2, *pre_ctas), n_units, units_per_tile);
      const int h0 = (u % units_per_tile) * hpu, g = h0 / a.G;
      const int c0 = tile.c0, q_len = tile.q_len, past = tile.past;
      const int kv_len = past + q_len;
      const int n_kv = tile.n_kv;
      const int* bt = a.block_table + (int64_t)tile.b * a.max_blocks;
      const int mirror_row0 = tile.mirror_row0;
      if (lane == 0) {
        if (unit_cnt > 0) mbar_wait(q_empty, (unit_cnt - 1) & 1, abort, err);
        mbar_arrive_expect_tx(q_full, hpu * L::kQBytes);
        for (int x = 0; x < hpu; ++x)
#pragma unroll
          for (int hh = 0; hh < HALVES; ++hh)
            tma_load_2d(smem + L::kQ + x * L::kQBytes + hh * L::kHalfBytes, &tmQ, q_full, (h0 + x) * HS + hh * 64,
                        c0 + tile.j0);
        if (un < n_units) {
          // the next unit's Q into L2 now, so its load at the unit boundary is short
          const int h0n = (un % units_per_tile) * hpu;
          for (int x = 0; x < hpu; ++x)
#pragma unroll
            for (int hh = 0; hh < HALVES; ++hh) tma_prefetch_l2_2d(&tmQ, (h0n + x) * HS + hh * 64, next.c0 + next.j0);
        }
      }
      for (int t = 0; t < n_kv; ++t, ++gs) {
        const int st = gs & 1;
        const uint32_t ph = (gs >> 1) & 1;
        int z = (int)cache_rows;  // past the end: zero fill
        int zv = v16 ? a.mirror_keys : z;
        if (lane < nseg) {
          const int key = t * kPreTileK + lane * seg_rows;
          if (key < kv_len) {
            const int blk = bt[key / a.bs];
            if (blk >= 0 && blk < a.num_blocks) z = blk * a.bs + key % a.bs;
            else if (!v16) atomicOr(err, PA_DEVERR_BAD_BLOCK);  // (the copy kernel flags it otherwise)
            zv = v16 ? mirror_row0 + key : z;
          }
        }
        if constexpr (KQ != 0) {
          // code rows (128 bytes from this head's row start) into the tiles' last slabs
          constexpr int kCodeSlab = (HALVES - 1) * L::kHalfBytes;
          if (lane == 0) {
            mbar_wait(&k_empty[st], ph ^ 1, abort, err);
            mbar_arrive_expect_tx(&kc_full[st], kPreTileK * 128);
          }
          __syncwarp();
          if (lane < nseg)
            tma_load_2d(smem + L::kK0 + st * L::kKVBytes + kCodeSlab + lane * seg_rows * 128, &tmK, &kc_full[st],
                        g * RB, z);
          if (lane == 0) {
            mbar_wait(&v_empty[st], ph ^ 1, abort, err);
            mbar_arrive_expect_tx(&vc_full[st], kPreTileK * 128);
          }
          __syncwarp();
          if (lane < nseg)
            tma_load_2d(smem + L::kV0 + st * L::kKVBytes + kCodeSlab + lane * seg_rows * 128, &tmV, &vc_full[st],
                        g * RB, z);
          __syncwarp();
          continue;
        }
        if (lane == 0) {
          mbar_wait(&k_empty[st], ph ^ 1, abort, err);
          mbar_arrive_expect_tx(&k_full[st], L::kKVBytes);
        }
        __syncwarp();
        if (lane < nseg) {
          uint8_t* dst = smem + L::kK0 + st * L::kKVBytes + lane * seg_rows * 128;
#pragma unroll
          for (int hh = 0; hh < HALVES; ++hh) tma_load_3d(dst + hh * L::kHalfBytes, &tmK, &k_full[st], hh * 64, g, z);
        }
        if (lane == 0) {
          mbar_wait(&v_empty[st], ph ^ 1, abort, err);
          mbar_arrive_expect_tx(&v_full[st], L::kKVBytes);
        }
        __syncwarp();
        if (lane < nseg) {
          uint8_t* dst = smem + L::kV0 + st * L::kKVBytes + lane * seg_rows * 128;
#pragma unroll
          for (int hh = 0; hh < HALVES; ++hh)
            tma_load_3d(dst + hh * L::kHalfBytes, v16 ? &tmVm : &tmV, &v_full[st], hh * 64, g, zv);
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    // Shared-memory descriptors of the tile bases; an MMA's operand descriptor is its base
    // plus the operand's byte offset >> 4 (the start-address field, bits 0..13, never carries:
    // shared addresses stay below 2^18), so issuing an MMA costs a couple of additions.
    const uint64_t qdesc0 = sdesc_sw128(smem_u32(smem + L::kQ), 16, 1024);
    const uint64_t kdesc0 = sdesc_sw128(smem_u32(smem + L::kK0), 16, 1024);
    const uint64_t vdesc0 = sdesc_sw128(smem_u32(smem + L::kV0), L::kHalfBytes, 1024);
    uint32_t gs = 0, unit_cnt = 0;
    PrefillTile next = load_tile(a, snake_unit(0, *pre_ctas), n_units, units_per_tile);
    for (int u = snake_unit(0, *pre_ctas); u < n_units; u = snake_unit(++unit_cnt, *pre_ctas)) {
      const PrefillTile tile = next;  // loaded one unit ahead
      next = load_tile(a, snake_unit(unit_cnt + 1, *pre_ctas), n_units, units_per_tile);
      const int kv_len = tile.past + tile.q_len;
      const int n_kv = tile.n_kv;
      mbar_wait(q_full, unit_cnt & 1, abort, err);
      tc_fence_after();

      auto issue_qk = [&](int x, int t) {
        const uint32_t gt = gs + t;
        const int st = gt & 1;
        const uint64_t qd = qdesc0 + (uint64_t)((x * L::kQBytes) >> 4);
        const uint64_t kd = kdesc0 + (uint64_t)((st * L::kKVBytes) >> 4);
        const uint32_t d_tmem = tmem + s_col(x);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk) {
            // 16 columns of head_size: slab kk / 4, 32-byte step kk % 4 inside the 128-byte row
            constexpr uint32_t kSlab = L::kHalfBytes >> 4;
            const uint64_t off = (uint64_t)((kk >> 2) * kSlab + (kk & 3) * 2);
            tc_mma_ss(d_tmem, qd + off, kd + off, IDESC_QK, kk > 0 ? 1u : 0u);
          }
          tc_commit(&s_full[x]);
          if (x == hpu - 1) {  // both heads have read this K tile
            tc_commit(&k_empty[st]);
            if (t == n_kv - 1) tc_commit(q_empty);
          }
        }
        __syncwarp();
      };
      auto issue_pv = [&](int x, int i) {
        const uint32_t gi = gs + i;
        const int st = gi & 1;
        const uint32_t ph = (gi >> 1) & 1;
        mbar_wait(&p_full[x], gi & 1, abort, err);
        if (x == 0) mbar_wait(&v_full[st], ph, abort, err);
        if (i == 0 && unit_cnt > 0) mbar_wait(&o_free[x], (unit_cnt - 1) & 1, abort, err);
        tc_fence_after();
        uint8_t* vtile = smem + L::kV0 + st * L::kKVBytes;
        const int valid = kv_len - i * kPreTileK;  // keys of this tile inside the sequence
        if (KQ == 0 && x == 0 && valid < kPreTileK) {  // (codes are finite)
          // keys past the sequence may be unwritten cache rows; P is 0 there but 0 * NaN
          // is not, so clear those V rows (whole 128-byte rows: the swizzle stays inside)
          const int rows = kPreTileK - valid;
          for (int c = lane; c < rows * 8 * HALVES; c += 32) {
            const int hh = c / (rows * 8), rem = c % (rows * 8);
            const int r = valid + rem / 8, ch = rem % 8;
            *reinterpret_cast<uint4*>(vtile + hh * L::kHalfBytes + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        const uint64_t vd = vdesc0 + (uint64_t)((st * L::kKVBytes) >> 4);
        const uint32_t p_tmem = tmem + s_col(x);
        const uint32_t d_tmem = tmem + o_col(x);
        const uint32_t acc0 = i > 0 ? 1u : 0u;
        if (elect_one()) {
          // 16 keys of V per MMA: rows 16kk.. (K dimension, 8-row atoms 1024 B apart), the
          // two 64-column slabs of head_size 16 KB apart (MN dimension)
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
          tc_commit(&o_done[x]);
          if (x == hpu - 1) tc_commit(&v_empty[st]);  // both heads have read this V tile
        }
        __syncwarp();
      };

      for (int t = 0; t < n_kv; ++t) {
        const uint32_t gt = gs + t;
        mbar_wait(&k_full[gt & 1], (gt >> 1) & 1, abort, err);
        tc_fence_after();
        issue_qk(0, t);
        if (pair) {
          if (t > 0) issue_pv(1, t - 1);
          issue_qk(1, t);
        }
        issue_pv(0, t);
      }
      if (pair) issue_pv(1, n_kv - 1);
      gs += n_kv;
    }
  } else if (warp < 2 + 2 * kSoftWarpsPerHead) {
    // ======================= softmax: warps 2..9 head A, 10..17 head B =======================
    // Two warps share each TMEM lane quarter (rows), one per half of the 128 score columns;
    // they exchange their partial row maxima through shared memory once per tile, meeting
    // at a 64-thread named barrier of their own.
    const int sw = warp - 2;
    const int x = sw / kSoftWarpsPerHead;  // head
    const int hsel = (sw >> 2) & 1;        // column half
    if (x == 0 || pair) {
      constexpr int COLS = kPreTileK / 2;  // score columns per thread
      constexpr int OCOLS = HS / 2;        // output columns per thread
      const int quarter = warp & 3;
      const int row = quarter * 32 + lane;
      const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
      const uint32_t s_base = tmem + lane_off + s_col(x);
      const uint32_t s_tmem = s_base + hsel * COLS;
      const uint32_t o_tmem = tmem + lane_off + o_col(x) + hsel * OCOLS;
      float* xmax = reinterpret_cast<float*>(smem + L::kXmax);
      float* xsum = reinterpret_cast<float*>(smem + L::kXsum);
      const int pair_bar = 2 + x * 4 + quarter;  // named barrier of the two warps of this lane quarter
      uint32_t gs = 0;
      PrefillTile next = load_tile(a, snake_unit(0, *pre_ctas), n_units, units_per_tile);
      for (int k = 0, u = snake_unit(0, *pre_ctas); u < n_units; u = snake_unit(++k, *pre_ctas)) {
        const PrefillTile tile = next;  // loaded during the previous unit's epilogue
        const int h = (u % units_per_tile) * hpu + x;
        const int c0 = tile.c0, q_len = tile.q_len, past = tile.past;
        const int kv_len = past + q_len;
        const int n_kv = tile.n_kv;
        const int lim = min(past + tile.j0 + row, kv_len - 1);  // last key this row sees
        const int lim_tile0 = past + tile.j0;                   // the smallest limit of the unit
        // the softmax constant scale * log2(e); integer caches: times 2^E, the exponent the
        // cache-write stage took out of this row's scaled query, and 2^24, the unit of the
        // K codes' subnormals (rows past the sequence: 1)
        float c = a.scale_log2;
        if constexpr (KQ != 0)
          if (tile.j0 + row < q_len) c = ldexpf(c, __ldg(a.qexp + (int64_t)(c0 + tile.j0 + row) * a.nh + h) + 24);
        float m_used = -INFINITY, l = 0.f;
        for (int t = 0; t < n_kv; ++t) {
          const uint32_t gt = gs + t;
          mbar_wait(&s_full[x], gt & 1, abort, err);
          tc_fence_after();
          const int key0 = t * kPreTileK + hsel * COLS;  // first key of this thread's columns
          const bool masked = (t * kPreTileK + kPreTileK - 1 > lim_tile0) || (t * kPreTileK + kPreTileK > kv_len);
          uint32_t r[COLS];
          tmem_ld_x64(s_tmem, r);
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
              for (int k = 0; k < 4; ++k)
                mc[k] = fmax3(mc[k], __uint_as_float(r[e + 2 * k]), __uint_as_float(r[e + 2 * k + 1]));
          } else {
#pragma unroll
            for (int e = 0; e < COLS; e += 8)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mc[k] = fmin3(mc[k], __uint_as_float(r[e + 2 * k]), __uint_as_float(r[e + 2 * k + 1]));
          }
          const float mr = c > 0.f ? fmax3(fmaxf(mc[0], mc[1]), mc[2], mc[3]) : fmin3(fminf(mc[0], mc[1]), mc[2], mc[3]);
          float* xm = xmax + ((gt & 1) * 2 + x) * (kPreTileQ * 2) + row * 2;
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
          // ---- P = exp2(s * c - m), written over S in place, 16 keys at a time: the fp16
          // word (or, against bf16 V, the bf16 hi and lo words) of each key pair replaces
          // that pair's two score registers ----
          const float neg_m = -m_used;
          bool p_done = false;
          if constexpr (MB) {
            if (!v16) {  // against bf16 V: P as hi and lo bf16 parts
              float lc[2] = {0.f, 0.f};
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
              l += lc[0] + lc[1];
              p_done = true;
            }
          }
          if (!p_done) {
            // fp16 P (fp16 V, or the fp16 copy of bf16 V): s * c - m and the row sums on packed
            // fp32 pairs (one instruction per key pair)
            const uint64_t c2 = f2_make(c, c), nm2 = f2_make(neg_m, neg_m);
            uint64_t lsum[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
#pragma unroll
            for (int g2 = 0; g2 < COLS / 16; ++g2) {
              uint32_t* q = r + g2 * 16;
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const uint64_t x2 = f2_fma(f2_make(__uint_as_float(q[2 * e]), __uint_as_float(q[2 * e + 1])), c2, nm2);
                float x0, x1;
                f2_split(x2, x0, x1);
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
            mbar_wait(&o_done[x], (gt - 1) & 1, abort, err);
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
          mbar_arrive(&p_full[x]);
        }
        // ---- epilogue: wait for the last P V, normalise, store the valid rows ----
        // (the next unit's record is loaded here, where few registers are live, and
        // arrives while this unit's output is written)
        next = load_tile(a, snake_unit(k + 1, *pre_ctas), n_units, units_per_tile);
        mbar_wait(&o_done[x], (gs + n_kv - 1) & 1, abort, err);
        tc_fence_after();
        {
          float* xs = xsum + x * (kPreTileQ * 2) + row * 2;
          xs[hsel] = l;
          named_bar_sync(pair_bar, 64);
          const float l_row = xs[0] + xs[1];
          const float inv = 1.f / l_row;
          const bool store = tile.j0 + row < q_len;
          if (a.lse && store && hsel == 0) {  // natural log; m_used is the base-2 max of s * scale
            float bias = 0.f;  // (integer caches) the K codes' offset in the row's scores
            if constexpr (KQ != 0) {
              const int64_t qr = (int64_t)(c0 + tile.j0 + row) * a.nh + h;
              const uint4* qp = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.query) + qr * HS);
              float sq = 0.f;
              for (int i = 0; i < HS / 8; ++i) {
                const uint4 q4 = __ldg(qp + i);
                const uint32_t qw[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  sq += __half2float(__ushort_as_half((unsigned short)(qw[e] & 0xFFFFu))) +
                        __half2float(__ushort_as_half((unsigned short)(qw[e] >> 16)));
              }
              bias = (KQ == 1 ? 128.f : 8.f) * sq * ldexpf(a.scale_log2, __ldg(a.qexp + qr));
            }
            a.lse[(int64_t)(c0 + tile.j0 + row) * a.nh + h] = (m_used + fast_log2(l_row) - bias) * 0.69314718055994531f;
          }
          uint16_t* dst =
              reinterpret_cast<uint16_t*>(a.output) + ((int64_t)(c0 + tile.j0 + row) * a.nh + h) * HS + hsel * OCOLS;
          // this thread's half row of O in registers, then O is released to the next unit
          uint32_t ov[OCOLS];
          if constexpr (OCOLS == 64) tmem_ld_x64(o_tmem, ov);
          else tmem_ld_x32(o_tmem, ov);
          tc_fence_before();
          mbar_arrive(&o_free[x]);
          if (store) {
            const uint16_t* gsrc = a.gate + ((int64_t)(c0 + tile.j0 + row) * a.nh + h) * HS + hsel * OCOLS;
            if constexpr (KQ != 0) {
              // integer caches: O holds sum p code over the V codes; the row's output is O / l
              // times the V scale of each channel (then the gate), 8 at a time, packed in place
              // (word v from words 2v, 2v + 1)
              const float4* vs = reinterpret_cast<const float4*>(a.v_scale + (h / a.G) * HS + hsel * OCOLS);
#pragma unroll
              for (int v = 0; v < OCOLS; v += 8) {
                const float4 s0 = __ldg(vs + v / 4), s1 = __ldg(vs + v / 4 + 1);
                const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(ov[v + e]) * inv * sv[e];
                if (a.gate) apply_gate8<BF16>(gsrc + v, x);
#pragma unroll
                for (int e = 0; e < 8; e += 2) ov[(v + e) / 2] = pack2<BF16>(x[e], x[e + 1]);
              }
            } else {
              if (a.gate) {  // output gate: times sigmoid(gate), elementwise
#pragma unroll
                for (int v = 0; v < OCOLS; v += 8) apply_gate8<BF16>(gsrc + v, reinterpret_cast<float*>(ov + v));
              }
#pragma unroll
              for (int v = 0; v < OCOLS / 2; ++v)  // packed in place (word v from words 2v, 2v + 1)
                ov[v] = pack2<BF16>(__uint_as_float(ov[2 * v]) * inv, __uint_as_float(ov[2 * v + 1]) * inv);
            }
            if (a.out_v8) {  // 32-byte stores where the output allows them: half the store wavefronts
#pragma unroll
              for (int v = 0; v < OCOLS / 2; v += 8) st_global_v8(dst + 2 * v, &ov[v]);
            } else {
#pragma unroll
              for (int v = 0; v < OCOLS / 2; v += 4)
                *reinterpret_cast<uint4*>(dst + 2 * v) = make_uint4(ov[v], ov[v + 1], ov[v + 2], ov[v + 3]);
            }
          }
        }
        gs += n_kv;
      }
    }
  }

  if constexpr (KQ != 0) {
    if (warp >= 2 + 2 * kSoftWarpsPerHead) {
      // ======================= converters: warps 18, 19 (integer caches) =======================
      // the tiles in the producer's order: K then V of every KV tile of every unit
      const int cw = warp - (2 + 2 * kSoftWarpsPerHead);
      uint32_t gs = 0, unit_cnt = 0;
      for (int u = snake_unit(0, *pre_ctas); u < n_units; u = snake_unit(++unit_cnt, *pre_ctas)) {
        const int n_kv = load_tile(a, u, n_units, units_per_tile).n_kv;
        for (int t = 0; t < n_kv; ++t, ++gs) {
          const int st = gs & 1;
          const uint32_t ph = (gs >> 1) & 1;
          mbar_wait(&kc_full[st], ph, abort, err);
          convert_code_tile<HS, KQ, true>(smem + L::kK0 + st * L::kKVBytes, cw, lane);
          fence_proxy_async_smem();  // (the MMA reads the tile through the async proxy)
          __syncwarp();
          if (lane == 0) mbar_arrive(&k_full[st]);
          mbar_wait(&vc_full[st], ph, abort, err);
          convert_code_tile<HS, KQ>(smem + L::kV0 + st * L::kKVBytes, cw, lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&v_full[st]);
        }
      }
    }
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- host launcher ----
template <int HS, bool BF16, int KQ>
static cudaError_t launch_prefill_t(const Args& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                    const CUtensorMap& tvm, int seg, int grid, cudaStream_t s) {
  constexpr int smem = PreSmem<HS>::kBytes;
  cudaError_t e =
      cudaFuncSetAttribute(prefill_kernel<HS, BF16, KQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // On integer caches the kernel launches only once the quantizing cache write has finished:
  // launched early, its blocks (one per SM, taking the SM's registers) land on the SMs the
  // cache write frees first, and the mixed batch measured 450 -> 372 us (INT4) and 381 ->
  // 364 us (INT8) without that, the fp16 workloads no change either way.
  return launch_pdl_if(KQ == 0, prefill_kernel<HS, BF16, KQ>, dim3(grid), dim3(kPreThreads), smem, s, a, tq, tk,
                       tv, tvm, seg);
}

template <int KQ>
static cudaError_t launch_prefill_kq(const Args& a, bool bf16, const CUtensorMap& tq, const CUtensorMap& tk,
                                     const CUtensorMap& tv, const CUtensorMap& tvm, int seg, int grid, cudaStream_t s) {
  if constexpr (KQ != 2) {  // (INT4 needs head_size 128 or more)
    if (a.hs == 64)
      return bf16 ? launch_prefill_t<64, true, KQ>(a, tq, tk, tv, tvm, seg, grid, s)
                  : launch_prefill_t<64, false, KQ>(a, tq, tk, tv, tvm, seg, grid, s);
  }
  return bf16 ? launch_prefill_t<128, true, KQ>(a, tq, tk, tv, tvm, seg, grid, s)
              : launch_prefill_t<128, false, KQ>(a, tq, tk, tv, tvm, seg, grid, s);
}

cudaError_t launch_prefill(const Args& a, bool bf16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tvm, int seg, int grid, cudaStream_t s) {
  if (a.hs == 256) return launch_prefill256(a, bf16, tq, tk, tv, tvm, seg, grid, s);
  if (a.kvq == 1) return launch_prefill_kq<1>(a, bf16, tq, tk, tv, tvm, seg, grid, s);
  if (a.kvq == 2) return launch_prefill_kq<2>(a, bf16, tq, tk, tv, tvm, seg, grid, s);
  return launch_prefill_kq<0>(a, bf16, tq, tk, tv, tvm, seg, grid, s);
}

}  // namespace pa
