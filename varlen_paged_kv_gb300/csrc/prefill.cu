// Prefill / chunked-prefill attention on the 5th-generation tensor cores.
//
// Work unit: 128 query rows [j0, j0 + 128) of one sequence for one query head h. Rows
// never straddle sequences; rows past the sequence end are computed and not stored.
// The CTA walks the 128-key KV tiles 0 .. ceil((past + last row + 1) / 128) - 1 of that
// sequence (bottom-right causal: row j sees keys 0 .. past + j), with the online softmax
// of FlashAttention.
//
// Roles (192 threads, persistent over the planner's tile list, longest tiles first):
//   warp 0      TMA producer: Q tile once per unit (2-D map over the query rows), then K
//               and V tiles into a 2-deep ring, each tile gathered page segment by page
//               segment through block_table (3-D map over (head_size, kv_heads, slots),
//               128-byte swizzle). Segments past the sequence read as zeros.
//   warp 1      TMEM owner and MMA issuer (one thread): S = Q K^T with tcgen05.mma
//               (both operands from shared memory, fp32 accumulator in TMEM, two S
//               buffers so QK^T of tile t+1 overlaps the softmax of tile t), then
//               O += P V with P read from TMEM (where the softmax wrote it over S) and V
//               from shared memory.
//   warps 2..5  softmax: thread i owns TMEM lane / query row i; loads its S row, masks,
//               updates the running max (the O rescale is skipped until the max has
//               grown by more than 2^8, which is exact because the final division uses
//               the same stale max), writes P as 16-bit pairs into TMEM (bf16: as a hi
//               and a lo part, bf16(p) and bf16(p - hi), multiplied by V separately, so
//               the weights keep ~16 bits instead of 8), and at the end normalises O and
//               stores the row.
// TMEM: S0 at column 0, S1 at 128, O at 256 (512 columns allocated).
#include "common.cuh"

namespace pa {

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol0 = 0, kSCol1 = 128, kOCol = 256;

template <int HS, bool BF16>
__global__ void __launch_bounds__(192, 1)
    prefill_kernel(const Args a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const int seg_rows) {
  using L = PreSmem<HS>;
  constexpr int HALVES = HS / 64;
  constexpr int KSTEPS = HS / 16;                      // k-steps of Q K^T
  constexpr uint32_t IDESC_QK = idesc_f16(BF16, kPreTileQ, kPreTileK, false);
  constexpr uint32_t IDESC_PV = idesc_f16(BF16, kPreTileQ, HS, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = bars + 4;
  uint64_t* v_full = bars + 6;
  uint64_t* v_empty = bars + 8;
  uint64_t* s_full = bars + 10;
  uint64_t* p_full = bars + 12;
  uint64_t* o_done = bars + 14;
  uint64_t* o_free = bars + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);
  uint32_t* err = &a.hdr->error;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
    }
    mbar_init(o_done, 1);
    mbar_init(o_free, 128);
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

  const int n_units = a.hdr->n_prefill_tiles * a.nh;
  const int64_t cache_rows = (int64_t)a.num_blocks * a.bs;

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    const int nseg = kPreTileK / seg_rows;
    uint32_t it_kv = 0, unit_cnt = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++unit_cnt) {
      const PrefillTile tile = a.tiles[u / a.nh];
      const int h = u % a.nh, g = h / a.G;
      const int c0 = a.cum[tile.b], q_len = a.cum[tile.b + 1] - c0, past = a.past[tile.b];
      const int kv_len = past + q_len;
      const int n_kv = (int)ceil_div(past + min(tile.j0 + kPreTileQ, q_len), kPreTileK);
      const int* bt = a.block_table + (int64_t)tile.b * a.max_blocks;
      if (lane == 0) {
        if (unit_cnt > 0) mbar_wait(q_empty, (unit_cnt - 1) & 1, abort, err);
        mbar_arrive_expect_tx(q_full, L::kQBytes);
#pragma unroll
        for (int hh = 0; hh < HALVES; ++hh)
          tma_load_2d(smem + L::kQ + hh * (kPreTileQ * 128), &tmQ, q_full, h * HS + hh * 64, c0 + tile.j0);
      }
      for (int t = 0; t < n_kv; ++t, ++it_kv) {
        const int st = it_kv & 1;
        const uint32_t ph = (it_kv >> 1) & 1;
        // physical row of this lane's page segment (lanes 0 .. nseg-1)
        int z = (int)cache_rows;  // past the end: zero fill
        if (lane < nseg) {
          const int key = t * kPreTileK + lane * seg_rows;
          if (key < kv_len) {
            const int blk = bt[key / a.bs];
            if (blk >= 0 && blk < a.num_blocks) z = blk * a.bs + key % a.bs;
            else atomicOr(err, PA_DEVERR_BAD_BLOCK);
          }
        }
        // K tile
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
        // V tile
        if (lane == 0) {
          mbar_wait(&v_empty[st], ph ^ 1, abort, err);
          mbar_arrive_expect_tx(&v_full[st], L::kKVBytes);
        }
        __syncwarp();
        if (lane < nseg) {
          uint8_t* dst = smem + L::kV0 + st * L::kKVBytes + lane * seg_rows * 128;
#pragma unroll
          for (int hh = 0; hh < HALVES; ++hh) tma_load_3d(dst + hh * L::kHalfBytes, &tmV, &v_full[st], hh * 64, g, z);
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    const uint32_t q_base = smem_u32(smem + L::kQ);
    uint32_t it_kv = 0, unit_cnt = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++unit_cnt) {
      const PrefillTile tile = a.tiles[u / a.nh];
      const int c0 = a.cum[tile.b], q_len = a.cum[tile.b + 1] - c0, past = a.past[tile.b];
      const int kv_len = past + q_len;
      const int n_kv = (int)ceil_div(past + min(tile.j0 + kPreTileQ, q_len), kPreTileK);
      mbar_wait(q_full, unit_cnt & 1, abort, err);
      tc_fence_after();

      auto issue_pv = [&](int i) {
        const uint32_t gi = it_kv + i;
        const int st = gi & 1;
        const uint32_t ph = (gi >> 1) & 1;
        mbar_wait(&p_full[st], ph, abort, err);
        mbar_wait(&v_full[st], ph, abort, err);
        if (i == 0 && unit_cnt > 0) mbar_wait(o_free, (unit_cnt - 1) & 1, abort, err);
        tc_fence_after();
        uint8_t* vtile = smem + L::kV0 + st * L::kKVBytes;
        const int valid = kv_len - i * kPreTileK;  // keys of this tile inside the sequence
        if (valid < kPreTileK) {
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
        if (lane == 0) {
          const uint32_t v_base = smem_u32(vtile);
          const uint32_t p_tmem = tmem + (st ? kSCol1 : kSCol0);
#pragma unroll
          for (int kk = 0; kk < kPreTileK / 16; ++kk) {
            // 16 keys of V: rows 16kk.. (K dimension, 8-row atoms 1024 B apart), the two
            // 64-column slabs of head_size 16 KB apart (MN dimension)
            const uint64_t vdesc = sdesc_sw128(v_base + kk * 16 * 128, L::kHalfBytes, 1024);
            tc_mma_ts(tmem + kOCol, p_tmem + kk * 8, vdesc, IDESC_PV, (i > 0 || kk > 0) ? 1u : 0u);
            if constexpr (BF16) tc_mma_ts(tmem + kOCol, p_tmem + 64 + kk * 8, vdesc, IDESC_PV, 1u);
          }
          tc_commit(&v_empty[st]);
          tc_commit(o_done);
        }
        __syncwarp();
      };

      for (int t = 0; t < n_kv; ++t) {
        const uint32_t gi = it_kv + t;
        const int st = gi & 1;
        const uint32_t ph = (gi >> 1) & 1;
        mbar_wait(&k_full[st], ph, abort, err);
        tc_fence_after();
        if (lane == 0) {
          const uint32_t k_base = smem_u32(smem + L::kK0 + st * L::kKVBytes);
          const uint32_t s_tmem = tmem + (st ? kSCol1 : kSCol0);
#pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk) {
            // 16 columns of head_size: slab kk / 4, 32-byte step kk % 4 inside the 128-byte row
            const uint32_t off = (kk >> 2) * L::kHalfBytes + (kk & 3) * 32;
            const uint64_t qdesc = sdesc_sw128(q_base + off, 16, 1024);
            const uint64_t kdesc = sdesc_sw128(k_base + off, 16, 1024);
            tc_mma_ss(s_tmem, qdesc, kdesc, IDESC_QK, kk > 0 ? 1u : 0u);
          }
          tc_commit(&s_full[st]);
          tc_commit(&k_empty[st]);
          if (t == n_kv - 1) tc_commit(q_empty);
        }
        __syncwarp();
        if (t > 0) issue_pv(t - 1);
      }
      issue_pv(n_kv - 1);
      it_kv += n_kv;
    }
  } else {
    // ======================= softmax warps 2..5 =======================
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint32_t it_kv = 0, o_seen = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const PrefillTile tile = a.tiles[u / a.nh];
      const int h = u % a.nh;
      const int c0 = a.cum[tile.b], q_len = a.cum[tile.b + 1] - c0, past = a.past[tile.b];
      const int kv_len = past + q_len;
      const int n_kv = (int)ceil_div(past + min(tile.j0 + kPreTileQ, q_len), kPreTileK);
      const int lim = min(past + tile.j0 + row, kv_len - 1);  // last key this row sees
      const int lim_tile0 = past + tile.j0;                   // the smallest limit of the tile
      float m_used = -INFINITY, l = 0.f;
      for (int t = 0; t < n_kv; ++t) {
        const uint32_t gi = it_kv + t;
        const int st = gi & 1;
        const uint32_t ph = (gi >> 1) & 1;
        const uint32_t s_tmem = tmem + lane_off + (st ? kSCol1 : kSCol0);
        mbar_wait(&s_full[st], ph, abort, err);
        tc_fence_after();
        uint32_t sr[kPreTileK];
        tmem_ld_x64(s_tmem, sr);
        tmem_ld_x64(s_tmem + 64, sr + 64);
        float x[kPreTileK];
        const int key0 = t * kPreTileK;
        const bool masked = (key0 + kPreTileK - 1 > lim_tile0) || (key0 + kPreTileK > kv_len);
        float mt = -INFINITY;
#pragma unroll
        for (int c = 0; c < kPreTileK; ++c) {
          float v = __uint_as_float(sr[c]) * a.scale_log2;
          if (masked && key0 + c > lim) v = -INFINITY;
          x[c] = v;
          mt = fmaxf(mt, v);
        }
        const float m_new = fmaxf(m_used, mt);
        const bool grow = m_new > m_used + 8.0f;  // also true on the first tile (m_used = -inf)
        const bool any_grow = __any_sync(0xffffffffu, grow);
        float alpha = 1.f;
        if (any_grow) {
          alpha = fast_exp2(m_used - m_new);  // 0 on the first tile; 1 where m_new == m_used
          m_used = m_new;
          l *= alpha;
        }
        // P = exp2(x - m) as 16-bit pairs, written over the first 64 columns of this S buffer
        // (bf16: P = hi + lo, hi over columns 0..63 and lo over 64..127 of the S buffer)
#pragma unroll
        for (int hcol = 0; hcol < 2; ++hcol) {
          uint32_t pw[32];
          uint32_t pl[BF16 ? 32 : 1];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float p0 = fast_exp2(x[hcol * 64 + 2 * c] - m_used);
            const float p1 = fast_exp2(x[hcol * 64 + 2 * c + 1] - m_used);
            l += p0 + p1;
            if constexpr (BF16) split_bf16x2(p0, p1, pw[c], pl[c]);
            else pw[c] = pack2<false>(p0, p1);
          }
          tmem_st_x32(s_tmem + hcol * 32, pw);
          if constexpr (BF16) tmem_st_x32(s_tmem + 64 + hcol * 32, pl);
        }
        if (t > 0) {
          // O holds P_0..P_{t-2} V; wait for P_{t-1} V before rescaling it
          mbar_wait(o_done, o_seen & 1, abort, err);
          ++o_seen;
          if (any_grow) {
            tc_fence_after();
            const uint32_t o_tmem = tmem + lane_off + kOCol;
#pragma unroll 1
            for (int c = 0; c < HS; c += 32) {
              uint32_t ov[32];
              tmem_ld_x32(o_tmem + c, ov);
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
              tmem_st_x32(o_tmem + c, ov);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&p_full[st]);
      }
      // ---- epilogue: wait for the last P V, normalise, store the valid rows ----
      mbar_wait(o_done, o_seen & 1, abort, err);
      ++o_seen;
      tc_fence_after();
      {
        const uint32_t o_tmem = tmem + lane_off + kOCol;
        const float inv = 1.f / l;
        const bool store = tile.j0 + row < q_len;
        uint16_t* dst = reinterpret_cast<uint16_t*>(a.output) + ((int64_t)(c0 + tile.j0 + row) * a.nh + h) * HS;
#pragma unroll 1
        for (int c = 0; c < HS; c += 32) {
          uint32_t ov[32];
          tmem_ld_x32(o_tmem + c, ov);
          if (store) {
#pragma unroll
            for (int v = 0; v < 32; v += 8) {
              uint4 pk;
              pk.x = pack2<BF16>(__uint_as_float(ov[v + 0]) * inv, __uint_as_float(ov[v + 1]) * inv);
              pk.y = pack2<BF16>(__uint_as_float(ov[v + 2]) * inv, __uint_as_float(ov[v + 3]) * inv);
              pk.z = pack2<BF16>(__uint_as_float(ov[v + 4]) * inv, __uint_as_float(ov[v + 5]) * inv);
              pk.w = pack2<BF16>(__uint_as_float(ov[v + 6]) * inv, __uint_as_float(ov[v + 7]) * inv);
              *reinterpret_cast<uint4*>(dst + c + v) = pk;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(o_free);
      it_kv += n_kv;
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
template <int HS, bool BF16>
static cudaError_t launch_prefill_t(const Args& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                    int seg, int grid, cudaStream_t s) {
  constexpr int smem = PreSmem<HS>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<HS, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  prefill_kernel<HS, BF16><<<grid, 192, smem, s>>>(a, tq, tk, tv, seg);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const Args& a, bool bf16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           int seg, int grid, cudaStream_t s) {
  if (a.hs == 64)
    return bf16 ? launch_prefill_t<64, true>(a, tq, tk, tv, seg, grid, s) : launch_prefill_t<64, false>(a, tq, tk, tv, seg, grid, s);
  return bf16 ? launch_prefill_t<128, true>(a, tq, tk, tv, seg, grid, s) : launch_prefill_t<128, false>(a, tq, tk, tv, seg, grid, s);
}

}  // namespace pa
