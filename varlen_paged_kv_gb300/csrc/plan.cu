// Device work partitioner. One CTA reads cumulative_sequence_length and past_seqlens
// (which stay on the device: the host never sees them) and writes the work lists the
// attention kernels consume:
//   - decode-class sequences (q_len * G <= 16 query rows per KV head): each (sequence,
//     KV head) pair is a unit of ceil(kv_len / 64) key tiles. The units' tiles, laid end
//     to end, are cut into dec_ctas equal contiguous ranges, one per resident decode CTA;
//     a unit crossing a cut becomes several items whose partial results are merged by
//     the last of them to finish. Each unit also counts a fixed cost of a few tiles, so a
//     CTA with more items streams fewer keys and the CTAs finish together. With a forced
//     split length the units are instead cut every S keys and the items dealt to the CTAs
//     in contiguous blocks (a test hook);
//   - prefill-class sequences: 128-row query tiles, sorted by their number of 128-key KV
//     tiles, largest first, so the persistent prefill grid takes the long causal tiles
//     first (longest-processing-time order).
// The lists depend only on the inputs, the decode grid size and compile-time constants,
// so results are bitwise reproducible on a given GPU. If the batch description is
// inconsistent (cum not a prefix sum ending at N, a negative past, a sequence longer than
// its block_table row, a q_len above the host's max_query_len bound) nothing is
// scheduled and PA_DEVERR_BAD_BATCH is raised.
// The file also holds the cache write (the K/V scatter, with the Q/K preparation or the
// integer codes when asked for, and the fp16 V copy of bf16 prefill sequences).
#include <limits.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"

namespace pa {

namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ bool is_decode_class(int64_t q, const Args& a) {
  return a.route == PA_ROUTE_AUTO && q >= 1 && q * a.G <= kDecRows;
}

// exclusive scan of three ints across the block; tot[] gets the block totals
__device__ void block_scan3(const int v[3], int ex[3], int tot[3], int (*s_warp)[32]) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    int x = v[k];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    inc[k] = x;
    if (lane == 31) s_warp[k][wid] = x;
  }
  __syncthreads();
  if (wid == 0) {
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      int x = lane < nw ? s_warp[k][lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      s_warp[k][lane] = x;  // inclusive prefix of warp totals
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    int before = wid > 0 ? s_warp[k][wid - 1] : 0;
    ex[k] = before + inc[k] - v[k];
    tot[k] = s_warp[k][nw - 1];
  }
  __syncthreads();
}

// one decode item as three 16-byte stores (an aggregate assignment of the record went
// through a local-memory temporary and cost microseconds per thousand items)
__device__ __forceinline__ void store_item(DecodeItem* dst, int b, int g, int key_begin, int key_end,
                                           int unit_first, int n_split, int c0, int q_len, int past) {
  int4* d = reinterpret_cast<int4*>(dst);
  d[0] = make_int4(b, g, key_begin, key_end);
  d[1] = make_int4(unit_first, n_split, c0, q_len);
  d[2] = make_int4(past, 0, 0, 0);
}

// exclusive scan of one int64 across the block; *tot gets the block total
__device__ void block_scan_i64(int64_t v, int64_t* ex, int64_t* tot, long long* s_w) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_w[wid] = x;
  __syncthreads();
  if (wid == 0) {
    long long y = lane < nw ? s_w[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long z = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += z;
    }
    s_w[lane] = y;
  }
  __syncthreads();
  *ex = (wid > 0 ? s_w[wid - 1] : 0) + x - v;
  *tot = s_w[nw - 1];
  __syncthreads();
}

// In-place suffix minimum of v[0 .. n) (n <= 4 blockDim.x) across the block: thread t takes
// the run v[k t .. k t + k), k = ceil(n / blockDim.x), and the runs' minima are scanned.
__device__ void block_suffix_min(int* v, int n, int* s_w) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  const int k = (n + (int)blockDim.x - 1) / (int)blockDim.x;  // 1 .. 4
  int run[4];
  int x = INT_MAX;  // minimum of this thread's run
#pragma unroll
  for (int j = 3; j >= 0; --j) {
    run[j] = j < k && k * tid + j < n ? v[k * tid + j] : INT_MAX;
    x = min(x, run[j]);
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x = min(x, y);
  }
  if (lane == 0) s_w[wid] = x;  // minimum of the warp's entries
  __syncthreads();
  if (wid == 0) {
    int y = lane < nw ? s_w[lane] : INT_MAX;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int z = __shfl_down_sync(0xffffffffu, y, o);
      if (lane + o < 32) y = min(y, z);
    }
    s_w[lane] = y;  // suffix minimum over warps lane ..
  }
  __syncthreads();
  if (wid + 1 < nw) x = min(x, s_w[wid + 1]);
  // x: the minimum of the runs from this thread's on; the run's own suffix minima, each
  // joined with the minimum of the later runs
  int after = __shfl_down_sync(0xffffffffu, x, 1);
  if (lane == 31) after = wid + 1 < nw ? s_w[wid + 1] : INT_MAX;
  __syncthreads();  // every thread has read v and s_w
#pragma unroll
  for (int j = 3; j >= 0; --j) {
    after = min(after, run[j]);
    if (j < k && k * tid + j < n) v[k * tid + j] = after;
  }
  __syncthreads();
}

__device__ __forceinline__ void refuse(WsHeader* hdr) {
  atomicOr(&hdr->error, PA_DEVERR_BAD_BATCH);
  hdr->valid = 0;
  hdr->n_decode_items = hdr->n_prefill_tiles = 0;
}

}  // namespace

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const Args a) {
  __shared__ int s_bad;
  __shared__ unsigned long long s_dec_tiles;
  __shared__ int s_warp[3][32];
  __shared__ int s_carry[3];
  __shared__ int s_cta_begin[kMaxDecCtas + 1];
  // the sort keys of the prefill tiles; before the sort, the per-round tables of the
  // decode partition (CTA starts, per-sequence first tile, tiles and length)
  __shared__ __align__(16) unsigned long long s_key[kSortCap];
  __shared__ long long s_w64[32];
  __shared__ long long s_mirror_carry;
  __shared__ int s_mseq_carry;
  __shared__ unsigned long long s_pre_tiles;  // (query tile, key tile) pairs of prefill-class rows
  __shared__ unsigned long long s_split;      // best (model time bits, decode SMs)

  const int tid = threadIdx.x;
  WsHeader* hdr = a.hdr;
  // the batch description into L2 while the previous kernel drains (a hint: the loads below
  // come after the wait)
  for (int i = tid * 32; i <= a.B; i += blockDim.x * 32) {
    prefetch_l2(a.cum + i);
    if (i < a.B) prefetch_l2(a.past + i);
  }
  pdl_wait();  // the previous call's kernels may still read this workspace
  pdl_launch_dependents();
  if (tid == 0) {
    s_bad = 0;
    s_dec_tiles = 0;
    s_pre_tiles = 0;
    s_split = ~0ull;
    s_carry[0] = s_carry[1] = s_carry[2] = 0;
    s_mirror_carry = 0;
    s_mseq_carry = 0;
    hdr->error = 0;  // error bits describe the most recent call
    hdr->v_mirror = 0;
    hdr->v_mirror_bad = 0;
    hdr->mirror_rows = 0;
  }
  for (int c = tid; c <= a.dec_ctas; c += blockDim.x) s_cta_begin[c] = INT_MAX;
  __syncthreads();

  // ---- validate the batch description; count the decode key tiles ----
  const int64_t max_kv = (int64_t)a.max_blocks * a.bs;
  if (tid == 0 && (a.cum[0] != 0 || a.cum[a.B] != a.N)) s_bad = 1;
  long long dec_tiles = 0, pre_tiles = 0;
  for (int b = tid; b < a.B; b += blockDim.x) {
    const int64_t q = (int64_t)a.cum[b + 1] - a.cum[b];
    const int64_t kv = (int64_t)a.past[b] + q;
    if (q < 0 || a.past[b] < 0 || kv > max_kv || (a.max_query_len > 0 && q > a.max_query_len)) {
      atomicOr(&s_bad, 1);
    } else if (is_decode_class(q, a)) {
      dec_tiles += ceil_div(kv, kDecTile) + dec_item_cost_tiles(a.hs, a.kvq);
    } else if (q > 0 && a.split_sms) {
      // key tiles seen by the query tiles t = 0 .. T-1: ceil((past + 128 (t + 1)) / 128) =
      // c + t + 1 with c = ceil(past / 128) for all but the last, which sees ceil(kv / 128)
      static_assert(kPreTileQ == kPreTileK, "the closed form assumes square tiles");
      const int64_t T = ceil_div(q, kPreTileQ), c = ceil_div(kv - q, kPreTileK);
      pre_tiles += (T - 1) * T / 2 + (T - 1) * c + ceil_div(kv, kPreTileK);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    dec_tiles += __shfl_xor_sync(0xffffffffu, dec_tiles, o);
    pre_tiles += __shfl_xor_sync(0xffffffffu, pre_tiles, o);
  }
  if ((tid & 31) == 0 && dec_tiles) atomicAdd(&s_dec_tiles, (unsigned long long)dec_tiles);
  if ((tid & 31) == 0 && pre_tiles) atomicAdd(&s_pre_tiles, (unsigned long long)pre_tiles);
  for (int u = tid; u < a.B * a.kvh; u += blockDim.x) a.unit_done[u] = 0;
  __syncthreads();
  if (s_bad) {
    if (tid == 0) refuse(hdr);
    return;
  }
  // ---- SMs of the two attention kernels of a whole call with prefill and decode rows ----
  // The prefill kernel keeps S - d SMs and the decode work is cut for the other d, so the
  // tensor-bound prefill and the HBM-bound decode run at the same time. d minimises the
  // larger of the two times of a model with rates measured on GB300: prefill at
  // kSplitPreFlops per SM (128 x 128 tiles counted whole), decode at kSplitDecBytes per SM
  // up to kSplitHbmBytes for the chip.
  const int S = a.sms;
  const bool split = a.split_sms && s_dec_tiles > 0 && s_pre_tiles > 0 && S > 1;
  if (split && a.decode_sms <= 0) {
    const float flops = (float)s_pre_tiles * (float)a.nh * (float)(kPreTileQ * kPreTileK) * (float)a.hs * 4.f;
    const float bytes = (float)s_dec_tiles * (float)a.kvh * (float)(kDecTile * a.hs * 2 * 2);
    // (bytes counts 16-bit K/V. On integer caches the decode side streams a half or a quarter
    // of them, three CTAs per SM, and the prefill side converts codes: per SM the decode
    // kernel gains about 20% on the prefill kernel, the optimum of a sweep on the mixed batch)
    const float dec_rate = kSplitDecBytes * (a.kvq ? 1.2f : 1.f);
    const float hbm = kSplitHbmBytes * (a.kvq == 1 ? 2.f : a.kvq == 2 ? 4.f : 1.f);
    for (int d = tid + 1; d < S; d += blockDim.x) {
      const float tp = flops / ((float)(S - d) * kSplitPreFlops);
      const float td = bytes / fminf(hbm, (float)d * dec_rate);
      atomicMin(&s_split, ((unsigned long long)__float_as_uint(fmaxf(tp, td)) << 32) | (unsigned)d);
    }
  }
  __syncthreads();
  int dec_sms = S;
  if (split) dec_sms = a.decode_sms > 0 ? min(a.decode_sms, S - 1) : (int)(s_split & 0xFFFFFFFFull);
  const int64_t P = split ? min((int64_t)dec_sms * dec_ctas_per_sm(a.hs, a.kvq), (int64_t)a.dec_ctas) : a.dec_ctas;
  const bool balanced = a.forced_split <= 0;
  // The decode units, laid end to end, each as V virtual tiles (the cost of an item beyond
  // its keys) followed by its key tiles, span W tiles; they are cut into P equal ranges:
  // CTA c owns [s_start[c], s_start[c + 1]), s_start[c] = floor(c W / P), and processes the
  // key tiles inside it. So a CTA whose range starts more units pays for them with fewer
  // keys, and the CTAs finish together.
  const int V = dec_item_cost_tiles(a.hs, a.kvq);
  int64_t* s_start = reinterpret_cast<int64_t*>(s_key);   // [kMaxDecCtas + 1]
  int* s_T = reinterpret_cast<int*>(s_start + (kMaxDecCtas + 1));  // [kPlanThreads] first tile of (b, head 0)
  int* s_nt = s_T + kPlanThreads;     // [kPlanThreads] tiles per unit (0: not decode)
  int* s_kv = s_nt + kPlanThreads;    // [kPlanThreads] keys
  int* s_c0 = s_kv + kPlanThreads;    // [kPlanThreads] first packed row
  int* s_past = s_c0 + kPlanThreads;  // [kPlanThreads] history
  static_assert((kMaxDecCtas + 1) * 8 + 5 * kPlanThreads * 4 <= kSortCap * 8, "tables fit s_key");
  const int64_t W = (int64_t)s_dec_tiles * a.kvh;
  {
    // floor(c W / P) = c (W / P) + floor(c (W % P) / P): one 64-bit division per thread, then
    // 32-bit arithmetic per entry (c (W % P) < P^2 <= 2^20)
    const int64_t wq = W / P;
    const uint32_t wr = (uint32_t)(W - wq * P);
    for (int64_t c = tid; c <= P; c += blockDim.x) s_start[c] = c * wq + (uint32_t)c * wr / (uint32_t)P;
  }
  const float pw = W > 0 ? (float)P / (float)W : 0.f;
  // the CTA whose range holds tile t (the largest c with s_start[c] <= t): a float
  // estimate corrected against the table
  auto cta_of = [&](int64_t t) {
    int c = min((int)((float)t * pw), (int)P - 1);
    while (c > 0 && s_start[c] > t) --c;
    while (c + 1 < P && s_start[c + 1] <= t) ++c;
    return c;
  };

  // ---- per-sequence counts, prefix sums, and the lists ----
  for (int base = 0; base < a.B; base += blockDim.x) {
    const int b = base + tid;
    const int carry0 = s_carry[0], carry1 = s_carry[1];
    int64_t q = 0, kv = 0, nt = 0;
    bool dec = false;
    int v[3] = {0, 0, 0};  // [decode tiles of b's units, prefill tiles, prefill-class]
    if (b < a.B) {
      q = (int64_t)a.cum[b + 1] - a.cum[b];
      kv = (int64_t)a.past[b] + q;
      dec = is_decode_class(q, a);
      if (dec) {
        nt = ceil_div(kv, kDecTile);
        v[0] = (int)((nt + V) * a.kvh);
      } else if (q > 0) {
        v[1] = (int)ceil_div(q, kPreTileQ);
      }
    }
    v[2] = v[1] > 0 ? 1 : 0;  // prefill-class sequences (rank among them, for the V copy)
    int ex[3], tot[3];
    block_scan3(v, ex, tot, s_warp);
    // rows of the fp16 V copy: every key of every prefill-class sequence, in sequence order
    int64_t m_ex = 0, m_tot = 0;
    int mrow0 = 0;
    if (a.mirror_keys > 0) {
      block_scan_i64(v[1] > 0 ? kv : 0, &m_ex, &m_tot, s_w64);
      const int64_t mb = s_mirror_carry + m_ex;
      if (v[1] > 0 && mb + kv <= a.mirror_keys) {
        mrow0 = (int)mb;
        a.mirror_base[b] = (int)mb;
        a.mirror_seq[s_mseq_carry + ex[2]] = make_int2(b, (int)mb);
      } else if (b < a.B) {
        a.mirror_base[b] = -1;  // no copy of this sequence's V
      }
    }
    s_T[tid] = carry0 + ex[0];
    s_nt[tid] = dec ? (int)nt : 0;
    s_kv[tid] = (int)kv;
    s_c0[tid] = b < a.B ? a.cum[b] : 0;
    s_past[tid] = (int)(kv - q);
    if (b < a.B) {
      for (int t = 0; t < v[1]; ++t) {
        const int ti = carry1 + ex[1] + t;
        if (ti < a.max_tiles) {
          const int j0 = t * kPreTileQ;
          const int n_kv = (int)ceil_div((int64_t)a.past[b] + min((int64_t)j0 + kPreTileQ, q), kPreTileK);
          a.tiles_unsorted[ti] = PrefillTile{b, j0, a.cum[b], (int)q, a.past[b], n_kv, mrow0, 0};
        }
      }
    }
    __syncthreads();
    // ---- decode items of this round's units, one (sequence, KV head) unit per thread ----
    const int units = min((int)blockDim.x, a.B - base) * a.kvh;
    for (int ub = 0; ub < units; ub += blockDim.x) {
      const int u = ub + tid;
      int sb = 0, g = 0, n_u = 0, kv_u = 0, c0 = 0, c1 = -1, w = 0;
      int64_t u0 = 0;
      if (u < units) {
        sb = u / a.kvh;
        g = u - sb * a.kvh;
        n_u = s_nt[sb];
        if (n_u > 0) {
          kv_u = s_kv[sb];
          u0 = s_T[sb] + (int64_t)g * (n_u + V);  // the unit's span starts here; its keys at u0 + V
          if (balanced) {
            c0 = cta_of(u0 + V);
            c1 = cta_of(u0 + V + n_u - 1);
            w = c1 - c0 + 1;
          } else {
            w = (int)ceil_div(kv_u, a.forced_split);
          }
        }
      }
      int wv[3] = {w, 0, 0}, exw[3], totw[3];
      block_scan3(wv, exw, totw, s_warp);
      int idx = s_carry[2] + exw[0];
      if (w > 0) {
        const int bb = base + sb, unit_first = idx;
        const int row0 = s_c0[sb], past = s_past[sb], q_u = kv_u - past;
        if (balanced) {
          const int64_t k0 = u0 + V, k1 = k0 + n_u;  // the unit's key tiles
          int64_t cs = s_start[c0];
          for (int c = c0; c <= c1; ++c, ++idx) {
            const int64_t ce = s_start[c + 1];
            const int64_t lo = max(k0, cs), hi = min(k1, ce);
            if (idx < a.max_items)
              store_item(a.items + idx, bb, g, (int)((lo - k0) * kDecTile), (int)min((hi - k0) * kDecTile, (int64_t)kv_u),
                         unit_first, w, row0, q_u, past);
            if (cs >= u0) s_cta_begin[c] = idx;  // CTA c's range starts in this unit's span
            cs = ce;
          }
        } else {
          const int64_t S = a.forced_split;
          for (int s2 = 0; s2 < w; ++s2, ++idx) {
            if (idx < a.max_items)
              store_item(a.items + idx, bb, g, (int)(s2 * S), (int)min((s2 + 1) * S, (int64_t)kv_u), unit_first, w, row0,
                         q_u, past);
          }
        }
      }
      __syncthreads();  // every thread has read s_carry[2]
      if (tid == 0) s_carry[2] += totw[0];
      __syncthreads();
    }
    __syncthreads();  // every thread has read the carries of this round
    if (tid == 0) {
      s_carry[0] += tot[0];
      s_carry[1] += tot[1];
      s_mirror_carry += m_tot;
      s_mseq_carry += tot[2];
    }
    __syncthreads();
  }

  const int n_items = s_carry[2], n_tiles = s_carry[1];
  if (n_items > a.max_items || n_tiles > a.max_tiles) {
    // cannot happen for a batch that passed validation (the bounds are proven in
    // ws_layout); refuse rather than run a truncated plan
    if (tid == 0) refuse(hdr);
    return;
  }

  // ---- item range of every decode CTA ----
  if (balanced) {
    // a CTA with an empty range (fewer tiles than CTAs) starts where the next range does
    __syncthreads();
    block_suffix_min(s_cta_begin, (int)P, s_warp[0]);
    for (int c = tid; c < P; c += blockDim.x) s_cta_begin[c] = min(s_cta_begin[c], n_items);
    if (tid == 0) s_cta_begin[P] = n_items;
  } else {
    for (int64_t c = tid; c <= P; c += blockDim.x) s_cta_begin[c] = (int)(c * n_items / P);
  }
  __syncthreads();
  for (int c = tid; c <= a.dec_ctas; c += blockDim.x) a.cta_begin[c] = c <= P ? s_cta_begin[c] : n_items;

  // ---- prefill tiles: sort by KV-tile count, descending (ties: list order) ----
  if (n_tiles <= 256) {
    // few tiles: each takes the place of its rank among the (distinct) keys, two barriers
    unsigned long long key = ~0ull;
    if (tid < n_tiles)
      key = ((unsigned long long)(0xFFFFFFFFull - (unsigned long long)a.tiles_unsorted[tid].n_kv) << 32) |
            (unsigned)tid;
    if (tid < n_tiles) s_key[tid] = key;
    __syncthreads();
    if (tid < n_tiles) {
      int rank = 0;
      for (int j = 0; j < n_tiles; ++j) rank += s_key[j] < key;
      a.tiles[rank] = a.tiles_unsorted[tid];
    }
  } else if (n_tiles <= kSortCap) {
    int n2 = 1;
    while (n2 < n_tiles) n2 <<= 1;
    for (int i = tid; i < n2; i += blockDim.x) {
      unsigned long long key = ~0ull;
      if (i < n_tiles) {
        const int64_t cost = a.tiles_unsorted[i].n_kv;
        key = ((unsigned long long)(0xFFFFFFFFull - (unsigned long long)cost) << 32) | (unsigned)i;
      }
      s_key[i] = key;
    }
    __syncthreads();
    for (int k = 2; k <= n2; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = tid; i < n2; i += blockDim.x) {
          const int ixj = i ^ j;
          if (ixj > i) {
            const unsigned long long x = s_key[i], y = s_key[ixj];
            const bool ascending = (i & k) == 0;
            if ((x > y) == ascending) {
              s_key[i] = y;
              s_key[ixj] = x;
            }
          }
        }
        __syncthreads();
      }
    }
    for (int i = tid; i < n_tiles; i += blockDim.x) a.tiles[i] = a.tiles_unsorted[(unsigned)(s_key[i] & 0xFFFFFFFFull)];
  } else {
    for (int i = tid; i < n_tiles; i += blockDim.x) a.tiles[i] = a.tiles_unsorted[i];
  }
  if (tid == 0) {
    if (a.mirror_keys > 0 && s_mirror_carry > 0 && s_mirror_carry <= a.mirror_keys) {
      hdr->v_mirror = 1;
      hdr->mirror_rows = (int)s_mirror_carry;
      hdr->mirror_seqs = s_mseq_carry;
    }
    hdr->valid = 1;
    hdr->n_decode_items = n_items;
    hdr->n_prefill_tiles = n_tiles;
    hdr->dec_ctas = (int)P;
    hdr->pre_ctas = split ? S - dec_sms : 0;
  }
}

// ---- fp16 copy of V for bf16 prefill ----------------------------------------------------
// Row r of the copy is key r - mirror_base[b] of prefill-class sequence b, read from the
// value cache after this call's cache write (so through block_table, as the attention
// reads it). One warp per row, 16-byte loads and stores. A value fp16 cannot represent
// (|v| >= 65520, inf, NaN) sets v_mirror_bad, and the prefill kernel then reads the bf16
// cache instead; a block outside the pool is flagged and its rows are zeros (as the
// attention reads them from the cache).

// bf16 -> fp16 of the 16-byte chunk w (8 values), folding |fp16| bits into big
__device__ __forceinline__ uint4 chunk_to_f16(uint4 w, uint32_t& big) {
  w.x = bf16x2_to_f16x2(w.x);
  w.y = bf16x2_to_f16x2(w.y);
  w.z = bf16x2_to_f16x2(w.z);
  w.w = bf16x2_to_f16x2(w.w);
  big = max_u16x2(big, max_u16x2(max_u16x2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                                 max_u16x2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu)));
  return w;
}

// copy row r of the fp16 V copy from the value cache (a warp); with history_only, rows of
// this call's keys (position >= past) are left to the cache write, which copies them from
// the inputs
__device__ __forceinline__ void mirror_row(const Args& a, int r, int n_seqs, bool history_only, int lane,
                                           uint32_t& big) {
  const int chunks = a.kv_row / 8;  // 16-byte chunks of a row
  int lo = 0, hi = n_seqs - 1;      // the last copied sequence whose first row is <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.mirror_seq[mid].y <= r) lo = mid; else hi = mid - 1;
  }
  const int b = a.mirror_seq[lo].x;
  const int key = r - a.mirror_seq[lo].y;
  if (history_only && key >= a.past[b]) return;
  const int blk = a.block_table[(int64_t)b * a.max_blocks + key / a.bs];
  const uint4* src = nullptr;
  if (blk >= 0 && blk < a.num_blocks)
    src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.value_cache) +
                                         ((int64_t)blk * a.bs + key % a.bs) * a.kv_row);
  else if (lane == 0)
    atomicOr(&a.hdr->error, PA_DEVERR_BAD_BLOCK);
  uint4* dst = reinterpret_cast<uint4*>(a.mirror + (int64_t)r * a.kv_row);
  for (int c0 = lane; c0 < chunks; c0 += 128) {  // four loads in flight before the stores
    uint4 w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + 32 * j;
      w[j] = (src && c < chunks) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 f = chunk_to_f16(w[j], big);
      if (c0 + 32 * j < chunks) dst[c0 + 32 * j] = f;
    }
  }
}

// ---- cache write ----------------------------------------------------------------------------
// The bit copy, one warp per token: the slot is found once (slot_mapping[i], or the token's
// logical position past_seqlens[b] + j through block_table), then the lanes copy the
// token's K and V rows with 16-byte loads and stores, all loads of a row issued before its
// stores. -1 skips the token; out-of-range slots and blocks are skipped and flagged. With
// the Q/K preparation or integer caches, one warp per query head of the token (prepared or
// scaled into the workspace) and one per KV head (prepared or quantized into the caches).

// RMSNorm and rotary embedding of one head vector spread over the warp, lane l holding
// components [E l, E l + E): x_c <- x_c / sqrt(mean x^2 + eps) * w_c (when w), then the
// pair (u, u + d/2) rotated by the angle whose cos / sin this lane holds (rot lanes).
template <int HS>
__device__ __forceinline__ void prep_vector(float (&x)[HS / 32], bool norm, const float (&w)[HS / 32], float eps,
                                            bool rot, bool first, int partner, const float (&cs)[HS / 32],
                                            const float (&sn)[HS / 32]) {
  constexpr int E = HS / 32;
  if (norm) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = 1.f / sqrtf(ss / HS + eps);
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = x[e] * r * w[e];
  }
  float px[E];
#pragma unroll
  for (int e = 0; e < E; ++e) px[e] = __shfl_sync(0xffffffffu, x[e], partner);
  if (rot) {
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = first ? x[e] * cs[e] - px[e] * sn[e] : x[e] * cs[e] + px[e] * sn[e];
  }
}

template <int HS>
__device__ __forceinline__ void load_vec(const uint16_t* src, bool bf16, float (&x)[HS / 32]) {
  constexpr int E = HS / 32;
  uint32_t wds[E / 2];
  if constexpr (E == 8) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
    wds[0] = v.x;
    wds[1] = v.y;
    wds[2] = v.z;
    wds[3] = v.w;
  } else if constexpr (E == 4) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
    wds[0] = v.x;
    wds[1] = v.y;
  } else {
    wds[0] = __ldg(reinterpret_cast<const uint32_t*>(src));
  }
#pragma unroll
  for (int k = 0; k < E / 2; ++k) {
    if (bf16) {
      x[2 * k] = __uint_as_float(wds[k] << 16);
      x[2 * k + 1] = __uint_as_float(wds[k] & 0xFFFF0000u);
    } else {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wds[k]));
      x[2 * k] = f.x;
      x[2 * k + 1] = f.y;
    }
  }
}

template <int HS>
__device__ __forceinline__ void store_vec(uint16_t* dst, bool bf16, const float (&x)[HS / 32]) {
  constexpr int E = HS / 32;
  uint32_t wds[E / 2];
#pragma unroll
  for (int k = 0; k < E / 2; ++k) wds[k] = bf16 ? pack2<true>(x[2 * k], x[2 * k + 1]) : pack2<false>(x[2 * k], x[2 * k + 1]);
  if constexpr (E == 8) *reinterpret_cast<uint4*>(dst) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
  else if constexpr (E == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(wds[0], wds[1]);
  else *reinterpret_cast<uint32_t*>(dst) = wds[0];
}

// The preparation's per-lane tables for a token at position pos: whether and how this lane's
// components rotate, cos / sin of their fp32 angles, and the norm weights.
template <int HS>
struct PrepLane {
  bool rot, first;
  int partner;
  float cs[HS / 32], sn[HS / 32], wq[HS / 32], wk[HS / 32];
};

template <int HS>
__device__ __forceinline__ void prep_lane(const Args& a, int64_t pos, int lane, PrepLane<HS>& t) {
  constexpr int E = HS / 32;
  const bool bf16 = a.bf16 != 0;
  const int d = a.rotary_dim, half = d / 2;
  const bool rot = d > 0 && lane * E < d;
  const bool first = lane * E < half;
  t.rot = rot;
  t.first = first;
  t.partner = rot ? (first ? lane + half / E : lane - half / E) : lane;
  float* cs = t.cs;
  float* sn = t.sn;
  float* wq = t.wq;
  float* wk = t.wk;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    cs[e] = 1.f;
    sn[e] = 0.f;
    if (rot) {
      const int u = first ? lane * E + e : lane * E + e - half;
      sincosf(__fmul_rn((float)pos, a.inv_freq[u]), &sn[e], &cs[e]);  // the fp32 rotary angle
    }
    wq[e] = a.q_norm_w ? (bf16 ? __uint_as_float((uint32_t)a.q_norm_w[lane * E + e] << 16)
                               : __half2float(*reinterpret_cast<const __half*>(a.q_norm_w + lane * E + e)))
                       : 1.f;
    wk[e] = a.k_norm_w ? (bf16 ? __uint_as_float((uint32_t)a.k_norm_w[lane * E + e] << 16)
                               : __half2float(*reinterpret_cast<const __half*>(a.k_norm_w + lane * E + e)))
                       : 1.f;
  }
}

// Unit u of token tok (a warp): u < nh, query head u prepared into the workspace; else KV
// head g = u - nh, when slot >= 0, its prepared key head into the key cache and its V head
// copied into the value cache.
template <int HS>
__device__ void prep_unit(const Args& a, int tok, int64_t pos, int64_t slot, int u, int lane) {
  constexpr int E = HS / 32;
  const bool bf16 = a.bf16 != 0;
  if (u >= a.nh && slot < 0) return;
  PrepLane<HS> t;
  prep_lane<HS>(a, pos, lane, t);
  const uint16_t* qrow = reinterpret_cast<const uint16_t*>(a.query) + (int64_t)tok * a.q_stride;
  float x[E];
  if (u < a.nh) {
    load_vec<HS>(qrow + u * HS + lane * E, bf16, x);
    prep_vector<HS>(x, a.q_norm_w != nullptr, t.wq, a.norm_eps, t.rot, t.first, t.partner, t.cs, t.sn);
    store_vec<HS>(a.qprep + ((int64_t)tok * a.nh + u) * HS + lane * E, bf16, x);
    return;
  }
  const int g = u - a.nh;
  const uint16_t* krow = a.packed ? qrow + a.k_offset
                                  : reinterpret_cast<const uint16_t*>(a.key) + (int64_t)tok * a.kv_row;
  const uint16_t* vrow = a.packed ? qrow + a.v_offset
                                  : reinterpret_cast<const uint16_t*>(a.value) + (int64_t)tok * a.kv_row;
  uint16_t* kdst = reinterpret_cast<uint16_t*>(a.key_cache) + slot * a.kv_row + g * HS;
  uint16_t* vdst = reinterpret_cast<uint16_t*>(a.value_cache) + slot * a.kv_row + g * HS;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (lane < HS / 8) v = __ldg(reinterpret_cast<const uint4*>(vrow + g * HS) + lane);
  load_vec<HS>(krow + g * HS + lane * E, bf16, x);
  prep_vector<HS>(x, a.k_norm_w != nullptr, t.wk, a.norm_eps, t.rot, t.first, t.partner, t.cs, t.sn);
  store_vec<HS>(kdst + lane * E, bf16, x);
  if (lane < HS / 8) reinterpret_cast<uint4*>(vdst)[lane] = v;
}

// ---- integer caches: this call's K and V rows as codes, the query rows scaled -------------

__device__ __forceinline__ float round_t(float x, bool bf16) {
  return bf16 ? __bfloat162float(__float2bfloat16_rn(x)) : __half2float(__float2half_rn(x));
}

// the code of x for scale s: min(max(rint(x / s), -Q), Q) with the IEEE fp32 quotient
__device__ __forceinline__ int quant_code(float x, float s, float qmax) {
  return (int)fminf(fmaxf(rintf(__fdiv_rn(x, s)), -qmax), qmax);
}

// E consecutive codes of one lane: INT8 one byte each, INT4 one nibble each (first channel
// in the low nibble), little-endian
template <int E, int KQ>
__device__ __forceinline__ void store_codes(uint8_t* dst, const int (&c)[E]) {
  if constexpr (KQ == 1) {
    uint32_t w[(E + 3) / 4] = {};
#pragma unroll
    for (int e = 0; e < E; ++e) w[e / 4] |= (uint32_t)(c[e] & 0xFF) << (8 * (e % 4));
    if constexpr (E == 8) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    else if constexpr (E == 4) *reinterpret_cast<uint32_t*>(dst) = w[0];
    else *reinterpret_cast<uint16_t*>(dst) = (uint16_t)w[0];
  } else {
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) w |= (uint32_t)(c[e] & 0xF) << (4 * e);
    if constexpr (E == 8) *reinterpret_cast<uint32_t*>(dst) = w;
    else if constexpr (E == 4) *reinterpret_cast<uint16_t*>(dst) = (uint16_t)w;
    else *dst = (uint8_t)w;
  }
}

template <int HS, int KQ>
__device__ __forceinline__ void quant_row(const Args& a, const uint16_t* src, const float* scale, uint8_t* dst,
                                          int lane, bool prep, const float (&w)[HS / 32], const PrepLane<HS>& t) {
  constexpr int E = HS / 32;
  const bool bf16 = a.bf16 != 0;
  float x[E];
  load_vec<HS>(src + lane * E, bf16, x);
  if (prep) {  // the prepared key, rounded to T, is what is quantized
    prep_vector<HS>(x, a.k_norm_w != nullptr, w, a.norm_eps, t.rot, t.first, t.partner, t.cs, t.sn);
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = round_t(x[e], bf16);
  }
  int c[E];
#pragma unroll
  for (int e = 0; e < E; ++e) c[e] = quant_code(x[e], __ldg(scale + lane * E + e), KQ == 1 ? 127.f : 7.f);
  store_codes<E, KQ>(dst + lane * E * (KQ == 1 ? 2 : 1) / 2, c);
}

// Unit u of token tok for integer caches (a warp): u < nh, query head u scaled by the K
// scales of its KV head (after the preparation, if any) and written as fp16 with a
// power-of-two row exponent; else KV head g = u - nh, unless the write is suppressed, its
// K and V rows as codes.
template <int HS, int KQ, bool PREP>
__device__ void quant_unit(const Args& a, int tok, int64_t pos, int64_t slot, int u, int lane) {
  constexpr int E = HS / 32;
  const bool bf16 = a.bf16 != 0;
  constexpr bool prep = PREP;
  if (u >= a.nh && slot < 0) return;
  PrepLane<HS> t;
  if constexpr (PREP) prep_lane<HS>(a, pos, lane, t);
  const uint16_t* qrow = reinterpret_cast<const uint16_t*>(a.query) + (int64_t)tok * a.q_stride;
  if (u < a.nh) {
    const int h = u;
    float x[E];
    load_vec<HS>(qrow + h * HS + lane * E, bf16, x);
    if (prep) {
      prep_vector<HS>(x, a.q_norm_w != nullptr, t.wq, a.norm_eps, t.rot, t.first, t.partner, t.cs, t.sn);
#pragma unroll
      for (int e = 0; e < E; ++e) x[e] = round_t(x[e], bf16);
    }
    // q * k_scale, brought to magnitudes in [2^14, 2^15) by 2^-ex: fp16 then keeps 11 bits
    // of every element without overflow, and the attention kernels multiply the scores by
    // 2^ex (exact)
    const float* ks = a.k_scale + (h / a.G) * HS + lane * E;
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      x[e] *= __ldg(ks + e);
      m = fmaxf(m, fabsf(x[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    // ex = floor(log2 m) - 14, from the exponent field of a normal m
    const uint32_t mb = __float_as_uint(m);
    const int ex = !(m > 0.f && m <= 3.4028234e38f) ? 0 : mb >= 0x00800000u ? (int)(mb >> 23) - 127 - 14 : ilogbf(m) - 14;
    // x * 2^-ex as two multiplications by normal powers of two (|ex| <= 163): exact where the
    // result is normal; a value it would take out of the normal range is far below the
    // row's largest and rounds to fp16 zero either way
    const int n0 = -ex / 2, n1 = -ex - n0;
    const float s0 = __uint_as_float((uint32_t)(n0 + 127) << 23), s1 = __uint_as_float((uint32_t)(n1 + 127) << 23);
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = x[e] * s0 * s1;
    store_vec<HS>(a.qprep + ((int64_t)tok * a.nh + h) * HS + lane * E, false, x);
    if (lane == 0) a.qexp[(int64_t)tok * a.nh + h] = ex;
    return;
  }
  const int g = u - a.nh;
  const uint16_t* krow = a.packed ? qrow + a.k_offset
                                  : reinterpret_cast<const uint16_t*>(a.key) + (int64_t)tok * a.kv_row;
  const uint16_t* vrow = a.packed ? qrow + a.v_offset
                                  : reinterpret_cast<const uint16_t*>(a.value) + (int64_t)tok * a.kv_row;
  constexpr int RB = KQ == 1 ? HS : HS / 2;  // bytes of one KV head's code row
  uint8_t* kdst = reinterpret_cast<uint8_t*>(a.key_cache) + slot * a.kvh * RB;
  uint8_t* vdst = reinterpret_cast<uint8_t*>(a.value_cache) + slot * a.kvh * RB;
  quant_row<HS, KQ>(a, krow + g * HS, a.k_scale + g * HS, kdst + g * RB, lane, prep, t.wk, t);
  quant_row<HS, KQ>(a, vrow + g * HS, a.v_scale + g * HS, vdst + g * RB, lane, false, t.wk, t);
}

// Integer caches without the Q/K preparation, in wider tasks: a task covers 256 values of
// one token, 8 per lane (one 16-byte load): 256 / HS consecutive query heads (scaled by the
// K scales of their KV heads and written as fp16 with a power-of-two row exponent, as in
// quant_unit) or 256 / HS consecutive KV heads' K and V rows (written as codes). A token's
// tasks are its query tasks, then its KV tasks; the last of each kind may cover fewer heads.
// Split into the loads and the rest, so that a warp keeps two tasks' loads in flight.
template <int HS, int KQ>
struct QuantTask {
  static constexpr int LPH = HS / 8;    // lanes per head row
  static constexpr int RPW = 32 / LPH;  // head rows per task
  int tok, h;                            // this lane's head (query or KV)
  bool kv, active;
  int64_t slot;
  uint4 x, y;  // this lane's 8 query values, or 8 K and 8 V values

  __device__ __forceinline__ void load(const Args& a, int tok_, int u, int QT, int64_t slot_, int lane) {
    tok = tok_;
    kv = u >= QT;
    h = (kv ? u - QT : u) * RPW + lane / LPH;
    slot = slot_;
    const uint16_t* qrow = reinterpret_cast<const uint16_t*>(a.query) + (int64_t)tok * a.q_stride;
    const int off = h * HS + (lane % LPH) * 8;
    if (!kv) {
      active = h < a.nh;
      if (active) x = __ldg(reinterpret_cast<const uint4*>(qrow + off));
    } else {
      active = h < a.kvh && slot >= 0;
      if (active) {
        const uint16_t* krow = a.packed ? qrow + a.k_offset
                                        : reinterpret_cast<const uint16_t*>(a.key) + (int64_t)tok * a.kv_row;
        const uint16_t* vrow = a.packed ? qrow + a.v_offset
                                        : reinterpret_cast<const uint16_t*>(a.value) + (int64_t)tok * a.kv_row;
        x = __ldg(reinterpret_cast<const uint4*>(krow + off));
        y = __ldg(reinterpret_cast<const uint4*>(vrow + off));
      }
    }
  }

  static __device__ __forceinline__ void pair_f32(uint32_t w, bool bf16, float& lo, float& hi) {
    if (bf16) {
      lo = __uint_as_float(w << 16);
      hi = __uint_as_float(w & 0xFFFF0000u);
    } else {
      lo = __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
      hi = __half2float(__ushort_as_half((unsigned short)(w >> 16)));
    }
  }
  static __device__ __forceinline__ void to_f32(uint4 w, bool bf16, float (&v)[8]) {
    pair_f32(w.x, bf16, v[0], v[1]);
    pair_f32(w.y, bf16, v[2], v[3]);
    pair_f32(w.z, bf16, v[4], v[5]);
    pair_f32(w.w, bf16, v[6], v[7]);
  }
  static __device__ __forceinline__ void scales8(const float* p, float (&s)[8]) {
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(p)), s1 = __ldg(reinterpret_cast<const float4*>(p + 4));
    s[0] = s0.x, s[1] = s0.y, s[2] = s0.z, s[3] = s0.w, s[4] = s1.x, s[5] = s1.y, s[6] = s1.z, s[7] = s1.w;
  }

  // (the whole warp: the query rows' maxima are reduced across each head's lanes)
  __device__ __forceinline__ void finish(const Args& a, int lane) {
    const bool bf16 = a.bf16 != 0;
    const int c0 = (lane % LPH) * 8;  // this lane's first channel
    if (!kv) {
      float v[8], sc[8];
      to_f32(active ? x : make_uint4(0, 0, 0, 0), bf16, v);
      scales8(a.k_scale + (active ? (h / a.G) * HS : 0) + c0, sc);
      float m = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v[e] *= sc[e];
        m = fmaxf(m, fabsf(v[e]));
      }
#pragma unroll
      for (int o = 1; o < LPH; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (!active) return;
      const uint32_t mb = __float_as_uint(m);
      const int ex = !(m > 0.f && m <= 3.4028234e38f) ? 0 : mb >= 0x00800000u ? (int)(mb >> 23) - 127 - 14 : ilogbf(m) - 14;
      const int n0 = -ex / 2, n1 = -ex - n0;
      const float s0 = __uint_as_float((uint32_t)(n0 + 127) << 23), s1 = __uint_as_float((uint32_t)(n1 + 127) << 23);
      uint32_t wds[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) wds[k] = pack2<false>(v[2 * k] * s0 * s1, v[2 * k + 1] * s0 * s1);
      *reinterpret_cast<uint4*>(a.qprep + ((int64_t)tok * a.nh + h) * HS + c0) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
      if (lane % LPH == 0) a.qexp[(int64_t)tok * a.nh + h] = ex;
      return;
    }
    if (!active) return;
    constexpr int RB = KQ == 1 ? HS : HS / 2;  // bytes of one KV head's code row
    const float qmax = KQ == 1 ? 127.f : 7.f;
    float v[8], sc[8];
    int c[8];
    to_f32(x, bf16, v);
    scales8(a.k_scale + h * HS + c0, sc);
#pragma unroll
    for (int e = 0; e < 8; ++e) c[e] = quant_code(v[e], sc[e], qmax);
    uint8_t* kdst = reinterpret_cast<uint8_t*>(a.key_cache) + (slot * a.kvh + h) * RB + c0 * RB / HS;
    store_codes<8, KQ>(kdst, c);
    to_f32(y, bf16, v);
    scales8(a.v_scale + h * HS + c0, sc);
#pragma unroll
    for (int e = 0; e < 8; ++e) c[e] = quant_code(v[e], sc[e], qmax);
    uint8_t* vdst = reinterpret_cast<uint8_t*>(a.value_cache) + (slot * a.kvh + h) * RB + c0 * RB / HS;
    store_codes<8, KQ>(vdst, c);
  }
};

// The slot of token tok (slot_mapping[tok], or its logical position through block_table),
// -1 for a suppressed write or an out-of-range block or slot (those also flagged: in the
// error word, or with DEFER in errs, which the caller adds to the word once the planner has
// reset it); pos is
// the token's logical position when the caller needs it (no slot_mapping, or prep). b is
// the sequence of the warp's previous token, tokens only grow within a warp.
// The last b in [b0, B) with cum[b] <= tok (given cum[b0] <= tok), found by the warp: each
// step has the 32 lanes test 32 evenly spaced entries of the range and keeps the bracket
// of the last one that holds, so up to 32^k sequences take k dependent loads instead of a
// binary search's log2 of them. Empty sequences (cum[b] = cum[b + 1]) are passed over.
__device__ __forceinline__ int warp_find_seq(const int* cum, int b0, int B, int tok, int lane) {
  int lo = b0, n = B - b0;
  while (n > 32) {
    const int stride = (n + 31) >> 5;
    const int idx = lo + lane * stride;
    const unsigned m = __ballot_sync(0xffffffffu, idx < lo + n && cum[idx] <= tok);
    const int k = 31 - __clz(m);  // lane 0 holds: cum[lo] <= tok
    lo += k * stride;
    n = min(stride, n - k * stride);
  }
  const unsigned m = __ballot_sync(0xffffffffu, lane < n && cum[lo + lane] <= tok);
  return lo + 31 - __clz(m);
}

template <bool DEFER = false>
__device__ __forceinline__ int64_t resolve_slot(const Args& a, int tok, bool need_pos, int& b, int64_t& pos,
                                                uint32_t& errs) {
  const int lane = threadIdx.x & 31;
  auto flag = [&](uint32_t bit) {
    if constexpr (DEFER) errs |= bit;
    else if (lane == 0) atomicOr(&a.hdr->error, bit);
  };
  pos = 0;
  if (!a.slot_mapping || need_pos) {
    b = warp_find_seq(a.cum, b, a.B, tok, lane);
    pos = (int64_t)a.past[b] + (tok - a.cum[b]);
  }
  int64_t slot;
  if (a.slot_mapping) {
    slot = a.slot_mapping[tok];
  } else {
    const int blk = a.block_table[(int64_t)b * a.max_blocks + pos / a.bs];
    if (blk < 0 || blk >= a.num_blocks) {
      flag(PA_DEVERR_BAD_BLOCK);
      slot = -1;
    } else {
      slot = (int64_t)blk * a.bs + pos % a.bs;
    }
  }
  if (slot != -1 && (slot < 0 || slot >= (int64_t)a.num_blocks * a.bs)) {
    flag(PA_DEVERR_BAD_SLOT);
    slot = -1;
  }
  return slot;
}

// A warp's contiguous run of the QuantTask list (the tokens' query tasks, then their KV
// tasks), two tasks at a time: both loads are issued before either task is finished. The
// token's slot is resolved once, when the run reaches the token.
template <int HS, int KQ>
__device__ void quant_tasks(const Args& a, int gw, int warps, int lane, uint32_t& errs) {
  using QT_ = QuantTask<HS, KQ>;
  const int QT = (a.nh + QT_::RPW - 1) / QT_::RPW, KT = (a.kvh + QT_::RPW - 1) / QT_::RPW, T = QT + KT;
  const int64_t total = (int64_t)a.N * T;
  const int64_t per = (total + warps - 1) / warps;
  const int64_t w0 = (int64_t)gw * per, w1 = min(total, w0 + per);
  int b = 0, cur = -1;
  int64_t pos = 0, slot = -1;
  auto start = [&](QT_& t, int64_t wj) {
    const int tok = (int)(wj / T), u = (int)(wj - (int64_t)tok * T);
    if (tok != cur) {
      cur = tok;
      slot = resolve_slot(a, tok, false, b, pos, errs);
    }
    t.load(a, tok, u, QT, slot, lane);
  };
  for (int64_t wi = w0; wi < w1; wi += 2) {
    const bool two = wi + 1 < w1;
    QT_ t0, t1;
    start(t0, wi);
    if (two) start(t1, wi + 1);
    t0.finish(a, lane);
    if (two) t1.finish(a, lane);
  }
}

// The first row of sequence b in the fp16 V copy, worked out by a warp as the planner lays
// the copy out (the keys of every prefill-class sequence in sequence order; the copy is made
// only if all of them fit), or -1 for a sequence without a copy: the bit copy beside the
// planner writes the copy of this call's rows without waiting for the plan.
__device__ __forceinline__ int own_mirror_base(const Args& a, int b, int lane) {
  int64_t before = 0, total = 0, mine = 0;
  for (int i = lane; i < a.B; i += 32) {
    const int64_t q = (int64_t)a.cum[i + 1] - a.cum[i];
    const int64_t rows = (q > 0 && !is_decode_class(q, a)) ? (int64_t)a.past[i] + q : 0;
    total += rows;
    if (i < b) before += rows;
    if (i == b) mine = rows;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    total += __shfl_xor_sync(0xffffffffu, total, o);
    before += __shfl_xor_sync(0xffffffffu, before, o);
    mine += __shfl_xor_sync(0xffffffffu, mine, o);
  }
  return (mine > 0 && total <= a.mirror_keys) ? (int)before : -1;
}

// One instantiation per kind of write, so that each keeps only the registers it needs and
// stays many warps deep (at most 64 registers: four blocks of 256 per SM): 0 = bit copy,
// one warp per token, 4 = the same beside this call's planner, 5 = that with the fp16 V
// copy; 1 = Q/K preparation, 2 = integer caches, 3 = both, over (token, unit) tasks, the
// units being the token's nh query heads and then its kvh KV heads (each a short dependent
// chain of a load, warp reductions and a store); each warp takes a contiguous run of them.
template <int MODE>
__global__ void __launch_bounds__(256, 4) cache_write_kernel(const Args a) {
  constexpr bool COPY = MODE == 0 || MODE >= 4;  // bit copy
  constexpr bool early = MODE >= 4;
  const int lane = threadIdx.x & 31;
  const int warps = (int)((gridDim.x * blockDim.x) >> 5);
  const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  // bit copy: each warp takes a contiguous run of tokens [tok0, tok1), so that consecutive
  // tokens of a sequence reuse its lookup (and usually its page)
  const int per_warp = (a.N + warps - 1) / warps;
  const int tok0 = min(a.N, gw * per_warp), tok1 = min(a.N, tok0 + per_warp);
  if constexpr (COPY) {
    // this warp's tokens' K and V rows and the batch description into L2 while the earlier
    // kernels finish and the tokens' slots are resolved (hints only)
    {
      const int lines = a.kv_row * 2 / 128;  // 128-byte lines of one K (or V) row
      const int64_t vdelta = a.packed ? (int64_t)(a.v_offset - a.k_offset) * 2
                                      : reinterpret_cast<const char*>(a.value) - reinterpret_cast<const char*>(a.key);
      for (int i = lane; i < 2 * lines * (tok1 - tok0); i += 32) {
        const int tk = tok0 + i / (2 * lines), li = i % (2 * lines);
        const char* src = a.packed ? reinterpret_cast<const char*>(a.query) + ((int64_t)tk * a.q_stride + a.k_offset) * 2
                                   : reinterpret_cast<const char*>(a.key) + (int64_t)tk * a.kv_row * 2;
        prefetch_l2(src + (li >= lines ? vdelta : 0) + (li % lines) * 128);
      }
    }
    if (threadIdx.x < 32)
      for (int i = lane * 32; i <= a.B; i += 32 * 32) {
        prefetch_l2(a.cum + i);
        if (i < a.B) prefetch_l2(a.past + i);
      }
  }
  // A bit copy launched right after this call's planner starts once the planner's own wait
  // has returned (so every earlier call is finished) and copies the rows beside it, after
  // checking the batch as the planner does, so that a refused batch writes nothing; it waits
  // for the plan before the fp16 V copy, its error bits (the planner resets the word) and
  // its exit, so its completion still implies the planner's.
  uint32_t errs = 0;  // (lane 0 of each warp flags bad blocks and slots)
  if constexpr (early) {
    bool bad = threadIdx.x == 0 && (a.cum[0] != 0 || a.cum[a.B] != a.N);
    for (int bb = threadIdx.x; bb < a.B; bb += blockDim.x) {
      const int64_t q = (int64_t)a.cum[bb + 1] - a.cum[bb], kv = (int64_t)a.past[bb] + q;
      bad |= q < 0 || a.past[bb] < 0 || kv > (int64_t)a.max_blocks * a.bs ||
             (a.max_query_len > 0 && q > a.max_query_len);
    }
    if (__syncthreads_or(bad)) {
      pdl_wait();
      return;
    }
  } else {
    pdl_wait();
    pdl_launch_dependents();
    if (!a.hdr->valid) return;
  }
  if constexpr (!COPY) {
    if (a.self_plan) {
      // no planner ran: refuse an inconsistent batch here as well (the decode kernel, which
      // checks it too, reports it), so that nothing is written
      bool bad = threadIdx.x == 0 && (a.cum[0] != 0 || a.cum[a.B] != a.N);
      for (int bb = threadIdx.x; bb < a.B; bb += blockDim.x) {
        const int64_t q = (int64_t)a.cum[bb + 1] - a.cum[bb], kv = (int64_t)a.past[bb] + q;
        bad |= q < 0 || a.past[bb] < 0 || kv > (int64_t)a.max_blocks * a.bs ||
               (a.max_query_len > 0 && q > a.max_query_len);
      }
      if (__syncthreads_or(bad)) return;
    }
  }
  if constexpr (MODE == 2) {  // integer caches without the preparation: the wider tasks
    if (a.kvq == 1) {
      if (a.hs == 128) quant_tasks<128, 1>(a, gw, warps, lane, errs);
      else if (a.hs == 256) quant_tasks<256, 1>(a, gw, warps, lane, errs);
      else quant_tasks<64, 1>(a, gw, warps, lane, errs);
    } else {
      if (a.hs == 128) quant_tasks<128, 2>(a, gw, warps, lane, errs);
      else quant_tasks<256, 2>(a, gw, warps, lane, errs);
    }
    return;
  }
  if constexpr (!COPY) {
    int b = 0;
    const int U = a.nh + a.kvh;
    const int64_t total = (int64_t)a.N * U;
    // Each warp takes a contiguous run of (token, unit) tasks: it resolves a token's slot once,
    // and when it starts on a token it asks for the token's rows in L2, so that the loads of
    // the token's units (one after the other, each a chain of load, reduction and store)
    // find them there.
    const int64_t per = (total + warps - 1) / warps;
    const int64_t w0 = (int64_t)gw * per, w1 = min(total, w0 + per);
    int cur = -1;
    int64_t pos = 0, slot = -1;
    for (int64_t wi = w0; wi < w1; ++wi) {
      const int tok = (int)(wi / U), u = (int)(wi - (int64_t)tok * U);
      if (tok != cur) {
        cur = tok;
        const char* q = reinterpret_cast<const char*>(a.query) + (int64_t)tok * a.q_stride * 2;
        const int qlines = a.q_stride * 2 / 128;  // (packed rows hold K and V too)
        for (int i = lane; i < qlines; i += 32) prefetch_l2(q + i * 128);
        if (!a.packed) {
          const int kvlines = a.kv_row * 2 / 128;
          for (int i = lane; i < 2 * kvlines; i += 32)
            prefetch_l2(reinterpret_cast<const char*>(i < kvlines ? a.key : a.value) +
                        ((int64_t)tok * a.kv_row * 2 + (i % kvlines) * 128));
        }
        slot = resolve_slot(a, tok, true, b, pos, errs);  // (after the wait: flagged at once)
      }
      if constexpr (MODE >= 2) {  // (the query rows are scaled even where the K/V write is skipped)
        constexpr bool PREP = MODE == 3;
        if (a.kvq == 1) {
          if (a.hs == 128) quant_unit<128, 1, PREP>(a, tok, pos, slot, u, lane);
          else if (a.hs == 256) quant_unit<256, 1, PREP>(a, tok, pos, slot, u, lane);
          else quant_unit<64, 1, PREP>(a, tok, pos, slot, u, lane);
        } else {
          if (a.hs == 128) quant_unit<128, 2, PREP>(a, tok, pos, slot, u, lane);
          else quant_unit<256, 2, PREP>(a, tok, pos, slot, u, lane);
        }
      } else {  // (the query rows are prepared even where the K/V write is skipped)
        if (a.hs == 128) prep_unit<128>(a, tok, pos, slot, u, lane);
        else if (a.hs == 256) prep_unit<256>(a, tok, pos, slot, u, lane);
        else prep_unit<64>(a, tok, pos, slot, u, lane);
      }
    }
    return;
  }
  const int chunks = a.kv_row / 8;  // 16-byte chunks in one K (or V) row
  uint32_t big = 0;  // per-half max of |fp16| bits of this lane's copied values
  // One pass over this warp's tokens: the K and V rows into the cache (kv) and, for bf16 with
  // derived slots, the fp16 copy of the prefill-class sequences' V (mirror): each new row
  // from the input it comes from (this call writes every derived position, and no other
  // position), the older rows from the cache afterwards; no copy kernel runs.
  // (compile-time flags, so that each pass keeps only its registers; mirror: 0 none, 1 by the
  // planner's layout, 2 by the layout worked out here)
  auto pass = [&](auto kv_c, auto mirror_c, auto defer_c) {
    constexpr bool kv = decltype(kv_c)::value;
    constexpr int mirror = decltype(mirror_c)::value;
    int b = 0, mb = -1, mb_of = -1;  // (the last sequence's first copy row)
    for (int tok = tok0; tok < tok1; ++tok) {
      int64_t pos;
      const int64_t slot = resolve_slot<decltype(defer_c)::value>(a, tok, false, b, pos, errs);
      int mrow = -1;  // the token's row of the fp16 V copy
      if constexpr (mirror == 1) {
        const int base = a.mirror_base[b];
        if (base >= 0) mrow = base + (int)pos;
      } else if constexpr (mirror == 2) {
        if (b != mb_of) {
          mb = own_mirror_base(a, b, lane);
          mb_of = b;
        }
        if (mb >= 0) mrow = mb + (int)pos;
      }
      if (slot == -1) {  // (derived slots: a block outside the pool, which reads as zeros)
        if (mrow >= 0)
          for (int c = lane; c < chunks; c += 32)
            reinterpret_cast<uint4*>(a.mirror + (int64_t)mrow * a.kv_row)[c] = make_uint4(0, 0, 0, 0);
        continue;
      }
      if (!kv && mrow < 0) continue;
      const uint16_t *src_k, *src_v;
      if (a.packed) {
        src_k = reinterpret_cast<const uint16_t*>(a.query) + (int64_t)tok * a.q_stride + a.k_offset;
        src_v = reinterpret_cast<const uint16_t*>(a.query) + (int64_t)tok * a.q_stride + a.v_offset;
      } else {
        src_k = reinterpret_cast<const uint16_t*>(a.key) + (int64_t)tok * a.kv_row;
        src_v = reinterpret_cast<const uint16_t*>(a.value) + (int64_t)tok * a.kv_row;
      }
      uint4* dst_k = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.key_cache) + slot * a.kv_row);
      uint4* dst_v = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.value_cache) + slot * a.kv_row);
      for (int c0 = lane; c0 < chunks; c0 += 128) {
        uint4 k[4], v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = c0 + 32 * j;
          if (c < chunks) {
            if constexpr (kv) k[j] = __ldg(reinterpret_cast<const uint4*>(src_k) + c);
            v[j] = __ldg(reinterpret_cast<const uint4*>(src_v) + c);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = c0 + 32 * j;
          if (c < chunks) {
            if constexpr (kv) {
              dst_k[c] = k[j];
              dst_v[c] = v[j];
            }
            if (mrow >= 0) reinterpret_cast<uint4*>(a.mirror + (int64_t)mrow * a.kv_row)[c] = chunk_to_f16(v[j], big);
          }
        }
      }
    }
  };
  using yes = std::true_type;
  using no = std::false_type;
  using m0 = std::integral_constant<int, 0>;
  using m1 = std::integral_constant<int, 1>;
  using m2 = std::integral_constant<int, 2>;
  if constexpr (early) {
    // (errors kept in errs: the planner resets the error word)
    if constexpr (MODE == 5) pass(yes{}, m2{}, yes{});
    else pass(yes{}, m0{}, yes{});
    pdl_wait();  // the plan (the copy's history rows), and the error word reset
    pdl_launch_dependents();
    if (lane == 0 && errs) atomicOr(&a.hdr->error, errs);
  }
  const bool mirror = a.mirror_keys > 0 && !a.slot_mapping && a.hdr->v_mirror;
  if constexpr (!early) {
    if (mirror) pass(yes{}, m1{}, no{});
    else pass(yes{}, m0{}, no{});
  }
  if (mirror) {  // the copy's rows of keys before this call
    const int rows = a.hdr->mirror_rows, n = a.hdr->mirror_seqs;
    for (int r = gw; r < rows; r += warps) mirror_row(a, r, n, true, lane, big);
  }
  if ((big & 0xFFFFu) >= 0x7C00u || (big >> 16) >= 0x7C00u) atomicOr(&a.hdr->v_mirror_bad, 1u);
}

__global__ void __launch_bounds__(256) v_mirror_kernel(const Args a) {
  pdl_wait();
  pdl_launch_dependents();
  const WsHeader* hdr = a.hdr;
  if (!hdr->valid || !hdr->v_mirror) return;
  const int rows = hdr->mirror_rows;
  const int lane = threadIdx.x & 31;
  uint32_t big = 0;  // per-half max of |fp16| bits over this lane's values
  const int n = hdr->mirror_seqs;
  for (int r = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); r < rows; r += (int)((gridDim.x * blockDim.x) >> 5))
    mirror_row(a, r, n, false, lane, big);
  if ((big & 0xFFFFu) >= 0x7C00u || (big >> 16) >= 0x7C00u) atomicOr(&a.hdr->v_mirror_bad, 1u);
}

// ---- host launchers ----
cudaError_t launch_plan(const Args& a, cudaStream_t s) {
  return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, a);
}

cudaError_t launch_cache_write(const Args& a, int sms, cudaStream_t s) {
  // a warp per token (bit copy) or per (token, unit): one resident wave of 8-warp blocks
  // (four per SM at 64 registers), each warp looping over its share
  // (integer caches without the preparation: tasks of 256 values, two per warp at a time)
  const int64_t warps = a.kvq && !a.prep ? ((int64_t)a.N * ((a.nh + a.kvh) * a.hs + 255) / 256 + 1) / 2
                                         : (int64_t)a.N * ((a.kvq || a.prep) ? a.nh + a.kvh : 1);
  const int grid = (int)std::min<int64_t>((warps + 7) / 8, (int64_t)sms * 4);
  if (a.kvq) return launch_pdl(a.prep ? cache_write_kernel<3> : cache_write_kernel<2>, dim3(grid), dim3(256), 0, s, a);
  if (a.prep) return launch_pdl(cache_write_kernel<1>, dim3(grid), dim3(256), 0, s, a);
  if (a.cw_early)
    return launch_pdl(a.mirror_keys > 0 && !a.slot_mapping ? cache_write_kernel<5> : cache_write_kernel<4>, dim3(grid),
                      dim3(256), 0, s, a);
  return launch_pdl(cache_write_kernel<0>, dim3(grid), dim3(256), 0, s, a);
}

cudaError_t launch_v_mirror(const Args& a, int grid, cudaStream_t s) {
  return launch_pdl(v_mirror_kernel, dim3(grid), dim3(256), 0, s, a);
}

}  // namespace pa
