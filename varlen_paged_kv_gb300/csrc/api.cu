// C ABI of the library (include/pagedattn.h): argument checks, workspace carving, TMA
// tensor-map encoding and the launch sequence plan -> cache write -> (bf16: fp16 copy of
// the prefill sequences' V) -> prefill -> decode (with its merge) on the caller's stream. No allocation, no host/device synchronisation.
#include <algorithm>
#include <cstdio>
#include <atomic>
#include <mutex>

#include "common.cuh"


namespace {

std::atomic<uint64_t> g_launches{0};
// coverage counters of the PA_COVERAGE debug library (pa_debug_coverage)
std::atomic<int32_t*> g_cov{nullptr};
std::atomic<int32_t> g_cov_keys{0};
thread_local const char* g_last_error = "no error";

// record a failing CUDA call's message (per host thread) and map it to PA_ERR_CUDA
pa_status cuda_fail(cudaError_t e, const char* what) {
  static thread_local char buf[256];
  snprintf(buf, sizeof(buf), "%s: %s", what, cudaGetErrorString(e));
  g_last_error = buf;
  return PA_ERR_CUDA;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D map over a cache viewed as (head_size, kv_heads, slots); box = 64 x 1 x rows, 128B swizzle
bool cache_map(CUtensorMap* m, void* base, pa_dtype dt, int hs, int kvh, int64_t slots, int rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)hs, (cuuint64_t)kvh, (cuuint64_t)slots};
  cuuint64_t strides[2] = {(cuuint64_t)hs * 2, (cuuint64_t)kvh * hs * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dt == PA_BFLOAT16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims,
             strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over the query rows (row width in elements, rows); box = 64 x 128, 128B swizzle
bool query_map(CUtensorMap* m, const void* base, pa_dtype dt, int64_t width, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)width * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)pa::kPreTileQ};
  cuuint32_t es[2] = {1, 1};
  return enc(m, dt == PA_BFLOAT16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
             const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gcd(int a, int b) {
  while (b) {
    int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct DeviceInfo {
  int dev = 0;
  int sms = 0;
};

bool device_info(DeviceInfo* info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  static std::mutex mu;
  static int cached_sms[64] = {0};
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return false;
  if (!cached_sms[dev]) {
    if (cudaDeviceGetAttribute(&cached_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
  }
  info->dev = dev;
  info->sms = cached_sms[dev];
  return true;
}

// Sizes-only validation (no pointers, no CUDA calls).
pa_status check_dims(const pa_dims* d, int32_t nh, int32_t kvh) {
  if (!d) return PA_ERR_INVALID_ARGUMENT;
  if (d->num_tokens < 0 || d->batch_size < 0 || d->num_blocks < 0 || d->max_blocks_per_sequence < 0)
    return PA_ERR_INVALID_ARGUMENT;
  if (d->num_tokens > 0 && d->batch_size == 0) return PA_ERR_INVALID_ARGUMENT;
  if (nh <= 0 || kvh <= 0 || nh % kvh != 0) return PA_ERR_INVALID_ARGUMENT;
  if (d->block_size <= 0 || d->head_size <= 0) return PA_ERR_INVALID_ARGUMENT;
  if (d->dtype != PA_FLOAT16 && d->dtype != PA_BFLOAT16) return PA_ERR_UNSUPPORTED;
  if (d->head_size != 64 && d->head_size != 128 && d->head_size != 256) return PA_ERR_UNSUPPORTED;
  if (d->kv_dtype != PA_KV_SAME && d->kv_dtype != PA_KV_INT8 && d->kv_dtype != PA_KV_INT4) return PA_ERR_UNSUPPORTED;
  if (d->kv_dtype == PA_KV_INT4 && d->head_size == 64) return PA_ERR_UNSUPPORTED;
  if (d->block_size % 16 != 0) return PA_ERR_UNSUPPORTED;
  if (d->route != PA_ROUTE_AUTO && d->route != PA_ROUTE_ALL_PREFILL) return PA_ERR_INVALID_ARGUMENT;
  if (d->decode_split_keys < 0 || d->decode_split_keys % pa::kDecTile != 0) return PA_ERR_INVALID_ARGUMENT;
  if (d->max_query_len < 0) return PA_ERR_INVALID_ARGUMENT;
  if ((int64_t)d->num_blocks * d->block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if ((int64_t)d->max_blocks_per_sequence * d->block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if ((int64_t)nh * d->head_size > 65536 || kvh > 65536) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

// Whether any sequence may take the prefill kernel: with the automatic route, a host bound
// max_query_len with max_query_len * G <= 16 proves every sequence decode-class.
bool prefill_possible(const pa_dims* d, int32_t G) {
  return !(d->route == PA_ROUTE_AUTO && d->max_query_len > 0 && (int64_t)d->max_query_len * G <= pa::kDecRows);
}

// Rows of the fp16 copy of V that bf16 prefill reads: room for an average of four keys of
// history (past and new) per new token, at most the cache's size. A call whose
// prefill-class sequences hold more keys than that, or whose V holds a value fp16 cannot
// represent, takes the two-product path on the bf16 cache instead (same results within
// rounding, slower).
int64_t mirror_keys(const pa_dims* d, int32_t nh, int32_t kvh) {
  if (d->dtype != PA_BFLOAT16 || d->kv_dtype != PA_KV_SAME || !prefill_possible(d, nh / kvh)) return 0;
  return std::min<int64_t>(4 * (int64_t)d->num_tokens, (int64_t)d->num_blocks * d->block_size);
}

// 16-bit values of the prepared (dims->qk_prep) or scaled (integer caches) query rows the
// workspace holds, and the scaled rows' exponents
int64_t qprep_values(const pa_dims* d, int32_t nh) {
  return (d->qk_prep || d->kv_dtype != PA_KV_SAME) ? (int64_t)d->num_tokens * nh * d->head_size : 0;
}
int64_t qexp_values(const pa_dims* d, int32_t nh) {
  return d->kv_dtype != PA_KV_SAME ? (int64_t)d->num_tokens * nh : 0;
}

// 3-D map over an integer cache viewed as (row bytes, kv_heads, slots), uint8 elements; box =
// min(row bytes, 128) x 1 x rows with the swizzle of that width
bool code_cache_map(CUtensorMap* m, void* base, int row_bytes, int kvh, int64_t slots, int rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const int box = row_bytes < 128 ? row_bytes : 128;
  cuuint64_t dims[3] = {(cuuint64_t)row_bytes, (cuuint64_t)kvh, (cuuint64_t)slots};
  cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)kvh * row_bytes};
  cuuint32_t boxd[3] = {(cuuint32_t)box, 1, (cuuint32_t)rows};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, boxd, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             box == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             // a box row is one head's code row: fetch what it covers (the next head's row
             // at the next 128 or 64 bytes belongs to another CTA's tile)
             box == 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over an integer cache viewed as (kv_heads * row bytes, slots), uint8 elements; box =
// 128 bytes x rows from a head's row start (that head's code row, then the next head's, read
// and not used; zeros past the last head), 128-byte swizzle: the prefill kernel's code tiles
bool code_tile_map(CUtensorMap* m, void* base, int row_bytes, int kvh, int64_t slots, int rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kvh * row_bytes, (cuuint64_t)slots};
  cuuint64_t strides[1] = {(cuuint64_t)kvh * row_bytes};
  cuuint32_t boxd[2] = {128, (cuuint32_t)rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, boxd, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

pa_status launch_all(pa::Args& args, const pa_dims* d, const void* query, void* kc, void* vc, uint32_t stages,
                     cudaStream_t stream) {
  DeviceInfo info;
  if (!device_info(&info)) return cuda_fail(cudaGetLastError(), "device query");
  args.dec_ctas = std::min(pa::dec_ctas_per_sm(args.hs, args.kvq) * info.sms, pa::kMaxDecCtas);
  args.sms = info.sms;
  // The program of a call (which kernels, on which SMs) follows from its arguments alone;
  // `stages` only picks which of its kernels this call launches. A call with prefill-class
  // and decode-class rows may run its two attention kernels side by side on split SMs (the
  // planner decides); they run side by side when one call launches both.
  args.split_sms = 1;
  const pa_dtype dt = (pa_dtype)d->dtype;
  const bool bf16 = dt == PA_BFLOAT16;
  const int hs = args.hs;
  const int64_t slots = (int64_t)d->num_blocks * d->block_size;

  // A decode-only call (proven by the host bound) with derived slots and a small batch
  // needs no planner and no cache-write kernel: a one-CTA reset, then the decode kernel plans
  // its own share and writes the new rows of the tiles it loads.
  // (With the Q/K preparation or integer caches the cache-write kernel still runs: it writes
  // the prepared or scaled query rows and the rows' codes, checking the batch itself.)
  // Its stages: PA_STAGE_PLAN is that reset, PA_STAGE_CACHE_WRITE is empty when the decode
  // kernel writes the rows, PA_STAGE_DECODE is the self-planned decode kernel.
  const bool self_plan = d->route == PA_ROUTE_AUTO && d->max_query_len > 0 &&
                         (int64_t)d->max_query_len * args.G <= pa::kDecRows && args.slot_mapping == nullptr &&
                         args.forced_split <= 0 && args.B >= 1 && args.B <= pa::self_max_b(hs) && args.N > 0 &&
                         slots > 0;
  const bool self_write_rows = self_plan && !args.prep && !args.kvq;
  // integer caches with every decode item at most 8 rows: the decode kernel's narrow form
  args.dec_narrow = args.kvq && d->max_query_len > 0 && (int64_t)d->max_query_len * args.G <= 8;
  args.self_plan = self_plan;  // (the cache-write kernel checks the batch itself)
  if (self_plan) {
    if (stages & PA_STAGE_PLAN) {
      ++g_launches;
      if (cudaError_t e = pa::launch_decode_prep(args, stream)) return cuda_fail(e, "decode_prep_kernel launch");
    }
    stages &= self_write_rows ? PA_STAGE_DECODE : PA_STAGE_CACHE_WRITE | PA_STAGE_DECODE;
  }
  if (stages & PA_STAGE_PLAN) {
    ++g_launches;
    if (cudaError_t e = pa::launch_plan(args, stream)) return cuda_fail(e, "plan_kernel launch");
  }
  const bool can_decode = d->route == PA_ROUTE_AUTO;
  const bool can_prefill = prefill_possible(d, args.G);
  if ((stages & PA_STAGE_CACHE_WRITE) && args.N > 0) {
    ++g_launches;
    // the bit copy right after this call's planner copies the rows beside it
    args.cw_early = (stages & PA_STAGE_PLAN) && !args.prep && !args.kvq && args.B <= pa::kEarlyWriteMaxB;
    if (cudaError_t e = pa::launch_cache_write(args, info.sms, stream)) return cuda_fail(e, "cache_write_kernel launch");
    args.cw_early = 0;
    if (can_prefill && args.mirror_keys > 0 && slots > 0 && (args.slot_mapping != nullptr || args.prep || args.kvq)) {
      // (with derived slots the bit-copy cache write makes the copy itself)
      // bf16: the fp16 copy of the prefill sequences' V, read from the cache just written
      // (the planner decides whether it is made and used)
      const int64_t warps = (int64_t)args.mirror_keys;
      const int64_t vb = std::min<int64_t>((warps + 7) / 8, (int64_t)info.sms * 8);
      ++g_launches;
      if (cudaError_t e = pa::launch_v_mirror(args, (int)vb, stream)) return cuda_fail(e, "v_mirror_kernel launch");
    }
  }
  // attention reads the prepared (or scaled) query rows when the cache-write stage wrote them
  pa::Args aq = args;
  if (args.prep || args.kvq) {
    aq.query = args.qprep;
    aq.q_stride = args.nh * hs;
    query = args.qprep;
  }
  bool prefill_launched = false;
  if ((stages & PA_STAGE_PREFILL) && can_prefill && args.N > 0 && slots > 0) {
    const int seg = gcd(d->block_size, pa::kPreTileK);
    CUtensorMap tq, tk, tv, tvm;
    // (integer caches: the scaled query rows are fp16, the caches code bytes)
    const int row_bytes = args.kvq == PA_KV_INT8 ? hs : hs / 2;
    const bool ok = args.kvq ? query_map(&tq, query, PA_FLOAT16, aq.q_stride, args.N) &&
                                   code_tile_map(&tk, kc, row_bytes, args.kvh, slots, seg) &&
                                   code_tile_map(&tv, vc, row_bytes, args.kvh, slots, seg)
                             : query_map(&tq, query, dt, aq.q_stride, args.N) &&
                                   cache_map(&tk, kc, dt, hs, args.kvh, slots, seg) &&
                                   cache_map(&tv, vc, dt, hs, args.kvh, slots, seg);
    if (!ok) {
      g_last_error = "cuTensorMapEncodeTiled failed (prefill maps)";
      return PA_ERR_CUDA;
    }
    if (args.mirror_keys > 0) {
      if (!cache_map(&tvm, args.mirror, PA_FLOAT16, hs, args.kvh, args.mirror_keys, seg)) {
        g_last_error = "cuTensorMapEncodeTiled failed (V copy map)";
        return PA_ERR_CUDA;
      }
    } else {
      tvm = tv;  // never read
    }
    // two heads of one KV group share a unit (one head for 256-wide heads: TMEM holds one O)
    const int heads_per_unit = (args.G % 2 == 0 && hs != 256) ? 2 : 1;
    const int grid = (int)std::min<int64_t>((int64_t)args.max_tiles * (args.nh / heads_per_unit), info.sms);
    if (grid > 0) {
      ++g_launches;
      if (cudaError_t e = pa::launch_prefill(aq, bf16, tq, tk, tv, tvm, seg, grid, stream))
        return cuda_fail(e, "prefill_kernel launch");
      prefill_launched = true;
    }
  }
  if ((stages & PA_STAGE_DECODE) && can_decode && args.N > 0 && slots > 0) {
    const int seg = gcd(d->block_size, pa::kDecTile);
    CUtensorMap tk, tv;
    const int row_bytes = args.kvq == PA_KV_INT8 ? hs : hs / 2;
    const bool ok = args.kvq ? code_cache_map(&tk, kc, row_bytes, args.kvh, slots, seg) &&
                                   code_cache_map(&tv, vc, row_bytes, args.kvh, slots, seg)
                             : cache_map(&tk, kc, dt, hs, args.kvh, slots, seg) &&
                                   cache_map(&tv, vc, dt, hs, args.kvh, slots, seg);
    if (!ok) {
      g_last_error = "cuTensorMapEncodeTiled failed (decode maps)";
      return PA_ERR_CUDA;
    }
    ++g_launches;
    aq.dec_after_prefill = prefill_launched;  // runs beside this call's prefill kernel
    aq.self_plan = self_plan;
    aq.self_write_rows = self_write_rows;
    if (cudaError_t e = pa::launch_decode(aq, bf16, tk, tv, seg, stream)) return cuda_fail(e, "decode_kernel launch");
  }
  return PA_OK;
}

}  // namespace

extern "C" {

size_t pa_workspace_size(const pa_dims* dims, int32_t num_heads, int32_t kv_num_heads) {
  if (check_dims(dims, num_heads, kv_num_heads) != PA_OK) return 0;
  return pa::ws_layout(dims->num_tokens, dims->batch_size, kv_num_heads, dims->head_size,
                       dims->max_blocks_per_sequence, dims->block_size, dims->decode_split_keys,
                       mirror_keys(dims, num_heads, kv_num_heads), qprep_values(dims, num_heads),
                       qexp_values(dims, num_heads))
      .total;
}

}  // extern "C"

namespace {

pa_status run(const void* query, const void* key, const void* value, void* key_cache, void* value_cache,
              const int32_t* cumulative_sequence_length, const int32_t* past_seqlens, const int32_t* block_table,
              const int32_t* slot_mapping, int32_t num_heads, int32_t kv_num_heads, float scale, void* output,
              float* lse, const pa_qk_prep* prep, const void* gate, const float* k_scale, const float* v_scale,
              const pa_dims* dims, void* workspace, size_t workspace_bytes, void* stream, uint32_t stages) {
  pa_status st = check_dims(dims, num_heads, kv_num_heads);
  if (st != PA_OK) return st;
  if (dims->kv_dtype != PA_KV_SAME) {
    if (!k_scale || !v_scale || !aligned(k_scale, 16) || !aligned(v_scale, 16)) return PA_ERR_INVALID_ARGUMENT;
  } else if (k_scale || v_scale) {
    return PA_ERR_INVALID_ARGUMENT;
  }
  if (prep) {
    if (!dims->qk_prep || prep->reserved != 0) return PA_ERR_INVALID_ARGUMENT;
    const int32_t d = prep->rotary_dim, step = dims->head_size / 16;
    if (d < 0 || d > dims->head_size || d % step != 0 || d % 2 != 0) return PA_ERR_UNSUPPORTED;
    if (d > 0 && !(prep->rope_theta > 0.f)) return PA_ERR_INVALID_ARGUMENT;
    if ((prep->q_norm_weight || prep->k_norm_weight) && !(prep->norm_eps > 0.f)) return PA_ERR_INVALID_ARGUMENT;
    if ((prep->q_norm_weight && !aligned(prep->q_norm_weight, 16)) ||
        (prep->k_norm_weight && !aligned(prep->k_norm_weight, 16)))
      return PA_ERR_INVALID_ARGUMENT;
  }
  if ((key == nullptr) != (value == nullptr)) return PA_ERR_INVALID_ARGUMENT;
  if (stages & ~PA_STAGE_ALL) return PA_ERR_INVALID_ARGUMENT;
  const int32_t N = dims->num_tokens, B = dims->batch_size, hs = dims->head_size;
  if (N == 0) return PA_OK;  // no rows: nothing is written or read
  if (!query || !key_cache || !value_cache || !cumulative_sequence_length || !past_seqlens || !block_table ||
      !output || !workspace)
    return PA_ERR_INVALID_ARGUMENT;
  if (!aligned(query, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) || !aligned(output, 16) ||
      (key && (!aligned(key, 16) || !aligned(value, 16))) || (lse && !aligned(lse, 4)) ||
      (gate && !aligned(gate, 16)) ||
      !aligned(cumulative_sequence_length, 4) ||
      !aligned(past_seqlens, 4) || !aligned(block_table, 4) || (slot_mapping && !aligned(slot_mapping, 4)) ||
      !aligned(workspace, 256))
    return PA_ERR_INVALID_ARGUMENT;
  if (dims->max_blocks_per_sequence == 0 || dims->num_blocks == 0) return PA_ERR_INVALID_ARGUMENT;
  const int64_t mkeys = mirror_keys(dims, num_heads, kv_num_heads);
  const pa::WsLayout L = pa::ws_layout(N, B, kv_num_heads, hs, dims->max_blocks_per_sequence, dims->block_size,
                                       dims->decode_split_keys, mkeys, qprep_values(dims, num_heads),
                                       qexp_values(dims, num_heads));
  if (workspace_bytes < L.total) return PA_ERR_WORKSPACE_TOO_SMALL;

  pa::Args a{};
  a.query = query;
  a.key = key;
  a.value = value;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.cum = cumulative_sequence_length;
  a.past = past_seqlens;
  a.block_table = block_table;
  a.slot_mapping = slot_mapping;
  a.output = output;
  a.lse = lse;
  a.gate = static_cast<const uint16_t*>(gate);
  a.N = N;
  a.B = B;
  a.nh = num_heads;
  a.kvh = kv_num_heads;
  a.G = num_heads / kv_num_heads;
  a.hs = hs;
  a.num_blocks = dims->num_blocks;
  a.bs = dims->block_size;
  a.max_blocks = dims->max_blocks_per_sequence;
  a.packed = key == nullptr;
  a.kv_row = kv_num_heads * hs;
  a.q_stride = a.packed ? (num_heads + 2 * kv_num_heads) * hs : num_heads * hs;
  a.k_offset = a.packed ? num_heads * hs : 0;
  a.v_offset = a.packed ? (num_heads + kv_num_heads) * hs : 0;
  a.forced_split = dims->decode_split_keys;
  a.decode_sms = dims->decode_sms;
  a.route = dims->route;
  a.max_query_len = dims->max_query_len;
  a.out_v8 = aligned(output, 32);
  a.bf16 = dims->dtype == PA_BFLOAT16;
  const float sc = scale == 0.0f ? 1.0f / sqrtf((float)hs) : scale;
  a.scale_log2 = sc * 1.4426950408889634f;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.hdr = reinterpret_cast<pa::WsHeader*>(ws + L.header);
  a.items = reinterpret_cast<pa::DecodeItem*>(ws + L.items);
  a.tiles = reinterpret_cast<pa::PrefillTile*>(ws + L.tiles);
  a.tiles_unsorted = reinterpret_cast<pa::PrefillTile*>(ws + L.tiles_unsorted);
  a.cta_begin = reinterpret_cast<int32_t*>(ws + L.cta_begin);
  a.unit_done = reinterpret_cast<int32_t*>(ws + L.unit_done);
  a.part_o = reinterpret_cast<float*>(ws + L.part_o);
  a.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  a.mirror_base = reinterpret_cast<int32_t*>(ws + L.mirror_base);
  a.mirror = reinterpret_cast<uint16_t*>(ws + L.mirror);
  a.mirror_seq = reinterpret_cast<int2*>(ws + L.mirror_seq);
  a.mirror_keys = (int32_t)mkeys;
  if (prep) {
    a.prep = 1;
    a.rotary_dim = prep->rotary_dim;
    a.norm_eps = prep->norm_eps;
    a.q_norm_w = static_cast<const uint16_t*>(prep->q_norm_weight);
    a.k_norm_w = static_cast<const uint16_t*>(prep->k_norm_weight);
    a.qprep = reinterpret_cast<uint16_t*>(ws + L.qprep);
    // the fp32 rotary table fl32(theta^(-2u/d)), formed in double and rounded once
    for (int u = 0; u < prep->rotary_dim / 2; ++u)
      a.inv_freq[u] = (float)pow((double)prep->rope_theta, -2.0 * u / prep->rotary_dim);
  }
  if (dims->kv_dtype != PA_KV_SAME) {
    a.kvq = dims->kv_dtype;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.qprep = reinterpret_cast<uint16_t*>(ws + L.qprep);
    a.qexp = reinterpret_cast<int32_t*>(ws + L.qexp);
  }
  a.max_items = L.max_items;
  a.max_tiles = L.max_tiles;
  a.cov = g_cov.load();
  a.cov_keys = g_cov_keys.load();

  return launch_all(a, dims, query, key_cache, value_cache, stages, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

pa_status pa_paged_attention_stages(const void* query, const void* key, const void* value, void* key_cache,
                                    void* value_cache, const int32_t* cumulative_sequence_length,
                                    const int32_t* past_seqlens, const int32_t* block_table,
                                    const int32_t* slot_mapping, int32_t num_heads, int32_t kv_num_heads, float scale,
                                    void* output, const pa_dims* dims, void* workspace, size_t workspace_bytes,
                                    void* stream, uint32_t stages) {
  return run(query, key, value, key_cache, value_cache, cumulative_sequence_length, past_seqlens, block_table,
             slot_mapping, num_heads, kv_num_heads, scale, output, nullptr, nullptr, nullptr, nullptr, nullptr, dims,
             workspace, workspace_bytes, stream, stages);
}

pa_status pa_paged_attention(const void* query, const void* key, const void* value, void* key_cache,
                             void* value_cache, const int32_t* cumulative_sequence_length,
                             const int32_t* past_seqlens, const int32_t* block_table, const int32_t* slot_mapping,
                             int32_t num_heads, int32_t kv_num_heads, float scale, void* output,
                             const pa_dims* dims, void* workspace, size_t workspace_bytes, void* stream) {
  return run(query, key, value, key_cache, value_cache, cumulative_sequence_length, past_seqlens, block_table,
             slot_mapping, num_heads, kv_num_heads, scale, output, nullptr, nullptr, nullptr, nullptr, nullptr, dims,
             workspace, workspace_bytes, stream, PA_STAGE_ALL);
}

pa_status pa_paged_attention_lse(const void* query, const void* key, const void* value, void* key_cache,
                                 void* value_cache, const int32_t* cumulative_sequence_length,
                                 const int32_t* past_seqlens, const int32_t* block_table,
                                 const int32_t* slot_mapping, int32_t num_heads, int32_t kv_num_heads, float scale,
                                 void* output, float* lse, const pa_dims* dims, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  return run(query, key, value, key_cache, value_cache, cumulative_sequence_length, past_seqlens, block_table,
             slot_mapping, num_heads, kv_num_heads, scale, output, lse, nullptr, nullptr, nullptr, nullptr, dims,
             workspace, workspace_bytes, stream, PA_STAGE_ALL);
}

pa_status pa_paged_attention_ex(const void* query, const void* key, const void* value, void* key_cache,
                                void* value_cache, const int32_t* cumulative_sequence_length,
                                const int32_t* past_seqlens, const int32_t* block_table, const int32_t* slot_mapping,
                                int32_t num_heads, int32_t kv_num_heads, float scale, void* output,
                                const pa_extensions* ext, const pa_dims* dims, void* workspace,
                                size_t workspace_bytes, void* stream) {
  return run(query, key, value, key_cache, value_cache, cumulative_sequence_length, past_seqlens, block_table,
             slot_mapping, num_heads, kv_num_heads, scale, output, ext ? ext->lse : nullptr,
             ext ? ext->qk_prep : nullptr, ext ? ext->output_gate : nullptr, ext ? ext->k_scale : nullptr,
             ext ? ext->v_scale : nullptr, dims, workspace, workspace_bytes, stream,
             ext && ext->stages ? ext->stages : PA_STAGE_ALL);
}

const char* pa_last_error(void) { return g_last_error; }

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PA_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

pa_status pa_read_device_error(void* workspace, void* stream, uint32_t* error_bits) {
  if (!workspace || !error_bits) return PA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaError_t e = cudaStreamSynchronize(s)) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t v = 0;
  if (cudaError_t e = cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost)) return cuda_fail(e, "cudaMemcpy");
  if (cudaError_t e = cudaMemset(workspace, 0, sizeof(v))) return cuda_fail(e, "cudaMemset");
  *error_bits = v;
  return PA_OK;
}

uint64_t pa_kernel_launch_count(void) { return g_launches.load(); }

pa_status pa_debug_coverage(int32_t* counts, int32_t max_keys) {
#ifdef PA_COVERAGE
  if (counts && max_keys <= 0) return PA_ERR_INVALID_ARGUMENT;
  g_cov_keys = counts ? max_keys : 0;
  g_cov = counts;
  return PA_OK;
#else
  (void)counts;
  (void)max_keys;
  return PA_ERR_UNSUPPORTED;
#endif
}

int32_t pa_abi_version(void) { return PA_ABI_VERSION; }

}  // extern "C"
