// pa_paged_attention_static_workspace: the operator for callers that cannot hand the
// library a device workspace because they cannot allocate device memory themselves -
// for example a plugin whose device memory is owned and budgeted by a host framework
// that exposes no allocator, or a latency-critical path that must not call cudaMalloc
// (which may synchronise the device). Instead of a caller buffer, the call uses a
// workspace built into the library: one file-scope device array of
// PA_STATIC_WORKSPACE_BYTES per GPU, created when the library's code is loaded on that
// GPU and kept until the process exits.
//
// The array's host-side name is only a stand-in for the symbol, never a device address,
// so the device address is looked up with cudaGetSymbolAddress once per device (with that
// device current) and cached; the first call on each device does this lookup. Every call
// on a device shares the same array and leaves its contents behind. Each call's first
// kernel - the planner, or, for a decode-only call whose decode kernel plans itself, the
// one-CTA reset before it - rewrites the header, the error word and the merge counters,
// and every other field a later kernel reads is written earlier in the same call, so
// nothing has to be cleared between calls. Calls whose GPU work overlaps (different
// streams, or different host threads without ordering) race on the array and must be
// serialised by the caller.
//
// pa_static_workspace_read_device_error gives these callers the device error word that
// pa_read_device_error gives callers with their own workspace.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// device address of g_static_workspace on the current device, looked up once per device
pa_status static_workspace_address(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_paged_attention_static_workspace(
    const void* query, const void* key, const void* value, void* key_cache, void* value_cache,
    const int32_t* cumulative_sequence_length, const int32_t* past_seqlens, const int32_t* block_table,
    const int32_t* slot_mapping, int32_t num_heads, int32_t kv_num_heads, float scale, void* output,
    const pa_dims* dims, void* stream) {
  if (!dims) return PA_ERR_INVALID_ARGUMENT;
  if (dims->num_tokens == 0)  // nothing to do; let the regular entry point validate and return
    return pa_paged_attention(query, key, value, key_cache, value_cache, cumulative_sequence_length, past_seqlens,
                              block_table, slot_mapping, num_heads, kv_num_heads, scale, output, dims, nullptr, 0,
                              stream);
  const size_t need = pa_workspace_size(dims, num_heads, kv_num_heads);
  if (need > (size_t)PA_STATIC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  if (pa_status st = static_workspace_address(&ws)) return st;
  // sizes the regular entry point rejects (need == 0) come back with its typed error
  return pa_paged_attention(query, key, value, key_cache, value_cache, cumulative_sequence_length, past_seqlens,
                            block_table, slot_mapping, num_heads, kv_num_heads, scale, output, dims, ws,
                            (size_t)PA_STATIC_WORKSPACE_BYTES, stream);
}

extern "C" pa_status pa_static_workspace_read_device_error(void* stream, uint32_t* error_bits) {
  if (!error_bits) return PA_ERR_INVALID_ARGUMENT;
  void* ws = nullptr;
  if (pa_status st = static_workspace_address(&ws)) return st;
  return pa_read_device_error(ws, stream, error_bits);  // (the word is the array's first field)
}
