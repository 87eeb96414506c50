/*
 * pagedattn.h - C ABI of the GB300 (sm_103a) PagedAttention library (libpagedattn.so).
 *
 * The operation is com.microsoft.PagedAttention as stated in the
 * "com.microsoft.PagedAttention" README ("Description", "Inputs", "Outputs",
 * "Attributes"): the K/V rows of this step's tokens are written into a block-based
 * (paged) cache, then each sequence's query rows attend causally, with grouped-query
 * heads, to that sequence's history read back through block_table.
 *
 * Conventions for every entry point:
 *   - Tensor arguments are DEVICE pointers to dense row-major arrays owned by the
 *     caller. The library allocates no memory. Floating tensors share one element type
 *     T (pa_dtype); index tensors are int32. Every T pointer must be 16-byte aligned,
 *     every int32 pointer 4-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is enqueued
 *     asynchronously; apart from pa_read_device_error and
 *     pa_static_workspace_read_device_error no call synchronises, reads device memory
 *     back, or allocates, so a call can be captured in a CUDA graph.
 *   - Argument errors are found on the host before anything is launched and reported as
 *     PA_ERR_* codes. Inconsistencies that only device data can reveal (a
 *     cumulative_sequence_length that is not a prefix sum, an out-of-range block or
 *     slot) never fault: the affected work is skipped and a bit is set in the workspace's
 *     device error word, which pa_read_device_error returns.
 *   - Calls that share a workspace must be ordered (same stream, or synchronised).
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ABI_VERSION 7

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARGUMENT = 1,   /* null/misaligned pointer, inconsistent sizes, key xor value */
  PA_ERR_UNSUPPORTED = 2,        /* a valid request this build does not implement (head_size, block_size, dtype) */
  PA_ERR_WORKSPACE_TOO_SMALL = 3,
  PA_ERR_CUDA = 4                /* a CUDA runtime call or launch failed */
} pa_status;

typedef enum pa_dtype {
  PA_FLOAT16 = 0,
  PA_BFLOAT16 = 1
} pa_dtype;

/*
 * Element type of the two caches (pa_dims.kv_dtype). PA_KV_SAME: T, as in the operator
 * statement. The integer formats are an extension (the Mobius issue's scope list asks for an
 * INT8/INT4 per-channel paged KV cache with calibrated scale loading; no page gives a
 * format): the caches hold integer codes, and K and V each come with a caller-given fp32
 * scale per (KV head, channel), pa_extensions.k_scale / v_scale, fixed by calibration;
 * symmetric, no zero point. This call's K and V rows (of T) are stored as
 *   code = min(max(rint(fl32(x) / s), -Q), Q)   (IEEE fp32 quotient, rint half to even)
 * with Q = 127 (PA_KV_INT8: one two's complement byte per value) or 7 (PA_KV_INT4: two
 * values per byte, channel 2i in the low nibble, 2i + 1 in the high nibble, two's
 * complement), and attention reads the value code * s. A cache is then
 * (num_blocks, block_size, kv_num_heads, head_size) bytes for INT8 and
 * (num_blocks, block_size, kv_num_heads, head_size / 2) bytes for INT4.
 */
typedef enum pa_kv_dtype {
  PA_KV_SAME = 0,
  PA_KV_INT8 = 1,
  PA_KV_INT4 = 2
} pa_kv_dtype;

/* Bits of the device error word (pa_read_device_error). */
#define PA_DEVERR_BAD_BATCH 1u  /* cumulative_sequence_length / past_seqlens inconsistent: nothing was computed or written */
#define PA_DEVERR_BAD_BLOCK 2u  /* a block_table entry of an active page is outside [0, num_blocks): that page read as zeros */
#define PA_DEVERR_BAD_SLOT 4u   /* a slot (given or derived) is outside [0, num_blocks*block_size) and not -1: write skipped */
#define PA_DEVERR_TIMEOUT 8u    /* a pipeline wait inside a kernel gave up (results of that work item are undefined) */

/* Routing of sequences to kernels (pa_dims.route). */
#define PA_ROUTE_AUTO 0          /* q_len * (num_heads / kv_num_heads) <= 16: split-KV decode kernel; else prefill kernel */
#define PA_ROUTE_ALL_PREFILL 1   /* every sequence on the tcgen05 prefill kernel */

/* Host-side sizes of one invocation. */
typedef struct pa_dims {
  int32_t num_tokens;              /* N: rows of query, key, value, output and slot_mapping */
  int32_t batch_size;              /* B: sequences; cumulative_sequence_length has B + 1 entries */
  int32_t head_size;               /* 64, 128 or 256 */
  int32_t num_blocks;              /* pages in each cache */
  int32_t block_size;              /* tokens per page: a positive multiple of 16 */
  int32_t max_blocks_per_sequence; /* columns of block_table */
  int32_t dtype;                   /* pa_dtype of T */
  int32_t decode_split_keys;       /* 0: balanced automatic partition; else keys per split-KV decode work
                                      item (a multiple of 64; a test hook) */
  int32_t route;                   /* PA_ROUTE_* */
  int32_t max_query_len;           /* 0: unknown; else a host-side bound on every sequence's new-token count
                                      (the CPU-resident launch bound of the packed contract's
                                      attention_metadata). With route AUTO and max_query_len *
                                      (num_heads / kv_num_heads) <= 16 no prefill kernel is launched; if in
                                      addition slot_mapping is NULL and batch_size <= 256 (64 at
                                      head_size 256), no planner runs: a reset of the workspace's counters, then the decode
                                      kernel, which plans its own share of the work (with caches of T and
                                      no Q/K preparation it also writes this call's K/V rows itself, two
                                      kernels in all; else the cache-write kernel runs between the two and
                                      checks the batch itself). The device checks the bound: a sequence
                                      above it is a PA_DEVERR_BAD_BATCH and nothing is written. */
  int32_t qk_prep;                 /* non-zero: calls pass a pa_qk_prep, and the workspace also holds the
                                      prepared query rows (num_tokens * num_heads * head_size values of T) */
  int32_t kv_dtype;                /* pa_kv_dtype of the caches: INT8 with head_size 64, 128 or 256,
                                      INT4 with 128 or 256 (else PA_ERR_UNSUPPORTED); integer caches
                                      need pa_paged_attention_ex with both scales */
  int32_t decode_sms;              /* 0 (normal): when a whole call has both prefill-class and
                                      decode-class rows, the planner splits the SMs so that the
                                      prefill kernel (tensor-bound) and the decode kernel (HBM-bound)
                                      run at the same time, choosing the decode share from a model of
                                      their rates. > 0 fixes that share at this many SMs (at most all
                                      but one): a tuning and test hook. Results do not depend on it. */
} pa_dims;

/*
 * Q/K preparation before the cache write (pa_extensions.qk_prep): not part of the
 * operator statement, but the step the Qwen3.8 export issue ("Add Qwen3.8 packed hybrid
 * PagedAttention export for ORT GenAI Engine") runs right before PagedAttention and the
 * README ("Description") lists as not done by its package. For row j of sequence b, at
 * position p = past_seqlens[b] + j, every query head vector and every key head vector x
 * (head_size values) becomes
 *   RMSNorm (when its weight is given):  x_c <- x_c / sqrt(mean_c x_c^2 + norm_eps) * w_c
 *   then the rotary embedding (when rotary_dim = d > 0), pairing component u with u + d/2:
 *     a_u = fl32(fl32(p) * fl32(rope_theta^(-2u/d)))   (an fp32 rotary table)
 *     (x_u, x_{u+d/2}) <- (x_u cos a_u - x_{u+d/2} sin a_u,  x_{u+d/2} cos a_u + x_u sin a_u)
 *   components from d on unchanged; the result is rounded once to T.
 * The prepared K is what the cache receives; attention reads the prepared Q; V is
 * unchanged. Computed in fp32 (sincosf of the fp32 angle).
 */
typedef struct pa_qk_prep {
  const void* q_norm_weight;  /* T (head_size) device array, or NULL: no RMSNorm of the query heads */
  const void* k_norm_weight;  /* T (head_size) device array, or NULL: no RMSNorm of the key heads */
  float norm_eps;             /* RMSNorm epsilon (> 0 when a weight is given) */
  float rope_theta;           /* base of the rotary frequencies (> 0 when rotary_dim > 0) */
  int32_t rotary_dim;         /* 0, or an even multiple of head_size / 16 up to head_size (8 .. 128 in steps
                                 of 8 for head_size 128) */
  int32_t reserved;           /* 0 */
} pa_qk_prep;

/*
 * Bytes of device workspace pa_paged_attention needs for these sizes (0 on invalid
 * sizes). Pure host arithmetic; needs no GPU. The workspace holds the device-built work
 * plan, the split-KV partial results (fp32 output rows and their log-sum-exp), the
 * device error word and, for bf16 when prefill is possible, an fp16 copy of the V rows of
 * the prefill-class sequences with room for 4 * num_tokens keys (at most the cache's size).
 * The prefill kernel reads V from that copy (one fp16 P V product per 16 keys) when the
 * call's prefill-class sequences fit it and every copied value is representable in fp16;
 * otherwise it reads the bf16 cache and splits P into two bf16 terms. It must be 256-byte
 * aligned.
 */
size_t pa_workspace_size(const pa_dims* dims, int32_t num_heads, int32_t kv_num_heads);

/*
 * com.microsoft.PagedAttention ("com.microsoft.PagedAttention" README).
 *
 *   query        T (N, num_heads*head_size), or (N, (num_heads + 2*kv_num_heads)*head_size)
 *                holding packed [Q | K | V] rows when key and value are NULL ("Inputs", `query`).
 *                Within each part the heads are consecutive blocks of head_size.
 *   key, value   T (N, kv_num_heads*head_size), or both NULL ("Inputs", `key`, `value`).
 *   key_cache,   T (num_blocks, block_size, kv_num_heads, head_size), updated in place: row
 *   value_cache  i of key/value is copied to flat slot s = block_id*block_size + offset
 *                ("Inputs", `key_cache`, `value_cache`; "Outputs": both caches are updated).
 *   cumulative_sequence_length  int32 (B+1): exclusive prefix sums; sequence b owns rows
 *                [cum[b], cum[b+1]).
 *   past_seqlens int32 (B): cached history length of each sequence before this call.
 *   block_table  int32 (B, max_blocks_per_sequence): logical block -> physical block; it
 *                defines the read path. Entries past ceil((past+q_len)/block_size) are
 *                never read. Rows may share physical pages (a read-only shared prefix),
 *                provided no row of this call writes into a shared page.
 *   slot_mapping int32 (N) or NULL: the slot of each row, -1 = do not write. When NULL the
 *                slot is derived: p = past_seqlens[b] + j for row j of sequence b,
 *                s = block_table[b][p / block_size]*block_size + p % block_size.
 *   num_heads, kv_num_heads  attributes; num_heads % kv_num_heads == 0; query head h
 *                reads KV head h / (num_heads / kv_num_heads).
 *   scale        attribute; 0 selects 1/sqrt(head_size) ("Attributes", `scale`).
 *   output       T (N, num_heads*head_size), must not overlap any input.
 *
 * Row j of sequence b attends the keys at logical positions 0 .. past_seqlens[b] + j
 * (bottom-right causal), all read from the caches after this call's writes. Softmax
 * and accumulation are fp32; the output is rounded once to T.
 *
 * Returns PA_OK once the work is enqueued on `stream`.
 */
pa_status pa_paged_attention(const void* query, const void* key, const void* value,
                             void* key_cache, void* value_cache,
                             const int32_t* cumulative_sequence_length,
                             const int32_t* past_seqlens, const int32_t* block_table,
                             const int32_t* slot_mapping, int32_t num_heads, int32_t kv_num_heads,
                             float scale, void* output, const pa_dims* dims, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Bytes of the device workspace built into the library for
 * pa_paged_attention_static_workspace (one array per GPU that loads the library). */
#define PA_STATIC_WORKSPACE_BYTES (16u << 20)

/*
 * pa_paged_attention for callers that cannot allocate device memory - for example a
 * plugin whose device memory belongs to a host framework that offers it no allocator,
 * or a latency-critical path that must not call cudaMalloc. Same arguments as
 * pa_paged_attention without the workspace: the call uses a workspace of
 * PA_STATIC_WORKSPACE_BYTES built into the library, which every GPU that loads the
 * library holds until the process exits. The pages have no counterpart to this entry
 * point: it is a deployment convenience, not part of the operator.
 *
 *   - Returns PA_ERR_WORKSPACE_TOO_SMALL, without launching anything, when
 *     pa_workspace_size(dims, num_heads, kv_num_heads) exceeds PA_STATIC_WORKSPACE_BYTES
 *     (use pa_paged_attention with your own workspace for such sizes).
 *   - Allocates nothing and calls no allocating routine. The first call on each device
 *     looks up the built-in array's device address (cudaGetSymbolAddress) and caches it;
 *     make that first call before any stream capture.
 *   - All calls on a device share the one array and it keeps the last call's contents.
 *     Each call's first kernel (the planner, or the one-CTA reset of a decode-only call
 *     whose decode kernel plans itself) rewrites the header, the device error word and
 *     the merge counters, and the call writes every other field before it reads it, so
 *     nothing needs clearing. Calls whose GPU work overlaps race on the array: order them
 *     (one stream, or synchronise between them).
 *   - Problems only device data reveals (a block or slot out of range, an inconsistent
 *     batch) set bits of the array's device error word, as with a caller workspace; read
 *     them with pa_static_workspace_read_device_error.
 */
pa_status pa_paged_attention_static_workspace(const void* query, const void* key, const void* value,
                                              void* key_cache, void* value_cache,
                                              const int32_t* cumulative_sequence_length,
                                              const int32_t* past_seqlens, const int32_t* block_table,
                                              const int32_t* slot_mapping, int32_t num_heads,
                                              int32_t kv_num_heads, float scale, void* output,
                                              const pa_dims* dims, void* stream);

/*
 * pa_read_device_error for the built-in workspace of pa_paged_attention_static_workspace:
 * waits for `stream`, copies the device error word (PA_DEVERR_* bits of the most recent
 * call on the current device) into *error_bits, then clears it. Synchronises; allocates
 * nothing. Like that entry point it has no counterpart on the pages.
 */
pa_status pa_static_workspace_read_device_error(void* stream, uint32_t* error_bits);

/* Stages of pa_paged_attention, in the order they must run. */
#define PA_STAGE_PLAN 1u        /* device work partitioner: classify sequences, build work lists */
#define PA_STAGE_CACHE_WRITE 2u /* scatter this step's K/V rows into the caches; for bf16, then
                                   the fp16 copy of the prefill sequences' V the prefill reads */
#define PA_STAGE_PREFILL 4u     /* tcgen05/TMEM attention for prefill-class sequences */
#define PA_STAGE_DECODE 8u      /* split-KV attention for decode-class sequences, including the
                                   deterministic (out, lse) merge of the splits */
#define PA_STAGE_ALL 15u

/*
 * Same arguments as pa_paged_attention; runs only the stages in `stages` (PA_STAGE_*
 * bits), in the order above. The kernels are those the whole call would run (the same
 * program: the same work partition, the same SM split of a mixed batch), and `stages`
 * picks which of them this call launches. For a decode-only call that the decode kernel
 * plans itself (see pa_dims.max_query_len) PA_STAGE_PLAN is the reset of the workspace's
 * counters and PA_STAGE_PREFILL is empty; PA_STAGE_CACHE_WRITE is empty too when the
 * decode kernel writes this call's rows. The two attention kernels of a mixed batch run
 * side by side only when one call launches both. A stage reads what earlier stages left
 * in the workspace, so a caller that splits a call across several calls must pass the
 * same arguments and workspace to each and keep them in stage order. Used to time one
 * kernel of a step with events around it. Otherwise identical to pa_paged_attention.
 */
pa_status pa_paged_attention_stages(const void* query, const void* key, const void* value,
                                    void* key_cache, void* value_cache,
                                    const int32_t* cumulative_sequence_length,
                                    const int32_t* past_seqlens, const int32_t* block_table,
                                    const int32_t* slot_mapping, int32_t num_heads,
                                    int32_t kv_num_heads, float scale, void* output,
                                    const pa_dims* dims, void* workspace, size_t workspace_bytes,
                                    void* stream, uint32_t stages);

/*
 * pa_paged_attention that also exports the log-sum-exp of every output row: lse is
 * float32 (N, num_heads), row i head h = ln sum_t exp(scale * <q_ih, k_t>) over the keys
 * the row attends, the natural-log, scale-included "attention-domain lse" that the
 * (out, lse) merge of context-parallel partials consumes (WS2 CP-Aware Attention
 * Contract, "Reduction Semantics"). lse must be 4-byte aligned and must not overlap any
 * other argument; NULL behaves as pa_paged_attention. Computed in fp32 from the same
 * running max and sum that normalise the output.
 */
pa_status pa_paged_attention_lse(const void* query, const void* key, const void* value,
                                 void* key_cache, void* value_cache,
                                 const int32_t* cumulative_sequence_length,
                                 const int32_t* past_seqlens, const int32_t* block_table,
                                 const int32_t* slot_mapping, int32_t num_heads,
                                 int32_t kv_num_heads, float scale, void* output, float* lse,
                                 const pa_dims* dims, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* Optional extensions of one call (pa_paged_attention_ex); every member may be NULL. */
typedef struct pa_extensions {
  float* lse;                 /* fp32 (N, num_heads): each output row's log-sum-exp, as pa_paged_attention_lse */
  const pa_qk_prep* qk_prep;  /* the Q/K preparation above; dims->qk_prep must then be non-zero and the
                                 workspace sized with it, else PA_ERR_INVALID_ARGUMENT; an unsupported
                                 rotary_dim is PA_ERR_UNSUPPORTED; norm weights 16-byte aligned */
  const void* output_gate;    /* T (N, num_heads*head_size), 16-byte aligned: every output element is
                                 multiplied by sigmoid of the matching gate element before the final
                                 rounding (the sigmoid-gated output of Qwen3.5's full-attention layers,
                                 "Add Qwen3.8 packed hybrid PagedAttention export for ORT GenAI Engine");
                                 lse is not gated */
  const float* k_scale;       /* fp32 (kv_num_heads, head_size), 16-byte aligned: the K scales of integer
                                 caches (dims->kv_dtype != PA_KV_SAME), finite and positive; NULL otherwise */
  const float* v_scale;       /* the same for V */
  uint32_t stages;            /* 0: the whole call; else PA_STAGE_* bits, as pa_paged_attention_stages */
} pa_extensions;

/* pa_paged_attention with the extensions in `ext` (NULL: none). */
pa_status pa_paged_attention_ex(const void* query, const void* key, const void* value,
                                void* key_cache, void* value_cache,
                                const int32_t* cumulative_sequence_length,
                                const int32_t* past_seqlens, const int32_t* block_table,
                                const int32_t* slot_mapping, int32_t num_heads,
                                int32_t kv_num_heads, float scale, void* output,
                                const pa_extensions* ext, const pa_dims* dims, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Static description of a status code. Never NULL. */
const char* pa_status_string(pa_status status);

/* Message of the last PA_ERR_CUDA returned to the calling host thread (the failing call and
 * the CUDA error string), "no error" before any. Valid until the thread's next failing call. */
const char* pa_last_error(void);

/*
 * Debug/test helper: waits for `stream`, copies the workspace's device error word
 * (PA_DEVERR_* bits, accumulated since the workspace was last cleared) into
 * *error_bits, then clears it. This is the only entry point that synchronises.
 */
pa_status pa_read_device_error(void* workspace, void* stream, uint32_t* error_bits);

/*
 * Test hook of the coverage build (libpagedattn_cov.so, compiled with PA_COVERAGE; the
 * product library returns PA_ERR_UNSUPPORTED). From the next call on, every (query row i,
 * head h, key t) that an attention kernel lets into its softmax adds one to the device int32
 * counts[(i * num_heads + h) * max_keys + t]; keys t >= max_keys add to the overflow counter
 * counts[num_tokens * num_heads * max_keys]. The caller zeroes the array. A correct work
 * partition counts every key 0 .. past_seqlens[b] + j of row j of sequence b exactly once
 * and nothing else. NULL switches counting off. No page describes a partitioner; this is
 * how the partition is checked (every (row, head, key) covered once).
 */
pa_status pa_debug_coverage(int32_t* counts, int32_t max_keys);

/* Number of kernels this library has launched in this process (monotonic). */
uint64_t pa_kernel_launch_count(void);

/* PA_ABI_VERSION of the loaded library. */
int32_t pa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
