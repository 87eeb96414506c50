"""GB300 (sm_103a) PagedAttention over packed variable-length batches.

``paged_attention`` follows the com.microsoft.PagedAttention operator statement
(com.microsoft.PagedAttention README, "Inputs", "Outputs", "Attributes"). This module
only marshals torch tensors into raw device pointers for the C ABI of
``libpagedattn.so`` (declared in ``include/pagedattn.h``); every step of the operator
runs in that library's CUDA kernels on the caller's current stream. There is no
fallback: without the compiled library every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_HERE, "libpagedattn.so")

STAGE_PLAN, STAGE_CACHE_WRITE, STAGE_PREFILL, STAGE_DECODE = 1, 2, 4, 8
STAGE_ALL = 15
ROUTE_AUTO, ROUTE_ALL_PREFILL = 0, 1
DEVERR_BAD_BATCH, DEVERR_BAD_BLOCK, DEVERR_BAD_SLOT, DEVERR_TIMEOUT = 1, 2, 4, 8

_STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID_ARGUMENT", 2: "PA_ERR_UNSUPPORTED",
           3: "PA_ERR_WORKSPACE_TOO_SMALL", 4: "PA_ERR_CUDA"}
_DTYPES = {torch.float16: 0, torch.bfloat16: 1}
KV_SAME, KV_INT8, KV_INT4 = 0, 1, 2
_KV_FORMATS = {None: KV_SAME, "int8": KV_INT8, "int4": KV_INT4}

_lib = None


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, where: str):
        detail = ""
        if status == 4 and _lib is not None:
            detail = " (" + _lib.pa_last_error().decode(errors="replace") + ")"
        super().__init__(f"{where}: {_STATUS.get(status, status)}{detail}")
        self.status = status


class PaDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_tokens", "batch_size", "head_size", "num_blocks", "block_size",
        "max_blocks_per_sequence", "dtype", "decode_split_keys", "route", "max_query_len", "qk_prep",
        "kv_dtype", "decode_sms")]


class PaQkPrep(ctypes.Structure):
    _fields_ = [("q_norm_weight", ctypes.c_void_p), ("k_norm_weight", ctypes.c_void_p),
                ("norm_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("rotary_dim", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class PaExtensions(ctypes.Structure):
    _fields_ = [("lse", ctypes.c_void_p), ("qk_prep", ctypes.POINTER(PaQkPrep)), ("output_gate", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p), ("stages", ctypes.c_uint32)]


def load_library():
    """Load libpagedattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBRARY_PATH):
        raise RuntimeError(f"{LIBRARY_PATH} is missing: build it with varlen_paged_kv_gb300.build.build()")
    lib = ctypes.CDLL(LIBRARY_PATH)
    p, i32, u32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t
    dims_p = ctypes.POINTER(PaDims)
    lib.pa_workspace_size.argtypes = [dims_p, i32, i32]
    lib.pa_workspace_size.restype = sz
    common = [p, p, p, p, p, p, p, p, p, i32, i32, f32, p, dims_p, p, sz, p]
    lib.pa_paged_attention.argtypes = common
    lib.pa_paged_attention.restype = ctypes.c_int
    lib.pa_paged_attention_stages.argtypes = common + [u32]
    lib.pa_paged_attention_stages.restype = ctypes.c_int
    lib.pa_paged_attention_lse.argtypes = common[:13] + [p] + common[13:]
    lib.pa_paged_attention_lse.restype = ctypes.c_int
    lib.pa_paged_attention_ex.argtypes = common[:13] + [ctypes.POINTER(PaExtensions)] + common[13:]
    lib.pa_paged_attention_ex.restype = ctypes.c_int
    lib.pa_status_string.argtypes = [ctypes.c_int]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_last_error.argtypes = []
    lib.pa_last_error.restype = ctypes.c_char_p
    lib.pa_read_device_error.argtypes = [p, p, ctypes.POINTER(u32)]
    lib.pa_read_device_error.restype = ctypes.c_int
    lib.pa_kernel_launch_count.argtypes = []
    lib.pa_kernel_launch_count.restype = ctypes.c_uint64
    lib.pa_abi_version.argtypes = []
    lib.pa_abi_version.restype = i32
    _lib = lib
    return lib


def make_dims(num_tokens, batch_size, head_size, num_blocks, block_size, max_blocks_per_sequence, dtype,
              decode_split_keys=0, route=ROUTE_AUTO, max_query_len=0, qk_prep=False, kv_dtype=KV_SAME,
              decode_sms=0) -> PaDims:
    code = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return PaDims(int(num_tokens), int(batch_size), int(head_size), int(num_blocks), int(block_size),
                  int(max_blocks_per_sequence), code, int(decode_split_keys), int(route), int(max_query_len),
                  int(bool(qk_prep)), int(_KV_FORMATS.get(kv_dtype, kv_dtype)), int(decode_sms))


def workspace_size(dims: PaDims, num_heads: int, kv_num_heads: int) -> int:
    return int(load_library().pa_workspace_size(ctypes.byref(dims), num_heads, kv_num_heads))


def kernel_launch_count() -> int:
    return int(load_library().pa_kernel_launch_count())


def read_device_error(workspace: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronises the stream, returns and clears the PA_DEVERR_* bits of the workspace."""
    s = (stream or torch.cuda.current_stream(workspace.device)).cuda_stream
    bits = ctypes.c_uint32(0)
    st = load_library().pa_read_device_error(ctypes.c_void_p(workspace.data_ptr()), ctypes.c_void_p(s),
                                             ctypes.byref(bits))
    if st:
        raise PagedAttentionError(st, "pa_read_device_error")
    return int(bits.value)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def paged_attention(query: torch.Tensor, key: Optional[torch.Tensor], value: Optional[torch.Tensor],
                    key_cache: torch.Tensor, value_cache: torch.Tensor,
                    cumulative_sequence_length: torch.Tensor, past_seqlens: torch.Tensor,
                    block_table: torch.Tensor, slot_mapping: Optional[torch.Tensor] = None, *,
                    num_heads: int, kv_num_heads: int, scale: float = 0.0,
                    output: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    decode_split_keys: int = 0, route: int = ROUTE_AUTO, max_query_len: int = 0,
                    stages: int = STAGE_ALL, stream: Optional[torch.cuda.Stream] = None,
                    lse: Optional[torch.Tensor] = None, qk_prep: Optional[dict] = None,
                    output_gate: Optional[torch.Tensor] = None, kv_quant: Optional[str] = None,
                    k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                    decode_sms: int = 0) -> torch.Tensor:
    """com.microsoft.PagedAttention on CUDA tensors. Writes key_cache / value_cache in
    place and returns ``output`` (num_tokens, num_heads * head_size).

    ``max_query_len`` (optional) is a host-side bound on every sequence's new-token count;
    it lets decode-only batches skip the prefill launch and is checked on the device.
    ``lse`` (optional, float32 (num_tokens, num_heads)) receives each output row's natural-log
    log-sum-exp of the scaled scores.
    ``stages`` (PA_STAGE_* bits) launches only those kernels of the call's program, as
    pa_paged_attention_stages does.
    ``qk_prep`` (optional): dict(q_norm_weight=tensor (head_size,) of the
    query dtype or None, k_norm_weight=... or None, eps=float, rotary_dim=int, theta=float):
    RMSNorm of the query and key heads, then the rotary embedding at each row's position,
    before the cache write (pa_qk_prep).
    ``output_gate`` (optional, shape and dtype of the output): the output is
    multiplied by sigmoid(output_gate) elementwise before the final rounding.
    ``kv_quant`` (optional): "int8" or "int4" integer caches (uint8 tensors
    (num_blocks, block_size, kv_num_heads, head_size), or head_size / 2 for int4) with the
    float32 (kv_num_heads, head_size) per-channel scales ``k_scale`` and ``v_scale``: this
    call's K and V rows are stored as codes, attention reads code * scale."""
    lib = load_library()
    if query.dtype not in _DTYPES:
        raise TypeError("query must be float16 or bfloat16")
    if kv_quant not in _KV_FORMATS:
        raise ValueError("kv_quant must be None, 'int8' or 'int4'")
    cache_dtype = query.dtype if kv_quant is None else torch.uint8
    for name, t in (("key", key), ("value", value)):
        if t is not None and t.dtype != query.dtype:
            raise TypeError(f"{name} must have the dtype of query")
    for name, t in (("key_cache", key_cache), ("value_cache", value_cache)):
        if t.dtype != cache_dtype:
            raise TypeError(f"{name} must be {cache_dtype}")
    head_size = key_cache.shape[3] * (2 if kv_quant == "int4" else 1)
    if kv_quant is not None:
        for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
            if t is None or t.dtype != torch.float32 or tuple(t.shape) != (kv_num_heads, head_size):
                raise ValueError(f"{name} must be float32 (kv_num_heads, head_size)")
    elif k_scale is not None or v_scale is not None:
        raise ValueError("k_scale / v_scale need integer caches (kv_quant)")
    for name, t in (("cumulative_sequence_length", cumulative_sequence_length), ("past_seqlens", past_seqlens),
                    ("block_table", block_table), ("slot_mapping", slot_mapping)):
        if t is not None and t.dtype != torch.int32:
            raise TypeError(f"{name} must be int32")
    if lse is not None:
        if lse.dtype != torch.float32 or tuple(lse.shape) != (query.shape[0], num_heads):
            raise ValueError("lse must be float32 (num_tokens, num_heads)")
    if output_gate is not None:
        if output_gate.dtype != query.dtype or output_gate.numel() != query.shape[0] * num_heads * head_size:
            raise ValueError("output_gate must have the output's shape and dtype")
    prep = None
    if qk_prep is not None:
        for k in ("q_norm_weight", "k_norm_weight"):
            t = qk_prep.get(k)
            if t is not None and (t.dtype != query.dtype or t.numel() != head_size or not t.is_cuda or
                                  not t.is_contiguous()):
                raise ValueError(f"{k} must be a contiguous CUDA tensor of head_size values of the query dtype")
        def addr(t):
            return None if t is None else t.data_ptr()
        prep = PaQkPrep(addr(qk_prep.get("q_norm_weight")), addr(qk_prep.get("k_norm_weight")),
                        float(qk_prep.get("eps", 1e-6)), float(qk_prep.get("theta", 10000.0)),
                        int(qk_prep.get("rotary_dim", 0)), 0)
    for t in (query, key, value, key_cache, value_cache, cumulative_sequence_length, past_seqlens, block_table,
              slot_mapping, output, workspace, lse, output_gate, k_scale, v_scale):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("all tensors must be contiguous CUDA tensors")
    N = query.shape[0]
    B = past_seqlens.shape[0]
    num_blocks, block_size, kvh_c = key_cache.shape[:3]
    if kvh_c != kv_num_heads or value_cache.shape != key_cache.shape:
        raise ValueError("cache shape must be (num_blocks, block_size, kv_num_heads, head_size) "
                         "(head_size / 2 bytes for int4)")
    width = (num_heads + 2 * kv_num_heads) * head_size if key is None else num_heads * head_size
    if query.shape[1] != width:
        raise ValueError(f"query rows must have {width} elements")
    if cumulative_sequence_length.shape[0] != B + 1 or block_table.shape[0] != B:
        raise ValueError("cumulative_sequence_length must have batch_size + 1 entries, block_table batch_size rows")
    dims = make_dims(N, B, head_size, num_blocks, block_size, block_table.shape[1], query.dtype,
                     decode_split_keys, route, max_query_len, qk_prep is not None, _KV_FORMATS[kv_quant],
                     decode_sms)
    if output is None:
        output = torch.empty((N, num_heads * head_size), dtype=query.dtype, device=query.device)
    if workspace is None:
        ws = lib.pa_workspace_size(ctypes.byref(dims), num_heads, kv_num_heads)
        workspace = torch.empty(max(int(ws), 256), dtype=torch.uint8, device=query.device)
    s = (stream or torch.cuda.current_stream(query.device)).cuda_stream
    if (prep is not None or output_gate is not None or kv_quant is not None or
            (lse is not None and stages != STAGE_ALL)):
        ext = PaExtensions(None if lse is None else lse.data_ptr(),
                           ctypes.pointer(prep) if prep is not None else None,
                           None if output_gate is None else output_gate.data_ptr(),
                           None if k_scale is None else k_scale.data_ptr(),
                           None if v_scale is None else v_scale.data_ptr(), int(stages))
        st = lib.pa_paged_attention_ex(
            _ptr(query), _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
            _ptr(cumulative_sequence_length), _ptr(past_seqlens), _ptr(block_table), _ptr(slot_mapping),
            int(num_heads), int(kv_num_heads), float(scale), _ptr(output), ctypes.byref(ext),
            ctypes.byref(dims), _ptr(workspace), int(workspace.numel()), ctypes.c_void_p(s))
    elif lse is not None:
        st = lib.pa_paged_attention_lse(
            _ptr(query), _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
            _ptr(cumulative_sequence_length), _ptr(past_seqlens), _ptr(block_table), _ptr(slot_mapping),
            int(num_heads), int(kv_num_heads), float(scale), _ptr(output), _ptr(lse), ctypes.byref(dims),
            _ptr(workspace), int(workspace.numel()), ctypes.c_void_p(s))
    else:
        st = lib.pa_paged_attention_stages(
            _ptr(query), _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
            _ptr(cumulative_sequence_length), _ptr(past_seqlens), _ptr(block_table), _ptr(slot_mapping),
            int(num_heads), int(kv_num_heads), float(scale), _ptr(output), ctypes.byref(dims),
            _ptr(workspace), int(workspace.numel()), ctypes.c_void_p(s), int(stages))
    if st:
        raise PagedAttentionError(st, "pa_paged_attention")
    return output


__all__ = ["KV_SAME", "KV_INT8", "KV_INT4", "paged_attention", "workspace_size", "make_dims", "PaQkPrep", "PaExtensions", "read_device_error", "kernel_launch_count",
           "load_library", "PagedAttentionError", "PaDims", "LIBRARY_PATH"]
