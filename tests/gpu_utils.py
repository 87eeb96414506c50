"""Run the CUDA path on a workloads.Problem and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import varlen_paged_kv_gb300 as pa
from helpers import bits_to_f64

TORCH_DT = {"fp16": torch.float16, "bf16": torch.bfloat16}

# elementwise bound |gpu - oracle| <= ATOL + RTOL * |oracle| (oracle in fp64, before rounding)
ATOL, RTOL = 2e-3, 1e-2


def to_dev(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(TORCH_DT[dtype])


def idx_dev(a, device="cuda"):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def upload(p):
    d = dict(
        query=to_dev(p.query, p.dtype),
        key=None if p.key is None else to_dev(p.key, p.dtype),
        value=None if p.value is None else to_dev(p.value, p.dtype),
        key_cache=to_dev(p.key_cache, p.dtype) if p.kv_quant is None else torch.from_numpy(
            np.ascontiguousarray(p.key_cache, dtype=np.uint8)).to(device="cuda"),
        value_cache=to_dev(p.value_cache, p.dtype) if p.kv_quant is None else torch.from_numpy(
            np.ascontiguousarray(p.value_cache, dtype=np.uint8)).to(device="cuda"),
        cumulative_sequence_length=idx_dev(p.cumulative_sequence_length),
        past_seqlens=idx_dev(p.past_seqlens),
        block_table=idx_dev(p.block_table),
        slot_mapping=idx_dev(p.slot_mapping),
    )
    if p.kv_quant is not None:  # integer caches: their per-channel scales
        d["k_scale"] = torch.from_numpy(np.ascontiguousarray(p.k_scale, dtype=np.float32)).cuda()
        d["v_scale"] = torch.from_numpy(np.ascontiguousarray(p.v_scale, dtype=np.float32)).cuda()
    return d


def cache_bytes(t: torch.Tensor) -> np.ndarray:
    """A cache's contents as the oracle holds them: 16-bit bits, or code bytes."""
    return t.cpu().numpy() if t.dtype == torch.uint8 else bits_of(t)


def run_gpu(p, *, decode_split_keys=0, route=pa.ROUTE_AUTO, dev=None, decode_sms=0, max_query_len=0):
    """Runs the operator once. Returns dict(out_bits (N, nh*hs), key_cache, value_cache (bits),
    err (device error bits), dev (the uploaded tensors, caches updated in place))."""
    d = dev if dev is not None else upload(p)
    ws = make_workspace(p, decode_split_keys, route, max_query_len)
    out = pa.paged_attention(
        d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"], d["cumulative_sequence_length"],
        d["past_seqlens"], d["block_table"], d["slot_mapping"], num_heads=p.num_heads,
        kv_num_heads=p.kv_num_heads, scale=p.scale, decode_split_keys=decode_split_keys, route=route,
        workspace=ws, decode_sms=decode_sms, max_query_len=max_query_len)
    err = pa.read_device_error(ws)
    return dict(out_bits=bits_of(out), key_cache=bits_of(d["key_cache"]), value_cache=bits_of(d["value_cache"]),
                err=err, dev=d)


def make_workspace(p, decode_split_keys=0, route=pa.ROUTE_AUTO, max_query_len=0):
    dims = pa.make_dims(p.num_tokens, p.batch_size, p.head_size, p.num_blocks, p.block_size,
                        p.max_blocks_per_sequence, TORCH_DT[p.dtype], decode_split_keys, route, max_query_len)
    n = pa.workspace_size(dims, p.num_heads, p.kv_num_heads)
    assert n > 0
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def assert_close(gpu_bits: np.ndarray, ref_f64: np.ndarray, dtype: str, what=""):
    """gpu_bits: (..., hs) 16-bit results; ref_f64: the oracle's unrounded fp64 values."""
    g = bits_to_f64(gpu_bits, dtype).reshape(ref_f64.shape)
    err = np.abs(g - ref_f64)
    bound = ATOL + RTOL * np.abs(ref_f64)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements outside {ATOL}+{RTOL}|ref| "
            f"(max abs err {np.nanmax(err):.3g}); first {idx.tolist()} "
            f"gpu {g[tuple(idx[0])]:.6g} ref {ref_f64[tuple(idx[0])]:.6g}")
    return float(np.max(err)) if err.size else 0.0
