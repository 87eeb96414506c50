"""The work partition covers every (query row, head, key) of the causal ranges exactly once.

The coverage build of the library (libpagedattn_cov.so, compiled with PA_COVERAGE) counts,
for every (row, head, key) that an attention kernel lets into its softmax, one in a device
array (pa_debug_coverage). Row j of sequence b must count each key 0 .. past_b + j exactly
once and nothing else, whatever the partition: forced split lengths, the balanced cut with
skewed units cut across CTAs, mixed batches on split SMs at several decode shares, the
decode kernel's own partition of a decode-only call (128 and 256 wide), the prefill
kernel's units (ragged tails, chunks with history, 64/128/256-wide heads) and integer
caches.
"""
import ctypes

import numpy as np
import pytest
import torch

import varlen_paged_kv_gb300 as pa
import workloads as w
from gpu_utils import TORCH_DT, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is required for the gpu tests")
    from varlen_paged_kv_gb300 import build
    lib = ctypes.CDLL(build.build(coverage=True))
    p, i32, u32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t
    dims_p = ctypes.POINTER(pa.PaDims)
    lib.pa_workspace_size.argtypes = [dims_p, i32, i32]
    lib.pa_workspace_size.restype = sz
    common = [p] * 9 + [i32, i32, f32, p]
    lib.pa_paged_attention_ex.argtypes = common + [ctypes.POINTER(pa.PaExtensions), dims_p, p, sz, p]
    lib.pa_paged_attention_ex.restype = ctypes.c_int
    lib.pa_debug_coverage.argtypes = [p, i32]
    lib.pa_debug_coverage.restype = ctypes.c_int
    lib.pa_read_device_error.argtypes = [p, p, ctypes.POINTER(u32)]
    lib.pa_read_device_error.restype = ctypes.c_int
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def coverage(lib, p, *, split=0, route=pa.ROUTE_AUTO, max_q=0, decode_sms=0):
    """Runs one call on the coverage build; returns the counts (N, nh, max_keys) and the
    overflow counter."""
    d = upload(p)
    dims = pa.make_dims(p.num_tokens, p.batch_size, p.head_size, p.num_blocks, p.block_size,
                        p.max_blocks_per_sequence, TORCH_DT[p.dtype], split, route, max_q, False,
                        p.kv_quant, decode_sms)
    ws = torch.zeros(lib.pa_workspace_size(ctypes.byref(dims), p.num_heads, p.kv_num_heads), dtype=torch.uint8,
                     device="cuda")
    keys = int(p.kv_lens.max()) + 256  # room past every causal range: a stray key is counted, not lost
    counts = torch.zeros(p.num_tokens * p.num_heads * keys + 1, dtype=torch.int32, device="cuda")
    ext = pa.PaExtensions(None, None, None, _ptr(d.get("k_scale")), _ptr(d.get("v_scale")), 0)
    out = torch.empty((p.num_tokens, p.num_heads * p.head_size), dtype=TORCH_DT[p.dtype], device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.pa_debug_coverage(_ptr(counts), keys) == 0
    try:
        st = lib.pa_paged_attention_ex(
            _ptr(d["query"]), _ptr(d["key"]), _ptr(d["value"]), _ptr(d["key_cache"]), _ptr(d["value_cache"]),
            _ptr(d["cumulative_sequence_length"]), _ptr(d["past_seqlens"]), _ptr(d["block_table"]),
            _ptr(d["slot_mapping"]), p.num_heads, p.kv_num_heads, float(p.scale), _ptr(out), ctypes.byref(ext),
            ctypes.byref(dims), _ptr(ws), ws.numel(), s)
        assert st == 0
        bits = ctypes.c_uint32(0)
        assert lib.pa_read_device_error(_ptr(ws), s, ctypes.byref(bits)) == 0
        assert bits.value == 0, f"device error bits {bits.value}"
    finally:
        assert lib.pa_debug_coverage(None, 0) == 0
    c = counts.cpu().numpy()
    return c[:-1].reshape(p.num_tokens, p.num_heads, keys), int(c[-1])


def check_exactly_once(lib, p, **kw):
    got, overflow = coverage(lib, p, **kw)
    assert overflow == 0
    pos = np.zeros(p.num_tokens, np.int64)  # each row's last visible key
    for b in range(p.batch_size):
        c0, c1 = int(p.cumulative_sequence_length[b]), int(p.cumulative_sequence_length[b + 1])
        pos[c0:c1] = int(p.past_seqlens[b]) + np.arange(c1 - c0)
    want = (np.arange(got.shape[2])[None, :] <= pos[:, None]).astype(np.int32)
    bad = got != want[:, None, :]
    if bad.any():
        i, h, t = np.argwhere(bad)[0]
        raise AssertionError(f"{p.name}: {bad.sum()} (row, head, key) counts wrong; first row {i} head {h} "
                             f"key {t}: counted {got[i, h, t]}, want {want[i, t]}")


def _prob(name, seed=5, **kw):
    return w.make_problem(name=name, seed=seed, **kw)


DECODE = dict(dtype="fp16", num_heads=32, kv_num_heads=8, head_size=128, block_size=16,
              past=[60000, 5, 17, 33000, 300, 1, 2, 3, 0, 4095], q_lens=[1, 2, 1, 3, 1, 4, 1, 1, 1, 2])


@pytest.mark.parametrize("split", [0, 64, 128, 448])
def test_decode_partition(lib, split):
    # skewed units: the long ones are cut across CTAs by the balanced cut, or by forced splits
    check_exactly_once(lib, _prob("cov-decode", **DECODE), split=split)


def test_self_planned_decode_partition(lib):
    p = _prob("cov-self", **DECODE)
    check_exactly_once(lib, p, max_q=int(p.q_lens.max()))


@pytest.mark.parametrize("fmt", [None, "int4"])
def test_self_planned_decode_partition_256(lib, fmt):
    p = _prob("cov-self-256", dtype="bf16", num_heads=16, kv_num_heads=2, head_size=256, block_size=16,
              past=[5000, 3, 700, 0, 2048, 64], q_lens=[1, 2, 1, 1, 2, 1], kv_quant=fmt)
    check_exactly_once(lib, p, max_q=2)


@pytest.mark.parametrize("hs,fmt", [(128, "int8"), (128, "int4"), (256, "int8")])
def test_narrow_decode_partition(lib, hs, fmt):
    # integer caches, at most 8 rows per item: the transposed (narrow) form of the decode kernel
    p = _prob("cov-narrow", dtype="fp16", num_heads=16, kv_num_heads=4, head_size=hs, block_size=32,
              past=[5000, 3, 800, 0, 129], q_lens=[1, 2, 2, 1, 2], kv_quant=fmt)
    check_exactly_once(lib, p, max_q=2)
    check_exactly_once(lib, p, max_q=2, split=64)


@pytest.mark.parametrize("dsm", [0, 1, 40, 151])
def test_mixed_batch_on_split_sms(lib, dsm):
    p = _prob("cov-mixed", dtype="bf16", num_heads=32, kv_num_heads=8, head_size=128, block_size=16,
              past=[3000, 0, 4000, 700, 5000, 33, 0], q_lens=[1, 300, 2, 1, 4, 129, 17])
    check_exactly_once(lib, p, decode_sms=dsm)


@pytest.mark.parametrize("hs,G", [(64, 1), (128, 4), (128, 3), (256, 8)])
def test_prefill_units(lib, hs, G):
    # every sequence on the prefill kernel: ragged tails, chunks with history not a multiple
    # of the tile, decode-length rows, head pairs (even G) and single heads (odd G, 256 wide)
    kvh = 2
    p = _prob(f"cov-prefill-{hs}-{G}", dtype="fp16", num_heads=kvh * G, kv_num_heads=kvh, head_size=hs,
              block_size=32, past=[0, 1000, 17, 255, 0], q_lens=[300, 129, 64, 1, 513])
    check_exactly_once(lib, p, route=pa.ROUTE_ALL_PREFILL)
    check_exactly_once(lib, p)


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_integer_cache_decode_partition(lib, fmt):
    p = _prob("cov-int", dtype="fp16", num_heads=16, kv_num_heads=4, head_size=128, block_size=64,
              past=[5000, 3, 800, 0], q_lens=[1, 2, 4, 1], kv_quant=fmt)
    check_exactly_once(lib, p, max_q=4)
    check_exactly_once(lib, p, max_q=4, split=64)


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_integer_cache_prefill_units(lib, fmt):
    p = _prob("cov-int-prefill", dtype="bf16", num_heads=16, kv_num_heads=4, head_size=128, block_size=32,
              past=[0, 700, 5], q_lens=[200, 1, 130], kv_quant=fmt)
    check_exactly_once(lib, p, max_q=200)
    check_exactly_once(lib, p, max_q=200, route=pa.ROUTE_ALL_PREFILL)
    q = _prob("cov-int-prefill-256", dtype="fp16", num_heads=8, kv_num_heads=2, head_size=256, block_size=32,
              past=[0, 300, 5], q_lens=[150, 1, 130], kv_quant=fmt)
    check_exactly_once(lib, q, max_q=150)
