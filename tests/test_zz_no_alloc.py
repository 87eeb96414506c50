"""The built-in-workspace entry point, for callers that cannot allocate device memory.

pa_paged_attention_static_workspace takes no workspace argument: it runs the operator in
a device array compiled into the library. This checks, through the C ABI, that calls in a
row on that one array give the same caches and the same outputs, bit for bit, as
pa_paged_attention with a caller-allocated workspace, and that both meet the oracle; that
decode-only calls whose decode kernel plans itself and planned calls can alternate on the
array without leaving stale state for each other; that the array's device error word is
readable through pa_static_workspace_read_device_error; and that a problem whose
workspace would not fit the built-in array is refused before any launch. Collected last,
so a run that stops at the first failure has already run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import varlen_paged_kv_gb300 as pa
import workloads as w
from gpu_utils import TORCH_DT, assert_close, bits_of, make_workspace, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is required for the gpu tests")
    from varlen_paged_kv_gb300 import build
    build.build()
    lib = pa.load_library()
    p = ctypes.c_void_p
    lib.pa_paged_attention_static_workspace.argtypes = [p] * 9 + [ctypes.c_int32, ctypes.c_int32, ctypes.c_float, p,
                                                        ctypes.POINTER(pa.PaDims), p]
    lib.pa_paged_attention_static_workspace.restype = ctypes.c_int
    lib.pa_static_workspace_read_device_error.argtypes = [p, ctypes.POINTER(ctypes.c_uint32)]
    lib.pa_static_workspace_read_device_error.restype = ctypes.c_int
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dims(prob, split, max_q):
    return pa.make_dims(prob.num_tokens, prob.batch_size, prob.head_size, prob.num_blocks, prob.block_size,
                        prob.max_blocks_per_sequence, TORCH_DT[prob.dtype], split, pa.ROUTE_AUTO, max_q)


def _call_static(lib, prob, d, dims, out):
    return lib.pa_paged_attention_static_workspace(
        _ptr(d["query"]), _ptr(d["key"]), _ptr(d["value"]), _ptr(d["key_cache"]), _ptr(d["value_cache"]),
        _ptr(d["cumulative_sequence_length"]), _ptr(d["past_seqlens"]), _ptr(d["block_table"]),
        _ptr(d["slot_mapping"]), prob.num_heads, prob.kv_num_heads, float(prob.scale), _ptr(out),
        ctypes.byref(dims), _stream())


def _static_error(lib):
    bits = ctypes.c_uint32(0)
    assert lib.pa_static_workspace_read_device_error(_stream(), ctypes.byref(bits)) == 0
    return int(bits.value)


def _caller_workspace_run(prob, split, max_q):
    """pa_paged_attention with its own workspace: (output bits, key cache bits, value cache bits)."""
    d = upload(prob)
    out = pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                             d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"],
                             d["slot_mapping"], num_heads=prob.num_heads, kv_num_heads=prob.kv_num_heads,
                             scale=prob.scale, decode_split_keys=split, max_query_len=max_q,
                             workspace=make_workspace(prob, split, pa.ROUTE_AUTO, max_q))
    return bits_of(out), bits_of(d["key_cache"]), bits_of(d["value_cache"])


CASES = {
    # the tiny workload with every decode unit cut into 64-key splits (partials and merge in the array)
    "tiny-split64": (lambda: w.config(1), 64, 0),
    # a mixed batch: the planner splits the SMs, split decode units are merged in the array
    "mixed": (lambda: w.make_problem(name="mixed", seed=11, dtype="bf16", num_heads=16, kv_num_heads=4,
                                     head_size=128, block_size=16, past=[3000, 17, 0, 900], q_lens=[1, 2, 200, 3]),
              0, 0),
    # a decode-only batch with the caller's bound: no planner, the decode kernel plans itself
    # (its merge counters and header reset by a one-CTA kernel)
    "self-planned": (lambda: w.make_problem(name="self", seed=12, dtype="fp16", num_heads=32, kv_num_heads=8,
                                            head_size=128, block_size=16, past=[6000, 5, 300, 2500, 0],
                                            q_lens=[1, 2, 1, 3, 1]), 0, 3),
}


def _expected(name):
    make, split, max_q = CASES[name]
    prob = make()
    ref = oracle.paged_attention(prob)
    return prob, split, max_q, ref, _caller_workspace_run(prob, split, max_q)


def _check_static(lib, prob, split, max_q, ref, caller):
    d = upload(prob)
    out = torch.empty((prob.num_tokens, prob.num_heads * prob.head_size), dtype=TORCH_DT[prob.dtype], device="cuda")
    assert _call_static(lib, prob, d, _dims(prob, split, max_q), out) == 0, lib.pa_last_error()
    assert _static_error(lib) == 0
    got = bits_of(out), bits_of(d["key_cache"]), bits_of(d["value_cache"])
    # the same kernels on the same plan: bit for bit the caller-workspace call
    assert np.array_equal(got[0], caller[0]), "output differs from the caller-workspace call"
    assert np.array_equal(got[1], caller[1]) and np.array_equal(got[2], caller[2])
    # and both meet the oracle
    assert np.array_equal(got[1], ref["key_cache"]) and np.array_equal(got[2], ref["value_cache"])
    assert_close(got[0].reshape(prob.num_tokens, prob.num_heads, prob.head_size), ref["out"], prob.dtype, prob.name)


@pytest.mark.parametrize("name", sorted(CASES))
def test_static_workspace_matches_caller_workspace_twice(lib, name):
    prob, split, max_q, ref, caller = _expected(name)
    for _ in range(2):  # two calls in a row on fresh copies of the inputs
        _check_static(lib, prob, split, max_q, ref, caller)


def test_self_planned_and_planned_calls_alternate_on_the_array(lib):
    # a self-planned call resets only what it uses; a planned call after it (and the next
    # self-planned call after that) must find nothing stale in the shared array
    a = _expected("self-planned")
    b = _expected("mixed")
    c = _expected("tiny-split64")
    for case in (a, b, a, c, a, b):
        _check_static(lib, *case)


def test_device_errors_are_readable_through_the_static_entry_point(lib):
    for name in ("self-planned", "mixed"):
        make, split, max_q = CASES[name]
        prob = make()
        prob.block_table = prob.block_table.copy()
        prob.block_table[0, 0] = 10 ** 6  # an active page outside the pool: read as zeros, flagged
        d = upload(prob)
        out = torch.empty((prob.num_tokens, prob.num_heads * prob.head_size), dtype=TORCH_DT[prob.dtype],
                          device="cuda")
        assert _call_static(lib, prob, d, _dims(prob, split, max_q), out) == 0, lib.pa_last_error()
        assert _static_error(lib) & pa.DEVERR_BAD_BLOCK
        assert _static_error(lib) == 0  # read and cleared
    # an inconsistent batch is refused on the device: nothing written, the bit readable
    make, split, max_q = CASES["mixed"]
    prob = make()
    prob.cumulative_sequence_length = prob.cumulative_sequence_length.copy()
    prob.cumulative_sequence_length[-1] -= 1
    d = upload(prob)
    before = bits_of(d["key_cache"]).copy()
    out = torch.empty((prob.num_tokens, prob.num_heads * prob.head_size), dtype=TORCH_DT[prob.dtype], device="cuda")
    assert _call_static(lib, prob, d, _dims(prob, split, max_q), out) == 0
    assert _static_error(lib) & pa.DEVERR_BAD_BATCH
    assert np.array_equal(bits_of(d["key_cache"]), before)


def test_static_workspace_refuses_sizes_beyond_its_array(lib):
    # a decode-only batch of 4096 sequences with 8 KV heads needs more workspace than the array holds
    dims = pa.make_dims(4096, 4096, 128, 8192, 16, 512, torch.float16)
    assert pa.workspace_size(dims, 32, 8) > 16 << 20
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    st = lib.pa_paged_attention_static_workspace(fake, fake, fake, fake, fake, fake, fake, fake, None, 32, 8, 0.0,
                                                 fake, ctypes.byref(dims), None)
    assert st == 3  # PA_ERR_WORKSPACE_TOO_SMALL
