"""The built-in-workspace entry point, for callers that cannot allocate device memory.

pa_paged_attention_static_workspace takes no workspace argument: it runs the operator in
a device array compiled into the library. This checks, through the C ABI, that two calls
in a row give the same caches (bit for bit) and the same outputs (within the tolerance
of the parity tests) as pa_paged_attention with a caller-allocated workspace, and that a
problem whose workspace would not fit the built-in array is refused before any launch.
Collected last, so a run that stops at the first failure has already run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import varlen_paged_kv_gb300 as pa
import workloads as w
from gpu_utils import ATOL, RTOL, TORCH_DT, bits_of, make_workspace, upload
from helpers import bits_to_f64

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
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_static(lib, prob, d, dims, out):
    s = torch.cuda.current_stream().cuda_stream
    return lib.pa_paged_attention_static_workspace(
        _ptr(d["query"]), _ptr(d["key"]), _ptr(d["value"]), _ptr(d["key_cache"]), _ptr(d["value_cache"]),
        _ptr(d["cumulative_sequence_length"]), _ptr(d["past_seqlens"]), _ptr(d["block_table"]),
        _ptr(d["slot_mapping"]), prob.num_heads, prob.kv_num_heads, float(prob.scale), _ptr(out),
        ctypes.byref(dims), ctypes.c_void_p(s))


def _close(a_bits, b_bits, dtype):
    a = bits_to_f64(a_bits, dtype)
    b = bits_to_f64(b_bits, dtype)
    assert np.all(np.abs(a - b) <= ATOL + RTOL * np.abs(b))


CASES = [
    # the tiny workload with every decode unit cut into 64-key splits (partials + merge in scratch)
    (lambda: w.config(1), 64),
    # decode batch with the balanced partition (split units merged in scratch) and a ragged prefill
    (lambda: w.make_problem(name="mixed", seed=11, dtype="bf16", num_heads=16, kv_num_heads=4, head_size=128,
                            block_size=16, past=[3000, 17, 0, 900], q_lens=[1, 2, 200, 3]), 0),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_static_workspace_matches_caller_workspace_twice(lib, case):
    make, split = CASES[case]
    prob = make()
    dims = pa.make_dims(prob.num_tokens, prob.batch_size, prob.head_size, prob.num_blocks, prob.block_size,
                        prob.max_blocks_per_sequence, TORCH_DT[prob.dtype], split)
    # the regular entry point with its own workspace
    ref = upload(prob)
    ref_out = pa.paged_attention(ref["query"], ref["key"], ref["value"], ref["key_cache"], ref["value_cache"],
                                 ref["cumulative_sequence_length"], ref["past_seqlens"], ref["block_table"],
                                 ref["slot_mapping"], num_heads=prob.num_heads, kv_num_heads=prob.kv_num_heads,
                                 scale=prob.scale, decode_split_keys=split, workspace=make_workspace(prob, split))
    torch.cuda.synchronize()
    # the built-in workspace, two calls in a row on fresh copies of the inputs
    for _ in range(2):
        d = upload(prob)
        out = torch.empty_like(ref_out)
        assert _call_static(lib, prob, d, dims, out) == 0, lib.pa_last_error()
        torch.cuda.synchronize()
        assert np.array_equal(bits_of(d["key_cache"]), bits_of(ref["key_cache"]))
        assert np.array_equal(bits_of(d["value_cache"]), bits_of(ref["value_cache"]))
        _close(bits_of(out), bits_of(ref_out), prob.dtype)


def test_static_workspace_refuses_sizes_beyond_its_array(lib):
    # a decode-only batch of 4096 sequences with 8 KV heads needs more workspace than the array holds
    dims = pa.make_dims(4096, 4096, 128, 8192, 16, 512, torch.float16)
    assert pa.workspace_size(dims, 32, 8) > 16 << 20
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    st = lib.pa_paged_attention_static_workspace(fake, fake, fake, fake, fake, fake, fake, fake, None, 32, 8, 0.0,
                                                 fake, ctypes.byref(dims), None)
    assert st == 3  # PA_ERR_WORKSPACE_TOO_SMALL
