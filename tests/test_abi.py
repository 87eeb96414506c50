"""The C ABI on the host: the library loads, exports every symbol the header declares,
sizes its workspace, and rejects bad arguments with typed errors before any CUDA call
(so none of this needs a GPU)."""
import ctypes
import os
import re

import pytest
import torch

import varlen_paged_kv_gb300 as pa
from varlen_paged_kv_gb300 import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pagedattn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pa.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "pa_paged_attention" in names and len(names) >= 7
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_status_strings(lib):
    assert lib.pa_abi_version() == 7
    for code in range(5):
        assert lib.pa_status_string(code)
    assert lib.pa_status_string(99) == b"unknown status"


def test_workspace_size_bounds(lib):
    d = pa.make_dims(64, 64, 128, 607, 256, 17, torch.float16)
    n = pa.workspace_size(d, 32, 8)
    assert 0 < n < 64 << 20
    # more sequences or a forced short split never need less
    d2 = pa.make_dims(64, 64, 128, 607, 256, 17, torch.float16, decode_split_keys=64)
    assert pa.workspace_size(d2, 32, 8) >= n
    assert pa.workspace_size(pa.make_dims(64, 64, 96, 607, 256, 17, torch.float16), 32, 8) == 0  # head_size 96
    assert pa.workspace_size(pa.make_dims(64, 64, 128, 607, 24, 17, torch.float16), 32, 8) == 0   # block 24
    assert pa.workspace_size(d, 32, 5) == 0                                                        # 32 % 5
    assert pa.workspace_size(pa.make_dims(64, 64, 256, 607, 256, 17, torch.float16), 32, 8) >= n  # head_size 256
    assert pa.workspace_size(pa.make_dims(64, 64, 512, 607, 256, 17, torch.float16), 32, 8) == 0  # head_size 512


FAKE = 1 << 20  # an aligned non-null address that is never dereferenced: every case fails validation first


def _call(lib, dims, *, key=FAKE, value=FAKE, nh=32, kvh=8, ws=FAKE, ws_bytes=1 << 30, query=FAKE, output=FAKE):
    p = ctypes.c_void_p
    return lib.pa_paged_attention(p(query), p(key) if key else None, p(value) if value else None, p(FAKE),
                                  p(FAKE), p(FAKE), p(FAKE), p(FAKE), None, nh, kvh, 0.0, p(output),
                                  ctypes.byref(dims), p(ws), ws_bytes, None)


def test_typed_errors_before_any_launch(lib):
    good = pa.make_dims(64, 64, 128, 607, 256, 17, torch.float16)
    assert _call(lib, good, key=FAKE, value=0) == 1                       # key without value
    assert _call(lib, good, nh=30, kvh=8) == 1                            # heads not divisible
    assert _call(lib, pa.make_dims(64, 64, 80, 607, 256, 17, torch.float16)) == 2   # head_size
    assert _call(lib, pa.make_dims(64, 64, 512, 607, 256, 17, torch.float16)) == 2  # head_size 512
    assert _call(lib, pa.make_dims(64, 64, 128, 607, 8, 17, torch.float16)) == 2    # block_size 8
    assert _call(lib, pa.make_dims(64, 64, 128, 607, 256, 17, 7)) == 2              # dtype code
    assert _call(lib, pa.make_dims(64, 0, 128, 607, 256, 17, torch.float16)) == 1   # rows without sequences
    assert _call(lib, pa.make_dims(64, 64, 128, 607, 256, 17, torch.float16, decode_split_keys=100)) == 1
    assert _call(lib, pa.make_dims(64, 64, 128, 607, 256, 17, torch.float16, route=5)) == 1
    assert _call(lib, good, query=FAKE + 8) == 1                          # misaligned
    assert _call(lib, good, output=0) == 1                                # null output
    assert _call(lib, good, ws_bytes=100) == 3                            # workspace too small
    assert _call(lib, pa.make_dims(0, 0, 128, 607, 256, 17, torch.float16)) == 0    # nothing to do


def test_lse_entry_point_checks_before_any_launch(lib):
    good = pa.make_dims(64, 64, 128, 607, 256, 17, torch.float16)
    ws_bytes = lib.pa_workspace_size(ctypes.byref(good), 32, 8)
    p = ctypes.c_void_p

    def call(lse, dims=good):
        return lib.pa_paged_attention_lse(p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE),
                                          None, 32, 8, 0.0, p(FAKE), lse, ctypes.byref(dims), p(FAKE), ws_bytes,
                                          None)
    assert call(p(FAKE + 2)) == 1                                         # misaligned lse
    assert call(p(FAKE), pa.make_dims(64, 64, 80, 607, 256, 17, torch.float16)) == 2   # head_size
    assert call(p(FAKE), pa.make_dims(0, 0, 128, 607, 256, 17, torch.float16)) == 0   # nothing to do


def test_integer_cache_checks_before_any_launch(lib):
    p = ctypes.c_void_p
    dec = dict(max_query_len=1)  # decode-only

    def dims(hs=128, fmt=pa.KV_INT8, **kw):
        return pa.make_dims(64, 64, hs, 607, 256, 17, torch.float16, kv_dtype=fmt, **{**dec, **kw})

    def call(d, k_scale=FAKE, v_scale=FAKE):
        ext = pa.PaExtensions(None, None, None, k_scale, v_scale)
        ws = max(lib.pa_workspace_size(ctypes.byref(d), 32, 8), 1 << 20)
        return lib.pa_paged_attention_ex(p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE),
                                         None, 32, 8, 0.0, p(FAKE), ctypes.byref(ext), ctypes.byref(d), p(FAKE), ws,
                                         None)
    assert pa.workspace_size(dims(), 32, 8) > pa.workspace_size(dims(fmt=pa.KV_SAME), 32, 8)  # scaled Q rows
    assert pa.workspace_size(dims(hs=64, fmt=pa.KV_INT4), 32, 8) == 0    # INT4 needs head_size 128 or 256
    assert pa.workspace_size(dims(fmt=3), 32, 8) == 0                    # unknown format
    assert pa.workspace_size(dims(max_query_len=0), 32, 8) > 0           # prefill rows: the prefill kernel
    assert pa.workspace_size(dims(max_query_len=5, fmt=pa.KV_INT4), 32, 8) > 0
    assert pa.workspace_size(dims(hs=256, max_query_len=0), 32, 8) > 0
    assert call(dims(hs=64, fmt=pa.KV_INT4)) == 2
    assert call(dims(), k_scale=None) == 1                               # scales required
    assert call(dims(), v_scale=FAKE + 4) == 1                           # misaligned scale
    assert call(dims(fmt=pa.KV_SAME)) == 1                               # scales without integer caches


def test_python_binding_refuses_cpu_tensors(lib):
    q = torch.zeros(2, 64, dtype=torch.float16)
    c = torch.zeros(1, 16, 1, 64, dtype=torch.float16)
    i = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError):
        pa.paged_attention(q, None, None, c, c, i, i[:1], i.reshape(1, 2), num_heads=1, kv_num_heads=1)
