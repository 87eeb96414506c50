"""CPU oracle for com.microsoft.PagedAttention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package. The product path never does; it shares no code with the CUDA
implementation.

``paged_attention_oracle.c`` is the definition of the operator written out in fp64
(com.microsoft.PagedAttention README, "Description", "Inputs", "Attributes"): the
cache write, then causal grouped-query attention of every query row over its
sequence's history read back through ``block_table``, rounded once to the 16-bit type.
This module compiles it with gcc (OpenMP over (sequence, head) pairs) and marshals
numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attention_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {
    -1: "bad shape", -2: "bad cumulative_sequence_length / past_seqlens",
    -3: "slot out of range", -4: "two tokens write one slot",
    -5: "block_table entry out of range for an active page", -6: "out of memory",
    -7: "sequence longer than max_blocks_per_sequence * block_size",
}


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle rejected the input: {ERRORS.get(code, code)} ({code})")
        self.code = code


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    i32, f32, p, u16, dbl = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_uint16, ctypes.c_double
    lib.oracle_f16_to_double.argtypes = [u16]
    lib.oracle_f16_to_double.restype = dbl
    lib.oracle_bf16_to_double.argtypes = [u16]
    lib.oracle_bf16_to_double.restype = dbl
    lib.oracle_double_to_f16.argtypes = [dbl]
    lib.oracle_double_to_f16.restype = u16
    lib.oracle_double_to_bf16.argtypes = [dbl]
    lib.oracle_double_to_bf16.restype = u16
    lib.oracle_scatter.argtypes = [i32] * 8 + [p] * 9
    lib.oracle_scatter.restype = ctypes.c_int
    lib.oracle_attention.argtypes = [ctypes.c_int] + [i32] * 9 + [p] * 6 + [f32, p, p, p, ctypes.c_int]
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention_rows.argtypes = ([ctypes.c_int] + [i32] * 9 + [p] * 6 + [f32, i32] +
                                          [p] * 4 + [ctypes.c_int])
    lib.oracle_attention_rows.restype = ctypes.c_int
    lib.oracle_qk_prep.argtypes = ([ctypes.c_int] + [i32] * 5 + [ctypes.c_int64] + [p] * 6 + [dbl, i32, dbl] +
                                   [p, p])
    lib.oracle_qk_prep.restype = ctypes.c_int
    lib.oracle_round_array.argtypes = [ctypes.c_int, p, ctypes.c_int64, p]
    lib.oracle_round_array.restype = None
    lib.oracle_apply_gate.argtypes = [ctypes.c_int, ctypes.c_int64, p, p, p, p]
    lib.oracle_apply_gate.restype = ctypes.c_int
    i64 = ctypes.c_int64
    lib.oracle_quantize_rows.argtypes = [ctypes.c_int, ctypes.c_int, i64, i32, i32, p, i64, p, p]
    lib.oracle_quantize_rows.restype = ctypes.c_int
    lib.oracle_scatter_codes.argtypes = [i32] * 5 + [i64] + [p] * 8
    lib.oracle_scatter_codes.restype = ctypes.c_int
    lib.oracle_attention_q.argtypes = ([ctypes.c_int, ctypes.c_int] + [i32] * 9 + [p] * 8 + [f32, p, p, p, ctypes.c_int])
    lib.oracle_attention_q.restype = ctypes.c_int
    lib.oracle_attention_rows_q.argtypes = ([ctypes.c_int, ctypes.c_int] + [i32] * 9 + [p] * 8 + [f32, i32] + [p] * 4 +
                                            [ctypes.c_int])
    lib.oracle_attention_rows_q.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB)
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return _load().oracle_max_threads()


# ---- scalar conversions (exposed for the pins) -------------------------------------

def f16_to_double(bits) -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_f16_to_double(int(b)) for b in np.ravel(bits)])


def bf16_to_double(bits) -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_bf16_to_double(int(b)) for b in np.ravel(bits)])


def double_to_f16(x) -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_double_to_f16(float(v)) for v in np.ravel(x)], dtype=np.uint16)


def double_to_bf16(x) -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_double_to_bf16(float(v)) for v in np.ravel(x)], dtype=np.uint16)


# ---- the operator ------------------------------------------------------------------

def _dims(p):
    N = int(p.query.shape[0])
    B = int(np.asarray(p.past_seqlens).shape[0])
    return (N, B, int(p.num_heads), int(p.kv_num_heads), int(p.head_size), int(p.num_blocks),
            int(p.block_size), int(np.asarray(p.block_table).shape[1]))


def scatter(p):
    """Step 1 on copies of the caches. Returns (key_cache, value_cache)."""
    lib = _load()
    kc = np.array(p.key_cache, dtype=np.uint16, copy=True)
    vc = np.array(p.value_cache, dtype=np.uint16, copy=True)
    q = _c(p.query, np.uint16)
    k = _c(p.key, np.uint16)
    v = _c(p.value, np.uint16)
    cum = _c(p.cumulative_sequence_length, np.int32)
    past = _c(p.past_seqlens, np.int32)
    bt = _c(p.block_table, np.int32)
    sm = _c(p.slot_mapping, np.int32)
    rc = lib.oracle_scatter(*_dims(p), _ptr(q), _ptr(k), _ptr(v), _ptr(kc), _ptr(vc), _ptr(cum),
                            _ptr(past), _ptr(bt), _ptr(sm))
    if rc:
        raise OracleError(rc)
    return kc, vc


def attention(p, key_cache, value_cache, nthreads: int = 0):
    """Step 2 given caches after the write. Returns (out f64 (N, nh, hs), lse (N, nh), out_bits (N, nh*hs))."""
    lib = _load()
    N, B, nh, kvh, hs, nblk, bs, mb = _dims(p)
    q = _c(p.query, np.uint16)
    out = np.zeros((N, nh, hs), dtype=np.float64)
    lse = np.zeros((N, nh), dtype=np.float64)
    bits = np.zeros((N, nh * hs), dtype=np.uint16)
    dt = 1 if p.dtype == "bf16" else 0
    rc = lib.oracle_attention(dt, N, B, nh, kvh, hs, nblk, bs, mb, int(q.shape[1]), _ptr(q),
                              _ptr(_c(key_cache, np.uint16)), _ptr(_c(value_cache, np.uint16)),
                              _ptr(_c(p.cumulative_sequence_length, np.int32)),
                              _ptr(_c(p.past_seqlens, np.int32)), _ptr(_c(p.block_table, np.int32)),
                              float(p.scale), _ptr(out), _ptr(lse), _ptr(bits), nthreads)
    if rc:
        raise OracleError(rc)
    return out, lse, bits


def attention_rows(p, key_cache, value_cache, tokens, heads, nthreads: int = 0):
    """Step 2 for selected (token, head) pairs only. Returns (out (n, hs), lse (n,))."""
    lib = _load()
    N, B, nh, kvh, hs, nblk, bs, mb = _dims(p)
    q = _c(p.query, np.uint16)
    tokens = _c(tokens, np.int32)
    heads = _c(heads, np.int32)
    n = int(tokens.shape[0])
    out = np.zeros((n, hs), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    dt = 1 if p.dtype == "bf16" else 0
    rc = lib.oracle_attention_rows(dt, N, B, nh, kvh, hs, nblk, bs, mb, int(q.shape[1]), _ptr(q),
                                   _ptr(_c(key_cache, np.uint16)), _ptr(_c(value_cache, np.uint16)),
                                   _ptr(_c(p.cumulative_sequence_length, np.int32)),
                                   _ptr(_c(p.past_seqlens, np.int32)), _ptr(_c(p.block_table, np.int32)),
                                   float(p.scale), n, _ptr(tokens), _ptr(heads), _ptr(out), _ptr(lse),
                                   nthreads)
    if rc:
        raise OracleError(rc)
    return out, lse


# ---- Q/K preparation (RMSNorm, rotary embedding) before the cache write -------------
# prep: dict(q_norm_weight=uint16 bits (hs,) or None, k_norm_weight=... or None, eps=float,
#            rotary_dim=int (0: none), theta=float)

def qk_prep_f64(p, prep):
    """The prepared Q (N, nh, hs) and K (N, kvh, hs), unrounded (oracle_qk_prep)."""
    lib = _load()
    N, B, nh, kvh, hs = _dims(p)[:5]
    q = _c(p.query, np.uint16)
    k = _c(p.key, np.uint16)
    oq = np.zeros((N, nh, hs), dtype=np.float64)
    ok = np.zeros((N, kvh, hs), dtype=np.float64)
    qw = _c(prep.get("q_norm_weight"), np.uint16)
    kw = _c(prep.get("k_norm_weight"), np.uint16)
    dt = 1 if p.dtype == "bf16" else 0
    rc = lib.oracle_qk_prep(dt, N, B, nh, kvh, hs, int(q.shape[1]), _ptr(q), _ptr(k),
                            _ptr(_c(p.cumulative_sequence_length, np.int32)), _ptr(_c(p.past_seqlens, np.int32)),
                            _ptr(qw), _ptr(kw), float(prep.get("eps", 1e-6)), int(prep.get("rotary_dim", 0)),
                            float(prep.get("theta", 10000.0)), _ptr(oq), _ptr(ok))
    if rc:
        raise OracleError(rc)
    return oq, ok


def round_bits(x, dtype: str) -> np.ndarray:
    """fp64 values rounded once to fp16 / bf16 bits (round to nearest even)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint16)
    _load().oracle_round_array(1 if dtype == "bf16" else 0, _ptr(x), int(x.size), _ptr(out))
    return out


def apply_qk_prep(p, prep):
    """A copy of the problem whose query and key rows are the prepared ones rounded to T
    (V and everything else unchanged): the operator with preparation is the operator on it."""
    import copy
    N, B, nh, kvh, hs = _dims(p)[:5]
    oq, ok = qk_prep_f64(p, prep)
    qb = round_bits(oq, p.dtype).reshape(N, nh * hs)
    kb = round_bits(ok, p.dtype).reshape(N, kvh * hs)
    r = copy.copy(p)
    if p.key is None:  # packed [Q | K | V] rows
        rows = np.array(p.query, dtype=np.uint16, copy=True)
        rows[:, :nh * hs] = qb
        rows[:, nh * hs:(nh + kvh) * hs] = kb
        r.query = rows
    else:
        r.query = qb
        r.key = kb
    return r


def apply_gate(out, gate_bits, dtype: str):
    """out (fp64, any shape) times sigmoid(gate) elementwise (oracle_apply_gate): returns
    (gated fp64, gated bits rounded to T)."""
    out = np.ascontiguousarray(out, dtype=np.float64)
    g = np.ascontiguousarray(gate_bits, dtype=np.uint16).reshape(out.shape)
    gated = np.zeros(out.shape, dtype=np.float64)
    bits = np.zeros(out.shape, dtype=np.uint16)
    rc = _load().oracle_apply_gate(1 if dtype == "bf16" else 0, int(out.size), _ptr(out), _ptr(g), _ptr(gated),
                                   _ptr(bits))
    if rc:
        raise OracleError(rc)
    return gated, bits


# ---- integer KV caches (INT8 / INT4 codes with per-(KV head, channel) fp32 scales) -------

KV_KIND = {"int8": 1, "int4": 2}


def quantize_rows(x_bits, dtype: str, fmt: str, kvh: int, hs: int, scale) -> np.ndarray:
    """Rows of kvh*hs values of T (bits, (n, kvh*hs) or wider rows sliced by the caller) to
    code rows (oracle_quantize_rows): uint8 (n, kvh*hs) for int8, (n, kvh*hs/2) for int4."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    n = int(x.shape[0])
    rb = kvh * hs if fmt == "int8" else kvh * hs // 2
    codes = np.zeros((n, rb), dtype=np.uint8)
    rc = _load().oracle_quantize_rows(1 if dtype == "bf16" else 0, KV_KIND[fmt], n, kvh, hs, _ptr(x),
                                      int(x.shape[1]) if x.ndim == 2 else kvh * hs,
                                      _ptr(_c(scale, np.float32)), _ptr(codes))
    if rc:
        raise OracleError(rc)
    return codes


def kv_rows(p):
    """This call's K and V rows (bits, (N, kvh*hs) each), from the packed rows if packed."""
    nh, kvh, hs = int(p.num_heads), int(p.kv_num_heads), int(p.head_size)
    if p.key is None:
        q = np.asarray(p.query, dtype=np.uint16)
        return q[:, nh * hs:(nh + kvh) * hs], q[:, (nh + kvh) * hs:]
    return p.key, p.value


def scatter_codes(p, k_codes, v_codes):
    """The cache write of an integer-cache problem on copies of its code caches."""
    lib = _load()
    N, B, nh, kvh, hs, nblk, bs, mb = _dims(p)
    kc = np.array(p.key_cache, dtype=np.uint8, copy=True)
    vc = np.array(p.value_cache, dtype=np.uint8, copy=True)
    rb = int(np.asarray(k_codes).shape[1]) if N else (kvh * hs if p.kv_quant == "int8" else kvh * hs // 2)
    rc = lib.oracle_scatter_codes(N, B, nblk, bs, mb, rb, _ptr(_c(k_codes, np.uint8)), _ptr(_c(v_codes, np.uint8)),
                                  _ptr(kc), _ptr(vc), _ptr(_c(p.cumulative_sequence_length, np.int32)),
                                  _ptr(_c(p.past_seqlens, np.int32)), _ptr(_c(p.block_table, np.int32)),
                                  _ptr(_c(p.slot_mapping, np.int32)))
    if rc:
        raise OracleError(rc)
    return kc, vc


def attention_q(p, key_cache, value_cache, nthreads: int = 0):
    """Attention over integer caches (after the write). Returns (out, lse, out_bits)."""
    lib = _load()
    N, B, nh, kvh, hs, nblk, bs, mb = _dims(p)
    q = _c(p.query, np.uint16)
    out = np.zeros((N, nh, hs), dtype=np.float64)
    lse = np.zeros((N, nh), dtype=np.float64)
    bits = np.zeros((N, nh * hs), dtype=np.uint16)
    rc = lib.oracle_attention_q(1 if p.dtype == "bf16" else 0, KV_KIND[p.kv_quant], N, B, nh, kvh, hs, nblk, bs, mb,
                                int(q.shape[1]), _ptr(q), _ptr(_c(key_cache, np.uint8)),
                                _ptr(_c(value_cache, np.uint8)), _ptr(_c(p.k_scale, np.float32)),
                                _ptr(_c(p.v_scale, np.float32)), _ptr(_c(p.cumulative_sequence_length, np.int32)),
                                _ptr(_c(p.past_seqlens, np.int32)), _ptr(_c(p.block_table, np.int32)),
                                float(p.scale), _ptr(out), _ptr(lse), _ptr(bits), nthreads)
    if rc:
        raise OracleError(rc)
    return out, lse, bits


def attention_rows_q(p, key_cache, value_cache, tokens, heads, nthreads: int = 0):
    """attention_q for selected (token, head) pairs only. Returns (out (n, hs), lse (n,))."""
    lib = _load()
    N, B, nh, kvh, hs, nblk, bs, mb = _dims(p)
    q = _c(p.query, np.uint16)
    tokens = _c(tokens, np.int32)
    heads = _c(heads, np.int32)
    n = int(tokens.shape[0])
    out = np.zeros((n, hs), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    rc = lib.oracle_attention_rows_q(1 if p.dtype == "bf16" else 0, KV_KIND[p.kv_quant], N, B, nh, kvh, hs, nblk,
                                     bs, mb, int(q.shape[1]), _ptr(q), _ptr(_c(key_cache, np.uint8)),
                                     _ptr(_c(value_cache, np.uint8)), _ptr(_c(p.k_scale, np.float32)),
                                     _ptr(_c(p.v_scale, np.float32)),
                                     _ptr(_c(p.cumulative_sequence_length, np.int32)),
                                     _ptr(_c(p.past_seqlens, np.int32)), _ptr(_c(p.block_table, np.int32)),
                                     float(p.scale), n, _ptr(tokens), _ptr(heads), _ptr(out), _ptr(lse), nthreads)
    if rc:
        raise OracleError(rc)
    return out, lse


def paged_attention(p, nthreads: int = 0, prep=None, gate=None):
    """The whole operator: returns dict(key_cache, value_cache, out, lse, out_bits). With
    `prep`, the query and key rows are prepared (RMSNorm, rotary embedding) first; with
    `gate` (bits, (N, nh*hs)), the output is multiplied by sigmoid(gate) before rounding.
    An integer-cache problem (p.kv_quant) quantizes this call's K and V rows with its
    scales, writes the codes and attends over code * scale."""
    if prep is not None:
        p = apply_qk_prep(p, prep)
    if p.kv_quant is not None:
        kr, vr = kv_rows(p)
        kvh, hs = int(p.kv_num_heads), int(p.head_size)
        kq = quantize_rows(kr, p.dtype, p.kv_quant, kvh, hs, p.k_scale)
        vq = quantize_rows(vr, p.dtype, p.kv_quant, kvh, hs, p.v_scale)
        kc, vc = scatter_codes(p, kq, vq)
        out, lse, bits = attention_q(p, kc, vc, nthreads)
    else:
        kc, vc = scatter(p)
        out, lse, bits = attention(p, kc, vc, nthreads)
    if gate is not None:
        out, b = apply_gate(out, gate, p.dtype)
        bits = b.reshape(bits.shape)
    return {"key_cache": kc, "value_cache": vc, "out": out, "lse": lse, "out_bits": bits}
