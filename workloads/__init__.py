"""Seeded synthetic inputs for paged attention over packed variable-length batches.

This module draws inputs and lays out the page pool; it holds none of the attention
arithmetic. Both the oracle and the CUDA path consume what it returns.

The recipes follow the workloads of the operator statement
(com.microsoft.PagedAttention README, "Inputs"): packed query rows
``(num_tokens, num_heads*head_size)`` or packed ``[Q|K|V]`` rows, K/V caches of shape
``(num_blocks, block_size, kv_num_heads, head_size)``, ``cumulative_sequence_length``,
``past_seqlens``, ``block_table`` and an optional ``slot_mapping``.

Random numbers come from ``synth.c`` (SplitMix64 over a Weyl sequence, Box-Muller
normals, round-to-nearest-even to fp16/bf16). Each array has its own stream id, so
the value of any element does not depend on the sizes of other arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# stream ids (one per drawn array)
S_PAST, S_QLEN, S_PAGES, S_QUERY, S_KEY, S_VALUE, S_KCACHE, S_VCACHE, S_DROP, S_ORDER = range(1, 11)
S_KSCALE, S_VSCALE = 11, 12

# integer KV caches: the largest code magnitude of each format (symmetric codes)
KV_QMAX = {"int8": 127, "int4": 7}

DTYPE_CODE = {"fp16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so next to it (gcc, OpenMP, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
             _SRC, "-o", tmp],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u64, i64, i32, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int, ctypes.c_double
            p = ctypes.c_void_p
            lib.synth_u64.argtypes = [u64, u64, u64, i64, p]
            lib.synth_uniform.argtypes = [u64, u64, u64, i64, p]
            lib.synth_normal_bits.argtypes = [u64, u64, u64, i64, i32, p]
            lib.synth_uniform_bits.argtypes = [u64, u64, u64, i64, dbl, dbl, i32, p]
            lib.synth_normal_f64.argtypes = [u64, u64, u64, i64, p]
            for f in (lib.synth_u64, lib.synth_uniform, lib.synth_normal_bits,
                      lib.synth_uniform_bits, lib.synth_normal_f64):
                f.restype = None
            _lib = lib
    return _lib


def u64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_u64(seed, stream, offset, n, out.ctypes.data)
    return out


def uniform(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_uniform(seed, stream, offset, n, out.ctypes.data)
    return out


def normal_f64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_normal_f64(seed, stream, offset, n, out.ctypes.data)
    return out


def normal_bits(seed: int, stream: int, shape, dtype: str) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_normal_bits(seed, stream, 0, out.size, DTYPE_CODE[dtype], out.ctypes.data)
    return out


def uniform_bits(seed: int, stream: int, shape, dtype: str, lo: float, hi: float) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_uniform_bits(seed, stream, 0, out.size, lo, hi, DTYPE_CODE[dtype], out.ctypes.data)
    return out


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] (inclusive)."""
    u = uniform(seed, stream, n)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64).clip(lo, hi)


def code_bytes(seed: int, stream: int, shape, fmt: str) -> np.ndarray:
    """Seeded contents of an integer cache of `shape` (..., hs) values: codes uniform in
    [-qmax, qmax], as bytes: int8 one two's complement byte per value, int4 two values per
    byte (even channel in the low nibble), shape (..., hs / 2)."""
    qm = KV_QMAX[fmt]
    n = int(np.prod(shape))
    nbytes = n if fmt == "int8" else n // 2
    raw = u64(seed, stream, (nbytes + 7) // 8).view(np.uint8)[:nbytes].astype(np.int32)
    if fmt == "int8":
        return ((raw % (2 * qm + 1)) - qm).astype(np.int8).view(np.uint8).reshape(shape)
    lo = ((raw & 0x0F) % (2 * qm + 1)) - qm
    hi = ((raw >> 4) % (2 * qm + 1)) - qm
    return ((lo & 0x0F) | ((hi & 0x0F) << 4)).astype(np.uint8).reshape(tuple(shape[:-1]) + (shape[-1] // 2,))


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """A seeded permutation of range(n): stable argsort of n 64-bit draws."""
    return np.argsort(u64(seed, stream, n), kind="stable").astype(np.int64)


@dataclass
class Problem:
    """One invocation's inputs. 16-bit floating arrays are held as raw bit patterns (uint16)."""

    name: str
    dtype: str                      # "fp16" | "bf16"
    num_heads: int
    kv_num_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    past_seqlens: np.ndarray        # int32 (B,)
    q_lens: np.ndarray              # int32 (B,)
    cumulative_sequence_length: np.ndarray  # int32 (B+1,)
    block_table: np.ndarray         # int32 (B, max_blocks_per_sequence)
    query: np.ndarray               # uint16 (N, W)
    key: Optional[np.ndarray]       # uint16 (N, kvh*hs) or None (packed [Q|K|V])
    value: Optional[np.ndarray]
    key_cache: np.ndarray           # uint16 (num_blocks, block_size, kvh, hs)
    value_cache: np.ndarray
    slot_mapping: Optional[np.ndarray]  # int32 (N,) or None
    scale: float = 0.0
    seed: int = 0
    notes: dict = field(default_factory=dict)
    # integer KV caches: "int8" | "int4" | None (caches of type T). With a format the caches
    # hold code bytes, uint8 (num_blocks, block_size, kvh, hs) for int8 and
    # (num_blocks, block_size, kvh, hs / 2) for int4 (channel 2i in the low nibble), and
    # k_scale / v_scale are the fp32 per-(KV head, channel) scales (kvh, hs).
    kv_quant: Optional[str] = None
    k_scale: Optional[np.ndarray] = None
    v_scale: Optional[np.ndarray] = None

    @property
    def batch_size(self) -> int:
        return int(self.past_seqlens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.query.shape[0])

    @property
    def packed(self) -> bool:
        return self.key is None

    @property
    def kv_lens(self) -> np.ndarray:
        return self.past_seqlens.astype(np.int64) + self.q_lens.astype(np.int64)

    @property
    def max_blocks_per_sequence(self) -> int:
        return int(self.block_table.shape[1])

    def copy(self) -> "Problem":
        c = Problem(**{k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in self.__dict__.items()})
        c.notes = dict(self.notes)
        return c


def make_problem(
    *,
    name: str,
    seed: int,
    dtype: str,
    num_heads: int,
    kv_num_heads: int,
    head_size: int,
    block_size: int,
    past,
    q_lens,
    packed: bool = False,
    dist: str = "normal",
    slot_mode: str = "omitted",      # "omitted" | "explicit"
    drop_count: int = 0,             # with slot_mode="explicit": tokens whose slot is -1
    num_blocks: Optional[int] = None,
    max_blocks_per_sequence: Optional[int] = None,
    table_fill: str = "pad",         # "pad": -1 after the active pages | "perm": all entries distinct ids
    scale: float = 0.0,
    kv_quant: Optional[str] = None,  # "int8" | "int4": integer caches with per-channel scales
) -> Problem:
    past = np.asarray(past, dtype=np.int64)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    B = past.shape[0]
    assert q_lens.shape == (B,)
    kv = past + q_lens
    bs = block_size
    pages = (kv + bs - 1) // bs
    need = int(pages.sum())
    if num_blocks is None:
        num_blocks = max(need, 1)
    if max_blocks_per_sequence is None:
        max_blocks_per_sequence = max(int(pages.max()) if B else 1, 1)
    assert num_blocks >= need and max_blocks_per_sequence >= (int(pages.max()) if B else 0)

    perm = permutation(seed, S_PAGES, num_blocks)
    bt = np.full((B, max_blocks_per_sequence), -1, dtype=np.int32)
    if table_fill == "perm":
        assert B * max_blocks_per_sequence == num_blocks
        bt[:] = perm.reshape(B, max_blocks_per_sequence)
    else:
        pos = 0
        for b in range(B):
            bt[b, : pages[b]] = perm[pos: pos + pages[b]]
            pos += int(pages[b])

    cum = np.zeros(B + 1, dtype=np.int32)
    cum[1:] = np.cumsum(q_lens)
    N = int(cum[-1])
    nh, kvh, hs = num_heads, kv_num_heads, head_size
    W = (nh + 2 * kvh) * hs if packed else nh * hs

    def draw(stream, shape):
        if dist == "normal":
            return normal_bits(seed, stream, shape, dtype)
        return uniform_bits(seed, stream, shape, dtype, -1.0, 1.0)

    query = draw(S_QUERY, (N, W))
    key = value = None
    if not packed:
        key = draw(S_KEY, (N, kvh * hs))
        value = draw(S_VALUE, (N, kvh * hs))
    k_scale = v_scale = None
    if kv_quant is None:
        kc = draw(S_KCACHE, (num_blocks, bs, kvh, hs))
        vc = draw(S_VCACHE, (num_blocks, bs, kvh, hs))
    else:
        kc = code_bytes(seed, S_KCACHE, (num_blocks, bs, kvh, hs), kv_quant)
        vc = code_bytes(seed, S_VCACHE, (num_blocks, bs, kvh, hs), kv_quant)
        # calibrated scales: a per-channel range of 2..4 (the draws are N(0, 1)) over the
        # largest code
        qm = KV_QMAX[kv_quant]
        k_scale = ((2.0 + 2.0 * uniform(seed, S_KSCALE, kvh * hs)) / qm).astype(np.float32).reshape(kvh, hs)
        v_scale = ((2.0 + 2.0 * uniform(seed, S_VSCALE, kvh * hs)) / qm).astype(np.float32).reshape(kvh, hs)

    slot = None
    if slot_mode == "explicit":
        # the pool layout this generator chose: logical position p of sequence b lives in
        # physical block block_table[b][p // bs] at row p % bs
        slot = np.empty(N, dtype=np.int32)
        for b in range(B):
            p = past[b] + np.arange(q_lens[b])
            slot[cum[b]: cum[b + 1]] = bt[b, p // bs].astype(np.int64) * bs + p % bs
        if drop_count:
            drop = permutation(seed, S_DROP, N)[:drop_count]
            slot[drop] = -1
    return Problem(
        name=name, dtype=dtype, num_heads=nh, kv_num_heads=kvh, head_size=hs, block_size=bs,
        num_blocks=num_blocks, past_seqlens=past.astype(np.int32), q_lens=q_lens.astype(np.int32),
        cumulative_sequence_length=cum, block_table=bt, query=query, key=key, value=value,
        key_cache=kc, value_cache=vc, slot_mapping=slot, scale=scale, seed=seed,
        kv_quant=kv_quant, k_scale=k_scale, v_scale=v_scale,
    )


# ---- the five workloads ------------------------------------------------------------

CONFIG_NAMES = {
    1: "tiny-correctness",
    2: "decode-b64",
    3: "causal-prefill-4x2048",
    4: "mixed-8x512-chunks+24-decode",
    5: "long-decode-b8-bs16",
}


def config(k: int) -> Problem:
    """Workload k (1..5) with seed 1000+k; see the recipe table in the design notes."""
    seed = 1000 + k
    if k == 1:
        return make_problem(
            name=CONFIG_NAMES[1], seed=seed, dtype="fp16", num_heads=4, kv_num_heads=2,
            head_size=64, block_size=16, past=[5, 20], q_lens=[3, 7], dist="uniform",
            num_blocks=16, max_blocks_per_sequence=8, table_fill="perm")
    if k == 2:
        past = uniform_int(seed, S_PAST, 64, 512, 4096)
        return make_problem(
            name=CONFIG_NAMES[2], seed=seed, dtype="fp16", num_heads=32, kv_num_heads=8,
            head_size=128, block_size=256, past=past, q_lens=np.ones(64, np.int64),
            max_blocks_per_sequence=(4096 + 1 + 255) // 256)
    if k == 3:
        return make_problem(
            name=CONFIG_NAMES[3], seed=seed, dtype="bf16", num_heads=32, kv_num_heads=8,
            head_size=128, block_size=256, past=np.zeros(4, np.int64),
            q_lens=np.full(4, 2048, np.int64))
    if k == 4:
        return _mixed(seed, CONFIG_NAMES[4], "fp16")
    if k == 5:
        past = uniform_int(seed, S_PAST, 8, 32768, 131072)
        return make_problem(
            name=CONFIG_NAMES[5], seed=seed, dtype="bf16", num_heads=32, kv_num_heads=8,
            head_size=128, block_size=16, past=past, q_lens=np.ones(8, np.int64),
            max_blocks_per_sequence=(131072 + 1 + 15) // 16)
    raise ValueError(f"no workload {k}")


def config_kv_quant(k: int, fmt: str) -> Problem:
    """Workload k's batch (same seed, lengths, pages and queries) with integer caches of
    format fmt ("int8" | "int4") and per-channel scales in place of the 16-bit caches: the
    decode batch (k = 2) or the mixed continuous batch (k = 4)."""
    seed = 1000 + k
    if k == 2:
        past = uniform_int(seed, S_PAST, 64, 512, 4096)
        return make_problem(
            name=f"{CONFIG_NAMES[2]}-{fmt}", seed=seed, dtype="fp16", num_heads=32, kv_num_heads=8,
            head_size=128, block_size=256, past=past, q_lens=np.ones(64, np.int64),
            max_blocks_per_sequence=(4096 + 1 + 255) // 256, kv_quant=fmt)
    if k == 4:
        return _mixed(seed, f"{CONFIG_NAMES[4]}-{fmt}", "fp16", kv_quant=fmt)
    raise ValueError("integer-cache variants exist for workloads 2 and 4")


def _mixed(seed, name, dtype, kv_quant=None):
    """The mixed continuous batch's recipe (8 chunks of 512 with past U[0, 8192] and 24 decode
    rows with past U[1024, 16384] in seeded order, packed rows, 10% of the slots -1)."""
    past_chunk = uniform_int(seed, S_PAST, 8, 0, 8192)
    past_dec = uniform_int(seed, S_QLEN, 24, 1024, 16384)
    past = np.concatenate([past_chunk, past_dec])
    q = np.concatenate([np.full(8, 512, np.int64), np.ones(24, np.int64)])
    order = permutation(seed, S_ORDER, 32)
    past, q = past[order], q[order]
    N = int(q.sum())
    return make_problem(
        name=name, seed=seed, dtype=dtype, num_heads=32, kv_num_heads=8,
        head_size=128, block_size=256, past=past, q_lens=q, packed=True,
        slot_mode="explicit", drop_count=N // 10,
        max_blocks_per_sequence=(16384 + 1 + 255) // 256, kv_quant=kv_quant)


# Further batches of the same recipes, for measurements of kernels the five workloads do not
# run: the causal prefill with an explicit slot_mapping (for bf16 the fp16 copy of V is then
# made by its own kernel after the cache write), and 256-wide heads (Qwen3.5's full-attention
# layers: 16 query and 2 KV heads of 256).
VARIANTS = ("causal-prefill-explicit-slots", "causal-prefill-hs256", "decode-b64-hs256")


def variant(name: str) -> Problem:
    if name == "causal-prefill-explicit-slots":
        return make_problem(
            name=name, seed=1104, dtype="bf16", num_heads=32, kv_num_heads=8, head_size=128, block_size=256,
            past=np.zeros(4, np.int64), q_lens=np.full(4, 2048, np.int64), slot_mode="explicit")
    if name == "causal-prefill-hs256":
        return make_problem(
            name=name, seed=1103, dtype="bf16", num_heads=16, kv_num_heads=2, head_size=256, block_size=256,
            past=np.zeros(4, np.int64), q_lens=np.full(4, 2048, np.int64))
    if name == "decode-b64-hs256":
        past = uniform_int(1102, S_PAST, 64, 512, 4096)
        return make_problem(
            name=name, seed=1102, dtype="fp16", num_heads=16, kv_num_heads=2, head_size=256, block_size=256,
            past=past, q_lens=np.ones(64, np.int64), max_blocks_per_sequence=(4096 + 1 + 255) // 256)
    raise ValueError(f"no variant {name}")
