"""Test-side constructions that do not go through the oracle.

``from_logical`` builds an invocation from per-sequence *logical* K/V histories by
placing whole pages into a shuffled pool. It is the inverse of the read path (a page
copy per logical block), written independently of the oracle's per-key gather, so the
oracle can be checked against attention computed directly on the logical sequences.
"""
from __future__ import annotations

import numpy as np
import torch

import workloads as w


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Values already representable in the 16-bit type -> their bit patterns."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "fp16":
        b = x.astype(np.float16)
        assert np.array_equal(b.astype(np.float64), x)
        return b.view(np.uint16)
    f = x.astype(np.float32)
    assert np.array_equal(f.astype(np.float64), x)
    u = f.view(np.uint32)
    assert not np.any(u & 0xFFFF)
    return (u >> 16).astype(np.uint16)


def rand_bits(rng: np.random.Generator, shape, dtype: str, lo=-1.0, hi=1.0) -> np.ndarray:
    """Random values already rounded to the 16-bit type (test-local; numpy RNG)."""
    x = rng.uniform(lo, hi, size=shape)
    if dtype == "fp16":
        return x.astype(np.float16).view(np.uint16)
    return (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def from_logical(
    rng: np.random.Generator,
    dtype: str,
    nh: int,
    kvh: int,
    hs: int,
    bs: int,
    past,
    q_lens,
    extra_blocks: int = 3,
    scale: float = 0.0,
):
    """Returns (problem, logical) where logical[b] = dict(q, k, v) in float64 with
    q: (q_len, nh, hs), k/v: (past+q_len, kvh, hs) = history followed by the new rows."""
    past = [int(x) for x in past]
    q_lens = [int(x) for x in q_lens]
    B = len(past)
    pages = [(p + q + bs - 1) // bs for p, q in zip(past, q_lens)]
    num_blocks = sum(pages) + extra_blocks
    maxb = max(max(pages), 1)
    perm = rng.permutation(num_blocks)
    bt = np.full((B, maxb), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        bt[b, : pages[b]] = perm[pos: pos + pages[b]]
        pos += pages[b]
    kc = rand_bits(rng, (num_blocks, bs, kvh, hs), dtype)
    vc = rand_bits(rng, (num_blocks, bs, kvh, hs), dtype)
    N = sum(q_lens)
    query = rand_bits(rng, (N, nh * hs), dtype)
    key = rand_bits(rng, (N, kvh * hs), dtype)
    value = rand_bits(rng, (N, kvh * hs), dtype)
    cum = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    logical = []
    for b in range(B):
        L = past[b] + q_lens[b]
        hk = np.empty((pages[b] * bs, kvh, hs), dtype=np.uint16)
        hv = np.empty_like(hk)
        for pg in range(pages[b]):  # page copy: logical block pg lives in physical block bt[b, pg]
            hk[pg * bs:(pg + 1) * bs] = kc[bt[b, pg]]
            hv[pg * bs:(pg + 1) * bs] = vc[bt[b, pg]]
        k = hk[:L].copy()
        v = hv[:L].copy()
        k[past[b]:L] = key[cum[b]:cum[b + 1]].reshape(-1, kvh, hs)
        v[past[b]:L] = value[cum[b]:cum[b + 1]].reshape(-1, kvh, hs)
        logical.append(dict(
            q=bits_to_f64(query[cum[b]:cum[b + 1]], dtype).reshape(-1, nh, hs),
            k=bits_to_f64(k, dtype), v=bits_to_f64(v, dtype), past=past[b]))
    prob = w.Problem(
        name="from-logical", dtype=dtype, num_heads=nh, kv_num_heads=kvh, head_size=hs,
        block_size=bs, num_blocks=num_blocks, past_seqlens=np.array(past, np.int32),
        q_lens=np.array(q_lens, np.int32), cumulative_sequence_length=cum, block_table=bt,
        query=query, key=key, value=value, key_cache=kc, value_cache=vc, slot_mapping=None,
        scale=scale)
    return prob, logical


def sdpa_reference(logical_b: dict, nh: int, kvh: int, scale_used: float, mode: str) -> np.ndarray:
    """torch CPU float64 scaled_dot_product_attention on one sequence's logical K/V.
    mode: "causal" (is_causal=True, needs past == 0), "nomask" (q_len == 1 sees all keys),
    "mask" (explicit boolean bottom-right mask). Returns (q_len, nh, hs)."""
    q = torch.from_numpy(logical_b["q"]).permute(1, 0, 2)          # (nh, q, hs)
    G = nh // kvh
    k = torch.from_numpy(logical_b["k"]).permute(1, 0, 2).repeat_interleave(G, dim=0)
    v = torch.from_numpy(logical_b["v"]).permute(1, 0, 2).repeat_interleave(G, dim=0)
    F = torch.nn.functional
    if mode == "causal":
        o = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=scale_used)
    elif mode == "nomask":
        o = F.scaled_dot_product_attention(q, k, v, scale=scale_used)
    else:
        ql, L = q.shape[1], k.shape[1]
        past = logical_b["past"]
        mask = torch.arange(L)[None, :] <= (past + torch.arange(ql))[:, None]
        o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale_used)
    return o.permute(1, 0, 2).numpy()
