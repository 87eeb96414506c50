"""Pins of the oracle's Q/K preparation (RMSNorm, then the rotary embedding) against
properties fixed by the mathematics, not by the oracle's own formula:

  - without a weight and with rotary_dim 0 the vectors pass through unchanged;
  - position 0 rotates by angle 0 (identity);
  - a rotation keeps the length of every rotated pair (u, u + d/2);
  - scores of rotated vectors depend on the positions only through their difference;
  - RMSNorm with unit weights leaves mean square ms / (ms + eps); a weight scales each
    component by itself;
  - a single nonzero component u moves only into u + d/2 ("rotate half" pairing), by the
    angle fl32(fl32(p) * fl32(base^(-2u/d))) (an fp32 rotary table), readable back with
    atan2; components from rotary_dim on are untouched.
"""
import numpy as np
import pytest

import oracle
import workloads as w
from helpers import bits_to_f64


def _problem(dtype="fp16", nh=4, kvh=2, hs=64, past=(0, 37), q=(5, 3), seed=5, packed=False):
    return w.make_problem(name="prep", seed=seed, dtype=dtype, num_heads=nh, kv_num_heads=kvh, head_size=hs,
                          block_size=16, past=list(past), q_lens=list(q), packed=packed)


def _inputs(p):
    N, nh, kvh, hs = p.num_tokens, p.num_heads, p.kv_num_heads, p.head_size
    if p.key is None:
        rows = bits_to_f64(p.query, p.dtype).reshape(N, -1)
        return rows[:, :nh * hs].reshape(N, nh, hs), rows[:, nh * hs:(nh + kvh) * hs].reshape(N, kvh, hs)
    return bits_to_f64(p.query, p.dtype).reshape(N, nh, hs), bits_to_f64(p.key, p.dtype).reshape(N, kvh, hs)


def _positions(p):
    pos = []
    for b in range(p.batch_size):
        pos += [int(p.past_seqlens[b]) + j for j in range(int(p.q_lens[b]))]
    return np.array(pos)


def test_no_norm_no_rotation_is_identity():
    for packed in (False, True):
        p = _problem(packed=packed)
        q, k = _inputs(p)
        oq, ok = oracle.qk_prep_f64(p, dict(rotary_dim=0))
        assert np.array_equal(oq, q) and np.array_equal(ok, k)


def test_position_zero_is_identity():
    p = _problem(past=(0,), q=(1,))
    q, k = _inputs(p)
    oq, ok = oracle.qk_prep_f64(p, dict(rotary_dim=64, theta=10000.0))
    assert np.array_equal(oq, q) and np.array_equal(ok, k)


@pytest.mark.parametrize("d", [64, 32])
def test_rotation_keeps_every_pair_length(d):
    p = _problem(past=(100, 5000), q=(4, 2))
    q, k = _inputs(p)
    oq, ok = oracle.qk_prep_f64(p, dict(rotary_dim=d, theta=500000.0))
    for x, y in ((q, oq), (k, ok)):
        before = x[..., :d // 2] ** 2 + x[..., d // 2:d] ** 2
        after = y[..., :d // 2] ** 2 + y[..., d // 2:d] ** 2
        assert np.allclose(after, before, rtol=1e-12, atol=1e-14)
        assert np.array_equal(y[..., d:], x[..., d:])  # past rotary_dim: untouched


def test_scores_depend_on_the_position_difference_only():
    # one sequence whose rows all carry the same q and k: rotated at positions 0..L-1,
    # <R(q, m), R(k, n)> is a function of m - n
    L = 12
    p = _problem(past=(0,), q=(L,), nh=2, kvh=1, hs=32)
    p.query = np.tile(p.query[:1], (L, 1))
    p.key = np.tile(p.key[:1], (L, 1))
    oq, ok = oracle.qk_prep_f64(p, dict(rotary_dim=32, theta=100.0))
    s = np.einsum("mc,nc->mn", oq[:, 0], ok[:, 0])
    for diff in range(-3, 4):
        vals = [s[m, m - diff] for m in range(L) if 0 <= m - diff < L]
        assert np.ptp(vals) <= 1e-5 * max(1.0, np.abs(vals).max())
    assert np.ptp([s[m, m] for m in range(L)]) <= 1e-5  # and they do change with it
    assert abs(s[5, 2] - s[5, 5]) > 1e-3


def test_rms_norm_with_unit_and_general_weights():
    p = _problem(hs=64)
    q, k = _inputs(p)
    hs = 64
    ones = oracle.double_to_f16(np.ones(hs))
    eps = 1e-3
    oq, ok = oracle.qk_prep_f64(p, dict(q_norm_weight=ones, k_norm_weight=ones, eps=eps, rotary_dim=0))
    ms = (q ** 2).mean(-1)
    assert np.allclose((oq ** 2).mean(-1), ms / (ms + eps), rtol=1e-12)
    wts = oracle.double_to_f16(np.linspace(0.5, 2.0, hs))
    oq2, ok2 = oracle.qk_prep_f64(p, dict(q_norm_weight=wts, k_norm_weight=None, eps=eps, rotary_dim=0))
    assert np.allclose(oq2, oq * oracle.f16_to_double(wts), rtol=1e-12, atol=1e-15)
    assert np.array_equal(ok2, k)  # no K weight: K untouched


@pytest.mark.parametrize("u", [0, 1, 7])
def test_single_component_rotates_into_its_half_partner(u):
    d, hs, base = 32, 32, 10000.0
    p = _problem(past=(0, 100003), q=(1, 2), nh=1, kvh=1, hs=hs)
    one = np.zeros(hs)
    one[u] = 1.0
    bits = oracle.double_to_f16(one)
    p.query = np.tile(bits, (p.num_tokens, 1))
    p.key = np.tile(bits, (p.num_tokens, 1))
    oq, _ = oracle.qk_prep_f64(p, dict(rotary_dim=d, theta=base))
    for i, pos in enumerate(_positions(p)):
        y = oq[i, 0]
        nz = set(np.flatnonzero(np.abs(y) > 1e-15)) - {u, u + d // 2}
        assert not nz
        freq = np.float32(base ** (-2.0 * u / d))
        want = np.float32(np.float32(pos) * freq)  # the fp32 rotary table
        got = np.arctan2(y[u + d // 2], y[u])
        assert abs(np.angle(np.exp(1j * (got - float(want))))) < 1e-9  # (fp64 atan2 of an angle near 1e5)
        assert abs(np.hypot(y[u], y[u + d // 2]) - 1.0) < 1e-14


def test_operator_with_preparation_is_the_operator_on_prepared_rows():
    p = _problem(dtype="bf16", packed=True)
    prep = dict(q_norm_weight=oracle.double_to_bf16(np.linspace(0.8, 1.2, 64)), k_norm_weight=None, eps=1e-6,
                rotary_dim=64, theta=1000.0)
    a = oracle.paged_attention(p, prep=prep)
    b = oracle.paged_attention(oracle.apply_qk_prep(p, prep))
    assert np.array_equal(a["out_bits"], b["out_bits"]) and np.array_equal(a["key_cache"], b["key_cache"])


# ---- the output gate: out * sigmoid(gate) ----

def _gated(dtype, gate_value):
    p = _problem(dtype=dtype)
    base = oracle.paged_attention(p)
    N, nh, hs = p.num_tokens, p.num_heads, p.head_size
    g = np.full((N, nh * hs), gate_value)
    gb = oracle.double_to_bf16(g) if dtype == "bf16" else oracle.double_to_f16(g)
    return base, oracle.paged_attention(p, gate=gb.reshape(N, nh * hs))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_gate_closed_forms(dtype):
    base, open_ = _gated(dtype, 40.0)        # sigmoid(40) = 1 - 4e-18: the ungated output
    assert np.array_equal(open_["out_bits"], base["out_bits"])
    base, half = _gated(dtype, 0.0)          # sigmoid(0) = 1/2 exactly
    assert np.array_equal(half["out"], base["out"] / 2)
    assert np.array_equal(half["lse"], base["lse"])  # the gate does not touch lse
    _, shut = _gated(dtype, -60.0)           # sigmoid(-60) ~ 9e-27: zero in T
    assert np.all(np.abs(shut["out"]) < 1e-20)


def test_gate_symmetry():
    # sigmoid(g) + sigmoid(-g) = 1: the two gated outputs add up to the ungated one
    p = _problem(dtype="fp16")
    N, nh, hs = p.num_tokens, p.num_heads, p.head_size
    g = np.linspace(-6, 6, N * nh * hs).reshape(N, nh * hs)
    plus = oracle.paged_attention(p, gate=oracle.double_to_f16(g).reshape(N, -1))
    minus = oracle.paged_attention(p, gate=oracle.double_to_f16(-g).reshape(N, -1))
    base = oracle.paged_attention(p)
    assert np.allclose(plus["out"] + minus["out"], base["out"], rtol=1e-12, atol=1e-15)
