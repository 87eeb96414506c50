"""Pins for the oracle: checks against things other than the oracle itself.

- the 16-bit conversions against numpy / torch and hand-derived ties;
- attention against torch's float64 scaled_dot_product_attention (a library routine)
  on logical K/V built without the oracle's gather;
- closed forms: one key returns its own v and lse = s; equal scores give the mean;
  constant V returns V; a dominant key returns its v;
- a hand-derived slot table (tests/golden/slots_tiny.json);
- invariants of the operator: physical page relabeling, packed [Q|K|V] == separate,
  per-sequence runs == packed batch, MHA with repeated heads == GQA, scale 0 ==
  1/sqrt(head_size), causality, -1 slots, explicit slots == derived slots.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as w
from helpers import bits_to_f64, f64_to_bits, from_logical, rand_bits, sdpa_reference

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- conversions ---------------------------------------------------------------------

def test_f16_decode_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decode_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_double(bits)
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
        rng.uniform(-70000, 70000, 2000),
        # exact ties halfway between neighbouring fp16 values, and their neighbours
        (np.arange(2048) + 0.5) * 2.0 ** -10, (np.arange(2048) + 0.5) * 2.0 ** -24,
        np.nextafter((np.arange(512) + 0.5) * 2.0 ** -10, 0), np.nextafter((np.arange(512) + 0.5) * 2.0 ** -10, 9),
        [65504.0, 65519.99, 65520.0, 1e-8, 2.0 ** -25, np.nextafter(2.0 ** -25, 1), 0.0, -0.0],
    ])
    got = oracle.double_to_f16(x)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rounding_matches_torch_and_hand_ties():
    rng = np.random.default_rng(8)
    x32 = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    got = oracle.double_to_bf16(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    # hand ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0 = 0x3F80);
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6 -> even (0x3F82);
    # 1 + 2^-8 + 2^-40 is just above the tie -> 0x3F81 (rounding through float32 would give 0x3F80)
    cases = {1 + 2.0 ** -8: 0x3F80, 1 + 3 * 2.0 ** -8: 0x3F82, 1 + 2.0 ** -8 + 2.0 ** -40: 0x3F81,
             -(1 + 2.0 ** -8 + 2.0 ** -40): 0xBF81, 3.0e38: 0x7F62, 3.4e38: 0x7F80}
    for v, b in cases.items():
        assert oracle.double_to_bf16([v])[0] == b, (v, hex(oracle.double_to_bf16([v])[0]), hex(b))


# ---- against torch's float64 SDPA ----------------------------------------------------

def _scale(hs, scale):
    return 1.0 / math.sqrt(hs) if scale == 0.0 else float(np.float32(scale))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("nh,kvh,hs,bs", [(4, 2, 64, 16), (6, 2, 32, 8), (2, 2, 16, 4)])
def test_prefill_from_empty_matches_sdpa_causal(dtype, nh, kvh, hs, bs):
    rng = np.random.default_rng(100 + nh + hs)
    prob, logical = from_logical(rng, dtype, nh, kvh, hs, bs, past=[0, 0], q_lens=[13, 5])
    r = oracle.paged_attention(prob)
    cum = prob.cumulative_sequence_length
    for b in range(2):
        ref = sdpa_reference(logical[b], nh, kvh, _scale(hs, 0.0), "causal")
        np.testing.assert_allclose(r["out"][cum[b]:cum[b + 1]], ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_decode_matches_sdpa_without_mask(dtype):
    rng = np.random.default_rng(11)
    nh, kvh, hs, bs = 8, 2, 64, 16
    past = [0, 1, 15, 16, 17, 40]
    prob, logical = from_logical(rng, dtype, nh, kvh, hs, bs, past=past, q_lens=[1] * 6, scale=0.3)
    r = oracle.paged_attention(prob)
    for b in range(6):
        ref = sdpa_reference(logical[b], nh, kvh, _scale(hs, 0.3), "nomask")
        np.testing.assert_allclose(r["out"][b:b + 1], ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_chunked_prefill_matches_sdpa_bottom_right_mask(dtype):
    rng = np.random.default_rng(12)
    nh, kvh, hs, bs = 4, 1, 32, 8
    past, q = [5, 0, 17, 31], [9, 3, 1, 20]
    prob, logical = from_logical(rng, dtype, nh, kvh, hs, bs, past=past, q_lens=q, scale=-0.2)
    r = oracle.paged_attention(prob)
    cum = prob.cumulative_sequence_length
    for b in range(4):
        ref = sdpa_reference(logical[b], nh, kvh, _scale(hs, -0.2), "mask")
        np.testing.assert_allclose(r["out"][cum[b]:cum[b + 1]], ref, rtol=1e-12, atol=1e-13)


def test_js_example_shapes_run_and_match_sdpa():
    spec = json.load(open(os.path.join(GOLDEN, "js_example_shapes.json")))
    nh, kvh = spec["num_heads"], spec["kv_num_heads"]
    hs = spec["query"][1] // nh
    nblk, bs = spec["key_cache"][0], spec["key_cache"][1]
    for past in (0, 3):
        rng = np.random.default_rng(past)
        prob, logical = from_logical(rng, "fp16", nh, kvh, hs, bs, past=[past], q_lens=[spec["query"][0]],
                                     extra_blocks=0)
        # pad the pool and the table to the example's shapes
        extra = nblk - prob.num_blocks
        prob.key_cache = np.concatenate([prob.key_cache, rand_bits(rng, (extra, bs, kvh, hs), "fp16")])
        prob.value_cache = np.concatenate([prob.value_cache, rand_bits(rng, (extra, bs, kvh, hs), "fp16")])
        prob.num_blocks = nblk
        bt = np.full((1, spec["block_table"][1]), -1, np.int32)
        bt[0, :prob.block_table.shape[1]] = prob.block_table[0]
        prob.block_table = bt
        assert list(prob.query.shape) == spec["query"] and list(prob.key.shape) == spec["key"]
        assert list(prob.key_cache.shape) == spec["key_cache"]
        r = oracle.paged_attention(prob)
        ref = sdpa_reference(logical[0], nh, kvh, _scale(hs, 0.0), "mask")
        np.testing.assert_allclose(r["out"], ref, rtol=1e-12, atol=1e-13)


# ---- closed forms ----------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_single_token_no_past_returns_its_own_v(dtype):
    rng = np.random.default_rng(3)
    nh, kvh, hs = 4, 2, 64
    prob, _ = from_logical(rng, dtype, nh, kvh, hs, 16, past=[0, 0, 0], q_lens=[1, 1, 1])
    r = oracle.paged_attention(prob)
    G = nh // kvh
    for i in range(3):
        q = bits_to_f64(prob.query[i], dtype).reshape(nh, hs)
        k = bits_to_f64(prob.key[i], dtype).reshape(kvh, hs)
        for h in range(nh):
            v_bits = prob.value[i].reshape(kvh, hs)[h // G]
            assert np.array_equal(r["out_bits"][i].reshape(nh, hs)[h], v_bits)
            s = float(np.dot(q[h], k[h // G])) / math.sqrt(hs)
            assert abs(r["lse"][i, h] - s) <= 1e-15 * max(1.0, abs(s))


def _two_key_problem(dtype, k1_scale, v0, v1, scale):
    """past = 1 (one cached key k0 = 0), one new token with k1 = k1_scale * e_0 and query e_0."""
    hs, bs = 16, 4
    kc = np.zeros((2, bs, 1, hs), np.uint16)
    vc = np.zeros((2, bs, 1, hs), np.uint16)
    vc[1, 0, 0] = f64_to_bits(v0, dtype)                 # logical key 0 lives in physical block 1
    q = np.zeros((1, hs)); q[0, 0] = 1.0
    k = np.zeros((1, hs)); k[0, 0] = k1_scale
    return w.Problem(
        name="two-key", dtype=dtype, num_heads=1, kv_num_heads=1, head_size=hs, block_size=bs,
        num_blocks=2, past_seqlens=np.array([1], np.int32), q_lens=np.array([1], np.int32),
        cumulative_sequence_length=np.array([0, 1], np.int32), block_table=np.array([[1]], np.int32),
        query=f64_to_bits(q, dtype), key=f64_to_bits(k, dtype), value=f64_to_bits(v1[None, :], dtype),
        key_cache=kc, value_cache=vc, slot_mapping=None, scale=scale)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_two_keys_closed_forms(dtype):
    rng = np.random.default_rng(5)
    v0 = bits_to_f64(rand_bits(rng, 16, dtype), dtype)
    v1 = bits_to_f64(rand_bits(rng, 16, dtype), dtype)
    # equal scores (k1 = 0 = k0): weights 1/2, 1/2; lse = ln 2
    r = oracle.paged_attention(_two_key_problem(dtype, 0.0, v0, v1, 0.5))
    np.testing.assert_allclose(r["out"][0, 0], (v0 + v1) / 2, rtol=0, atol=1e-15)
    assert abs(r["lse"][0, 0] - math.log(2.0)) < 1e-15
    # scores 0 and ln 2 (scale = float32(ln 2), q.k1 = 1): weights 1/3, 2/3 up to float32(ln 2)'s error
    r = oracle.paged_attention(_two_key_problem(dtype, 1.0, v0, v1, float(np.float32(math.log(2.0)))))
    np.testing.assert_allclose(r["out"][0, 0], (v0 + 2 * v1) / 3, rtol=0, atol=1e-7)
    assert abs(r["lse"][0, 0] - math.log(3.0)) < 1e-7
    # a dominant key (score gap 64): the output is that key's v
    r = oracle.paged_attention(_two_key_problem(dtype, 8.0, v0, v1, 8.0))
    np.testing.assert_allclose(r["out"][0, 0], v1, rtol=0, atol=1e-27)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_constant_v_returns_v(dtype):
    rng = np.random.default_rng(6)
    nh, kvh, hs, bs = 4, 2, 32, 8
    prob, _ = from_logical(rng, dtype, nh, kvh, hs, bs, past=[0, 7, 30], q_lens=[5, 1, 9])
    c = rand_bits(rng, (kvh, hs), dtype)
    prob.value_cache[:] = c[None, None]
    prob.value[:] = c.reshape(1, -1)
    r = oracle.paged_attention(prob)
    expect = np.repeat(c, nh // kvh, axis=0).reshape(-1)
    assert np.array_equal(r["out_bits"], np.broadcast_to(expect, r["out_bits"].shape))


# ---- the cache write --------------------------------------------------------------------

def test_slot_golden_table():
    g = json.load(open(os.path.join(GOLDEN, "slots_tiny.json")))
    bs, nblk = g["block_size"], g["num_blocks"]
    kvh, hs = 1, 8
    rng = np.random.default_rng(9)
    N = sum(g["q_lens"])
    prob = w.Problem(
        name="slots", dtype="fp16", num_heads=1, kv_num_heads=kvh, head_size=hs, block_size=bs,
        num_blocks=nblk, past_seqlens=np.array(g["past_seqlens"], np.int32),
        q_lens=np.array(g["q_lens"], np.int32),
        cumulative_sequence_length=np.concatenate([[0], np.cumsum(g["q_lens"])]).astype(np.int32),
        block_table=np.array(g["block_table"], np.int32), query=rand_bits(rng, (N, hs), "fp16"),
        key=rand_bits(rng, (N, hs), "fp16"), value=rand_bits(rng, (N, hs), "fp16"),
        key_cache=rand_bits(rng, (nblk, bs, kvh, hs), "fp16"), value_cache=rand_bits(rng, (nblk, bs, kvh, hs), "fp16"),
        slot_mapping=None)
    kc, vc = oracle.scatter(prob)
    ek, ev = prob.key_cache.reshape(-1, hs).copy(), prob.value_cache.reshape(-1, hs).copy()
    for i, s in enumerate(g["expected_slots"]):
        ek[s] = prob.key[i]
        ev[s] = prob.value[i]
    assert np.array_equal(kc.reshape(-1, hs), ek)
    assert np.array_equal(vc.reshape(-1, hs), ev)
    # and the same slots given explicitly
    prob.slot_mapping = np.array(g["expected_slots"], np.int32)
    kc2, vc2 = oracle.scatter(prob)
    assert np.array_equal(kc2, kc) and np.array_equal(vc2, vc)


def test_minus_one_slots_leave_cache_untouched_and_reads_use_cache():
    rng = np.random.default_rng(10)
    nh, kvh, hs, bs = 2, 1, 16, 4
    prob, _ = from_logical(rng, "fp16", nh, kvh, hs, bs, past=[0, 3], q_lens=[1, 2])
    # explicit slots: the layout's slots, with token 0 suppressed
    slots = []
    for b in range(2):
        for j in range(int(prob.q_lens[b])):
            p = int(prob.past_seqlens[b]) + j
            slots.append(int(prob.block_table[b, p // bs]) * bs + p % bs)
    sm = np.array(slots, np.int32)
    sm[0] = -1
    prob.slot_mapping = sm
    r = oracle.paged_attention(prob)
    kc0, vc0 = prob.key_cache.reshape(-1, kvh * hs), prob.value_cache.reshape(-1, kvh * hs)
    kc1, vc1 = r["key_cache"].reshape(-1, kvh * hs), r["value_cache"].reshape(-1, kvh * hs)
    assert np.array_equal(kc1[slots[0]], kc0[slots[0]]) and np.array_equal(vc1[slots[0]], vc0[slots[0]])
    for i in (1, 2):
        assert np.array_equal(kc1[slots[i]], prob.key[i]) and np.array_equal(vc1[slots[i]], prob.value[i])
    untouched = np.setdiff1d(np.arange(kc0.shape[0]), slots[1:])
    assert np.array_equal(kc1[untouched], kc0[untouched]) and np.array_equal(vc1[untouched], vc0[untouched])
    # token 0 (past 0, one key) reads its logical position back from the cache: the stale v there
    assert np.array_equal(r["out_bits"][0].reshape(nh, hs)[0], vc0[slots[0]].reshape(kvh, hs)[0])


def test_invalid_slots_are_rejected():
    rng = np.random.default_rng(13)
    prob, _ = from_logical(rng, "fp16", 2, 1, 16, 4, past=[0], q_lens=[2])
    prob.slot_mapping = np.array([3, 3], np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.scatter(prob)
    prob.slot_mapping = np.array([0, prob.num_blocks * 4], np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.scatter(prob)


# ---- invariants -------------------------------------------------------------------------

def test_physical_page_relabeling_is_invisible():
    rng = np.random.default_rng(14)
    prob, _ = from_logical(rng, "bf16", 4, 2, 32, 8, past=[3, 20, 0], q_lens=[4, 1, 11], extra_blocks=5)
    r0 = oracle.paged_attention(prob)
    perm = rng.permutation(prob.num_blocks)            # old block x moves to perm[x]
    p2 = prob.copy()
    p2.key_cache = np.empty_like(prob.key_cache)
    p2.value_cache = np.empty_like(prob.value_cache)
    p2.key_cache[perm] = prob.key_cache
    p2.value_cache[perm] = prob.value_cache
    p2.block_table = np.where(prob.block_table >= 0, perm[np.maximum(prob.block_table, 0)], -1).astype(np.int32)
    r1 = oracle.paged_attention(p2)
    assert np.array_equal(r0["out"], r1["out"]) and np.array_equal(r0["lse"], r1["lse"])
    assert np.array_equal(r1["key_cache"][perm], r0["key_cache"])


def test_packed_qkv_equals_separate():
    rng = np.random.default_rng(15)
    prob, _ = from_logical(rng, "fp16", 4, 2, 32, 8, past=[3, 9], q_lens=[5, 2])
    r0 = oracle.paged_attention(prob)
    p2 = prob.copy()
    p2.query = np.concatenate([prob.query, prob.key, prob.value], axis=1)
    p2.key = p2.value = None
    r1 = oracle.paged_attention(p2)
    for k in ("out", "lse", "key_cache", "value_cache"):
        assert np.array_equal(r0[k], r1[k]), k


def test_packed_batch_equals_per_sequence_runs():
    rng = np.random.default_rng(16)
    prob, _ = from_logical(rng, "bf16", 4, 1, 32, 8, past=[0, 13, 6], q_lens=[7, 1, 3])
    r = oracle.paged_attention(prob)
    cum = prob.cumulative_sequence_length
    for b in range(3):
        p1 = prob.copy()
        sl = slice(cum[b], cum[b + 1])
        p1.past_seqlens = prob.past_seqlens[b:b + 1]
        p1.q_lens = prob.q_lens[b:b + 1]
        p1.cumulative_sequence_length = np.array([0, cum[b + 1] - cum[b]], np.int32)
        p1.block_table = prob.block_table[b:b + 1]
        p1.query, p1.key, p1.value = prob.query[sl], prob.key[sl], prob.value[sl]
        r1 = oracle.paged_attention(p1)
        assert np.array_equal(r1["out"], r["out"][sl]) and np.array_equal(r1["lse"], r["lse"][sl])


def test_gqa_equals_mha_with_repeated_kv_heads():
    rng = np.random.default_rng(17)
    nh, kvh, hs = 6, 2, 16
    G = nh // kvh
    prob, _ = from_logical(rng, "fp16", nh, kvh, hs, 4, past=[2, 9], q_lens=[3, 4])
    r0 = oracle.paged_attention(prob)
    p2 = prob.copy()
    p2.kv_num_heads = nh
    p2.key_cache = np.repeat(prob.key_cache, G, axis=2)
    p2.value_cache = np.repeat(prob.value_cache, G, axis=2)
    p2.key = np.repeat(prob.key.reshape(-1, kvh, hs), G, axis=1).reshape(-1, nh * hs)
    p2.value = np.repeat(prob.value.reshape(-1, kvh, hs), G, axis=1).reshape(-1, nh * hs)
    r1 = oracle.paged_attention(p2)
    assert np.array_equal(r0["out"], r1["out"])


def test_scale_zero_means_inverse_sqrt_head_size():
    rng = np.random.default_rng(18)
    prob, _ = from_logical(rng, "fp16", 2, 1, 64, 8, past=[4], q_lens=[3])
    r0 = oracle.paged_attention(prob)
    p2 = prob.copy()
    p2.scale = 0.125
    r1 = oracle.paged_attention(p2)
    assert np.array_equal(r0["out"], r1["out"])


def test_causality_future_tokens_do_not_change_earlier_rows():
    rng = np.random.default_rng(19)
    prob, _ = from_logical(rng, "fp16", 2, 1, 16, 4, past=[5], q_lens=[6])
    r0 = oracle.paged_attention(prob)
    p2 = prob.copy()
    p2.key[3:] = rand_bits(rng, p2.key[3:].shape, "fp16")
    p2.value[3:] = rand_bits(rng, p2.value[3:].shape, "fp16")
    p2.query[3:] = rand_bits(rng, p2.query[3:].shape, "fp16")
    r1 = oracle.paged_attention(p2)
    assert np.array_equal(r0["out"][:3], r1["out"][:3])
    assert not np.array_equal(r0["out"][3:], r1["out"][3:])


def test_rows_entry_point_equals_full_attention():
    rng = np.random.default_rng(20)
    prob, _ = from_logical(rng, "bf16", 4, 2, 32, 8, past=[0, 11], q_lens=[6, 3])
    r = oracle.paged_attention(prob)
    toks = np.array([0, 5, 6, 8, 8], np.int32)
    heads = np.array([0, 3, 1, 2, 0], np.int32)
    out, lse = oracle.attention_rows(prob, r["key_cache"], r["value_cache"], toks, heads)
    assert np.array_equal(out, r["out"][toks, heads]) and np.array_equal(lse, r["lse"][toks, heads])


def test_explicit_layout_slots_equal_derived_on_generated_workload():
    p = w.config(1)
    p2 = w.make_problem(name="t", seed=p.seed, dtype="fp16", num_heads=4, kv_num_heads=2, head_size=64,
                        block_size=16, past=[5, 20], q_lens=[3, 7], dist="uniform", num_blocks=16,
                        max_blocks_per_sequence=8, table_fill="perm", slot_mode="explicit")
    r0 = oracle.paged_attention(p)
    r1 = oracle.paged_attention(p2)
    for k in ("out", "key_cache", "value_cache"):
        assert np.array_equal(r0[k], r1[k]), k
