"""The Q/K preparation before the cache write (pa_paged_attention_ex with a pa_qk_prep)
against the oracle's (oracle_qk_prep, pinned in test_oracle_prep_pins.py).

The kernel prepares in fp32 (sincosf of the same fp32 rotary angle the oracle uses), the
oracle in fp64, both rounding the prepared values once to T; so a prepared key in the
cache may sit one unit in the last place of T from the oracle's. Everything else in the
caches must match bit for bit (V rows, and every slot this call does not write), and the
outputs and lse must meet the usual tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
import varlen_paged_kv_gb300 as pa
import workloads as w
from gpu_utils import ATOL, RTOL, TORCH_DT, assert_close, bits_of, upload
from helpers import bits_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is required for the gpu tests")
    from varlen_paged_kv_gb300 import build
    build.build()


def _weights(p, lo, hi):
    x = np.linspace(lo, hi, p.head_size)
    return oracle.double_to_bf16(x) if p.dtype == "bf16" else oracle.double_to_f16(x)


def run(p, prep_bits, **opts):
    d = upload(p)
    dev = lambda b: None if b is None else torch.from_numpy(b.view(np.int16)).cuda().view(TORCH_DT[p.dtype])
    prep = dict(q_norm_weight=dev(prep_bits.get("q_norm_weight")), k_norm_weight=dev(prep_bits.get("k_norm_weight")),
                eps=prep_bits.get("eps", 1e-6), rotary_dim=prep_bits.get("rotary_dim", 0),
                theta=prep_bits.get("theta", 10000.0))
    lse = torch.empty((p.num_tokens, p.num_heads), dtype=torch.float32, device="cuda")
    ws = torch.zeros(pa.workspace_size(pa.make_dims(p.num_tokens, p.batch_size, p.head_size, p.num_blocks,
                                                    p.block_size, p.max_blocks_per_sequence, TORCH_DT[p.dtype],
                                                    opts.get("decode_split_keys", 0), opts.get("route", 0),
                                                    qk_prep=True), p.num_heads, p.kv_num_heads),
                     dtype=torch.uint8, device="cuda")
    out = pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                             d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], d["slot_mapping"],
                             num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, scale=p.scale, workspace=ws,
                             lse=lse, qk_prep=prep, **opts)
    assert pa.read_device_error(ws) == 0
    return d, out, lse


def check(p, prep_bits, **opts):
    ref = oracle.paged_attention(p, prep=prep_bits)
    d, out, lse = run(p, prep_bits, **opts)
    vc = bits_of(d["value_cache"])
    assert np.array_equal(vc, ref["value_cache"]), "value cache differs"
    kc = bits_of(d["key_cache"])
    diff = kc != ref["key_cache"]
    if diff.any():  # prepared keys: within one unit in the last place of T
        g, r = bits_to_f64(kc[diff], p.dtype), bits_to_f64(ref["key_cache"][diff], p.dtype)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(r), 1e-30))) - (7 if p.dtype == "bf16" else 10))
        ulp = np.maximum(ulp, 2.0 ** (-133 if p.dtype == "bf16" else -24))  # the subnormal spacing
        assert np.all(np.abs(g - r) <= ulp * 1.0000001), "a prepared key is more than one ulp off"
        assert diff.mean() < 0.01, f"{diff.mean():.3%} of the key cache differs"
    N, nh, hs = p.num_tokens, p.num_heads, p.head_size
    assert_close(bits_of(out).reshape(N, nh, hs), ref["out"], p.dtype, p.name)
    lg = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lg - ref["lse"]) <= 5e-4 + 1e-5 * np.abs(ref["lse"])), "lse differs"


def test_decode_norm_and_full_rotary():
    p = w.make_problem(name="prep-decode", seed=51, dtype="fp16", num_heads=32, kv_num_heads=8, head_size=128,
                       block_size=64, past=[3000, 17, 600, 1], q_lens=[1, 2, 1, 4])
    check(p, dict(q_norm_weight=_weights(p, 0.5, 1.5), k_norm_weight=_weights(p, 1.2, 0.8), eps=1e-6,
                  rotary_dim=128, theta=1e6))
    check(p, dict(q_norm_weight=None, k_norm_weight=None, rotary_dim=128, theta=1e4), decode_split_keys=64)


def test_prefill_bf16_partial_rotary_with_the_fp16_v_copy():
    p = w.make_problem(name="prep-prefill", seed=52, dtype="bf16", num_heads=16, kv_num_heads=4, head_size=128,
                       block_size=256, past=[0, 300], q_lens=[300, 129])
    check(p, dict(q_norm_weight=_weights(p, 0.9, 1.1), k_norm_weight=_weights(p, 0.9, 1.1), eps=1e-5,
                  rotary_dim=64, theta=1e4))


def test_packed_rows_with_dropped_slots():
    # a dropped token's K is not written, but its prepared Q still attends
    p = w.make_problem(name="prep-packed", seed=53, dtype="fp16", num_heads=32, kv_num_heads=8, head_size=128,
                       block_size=256, past=[0, 900, 50, 3000], q_lens=[130, 1, 40, 2], packed=True,
                       slot_mode="explicit", drop_count=9)
    check(p, dict(q_norm_weight=_weights(p, 0.7, 1.3), k_norm_weight=None, eps=1e-6, rotary_dim=96, theta=5e5))


@pytest.mark.parametrize("route", [pa.ROUTE_AUTO, pa.ROUTE_ALL_PREFILL])
def test_head_size_64_norm_only_and_rope_only(route):
    p = w.make_problem(name="prep-64", seed=54, dtype="bf16", num_heads=8, kv_num_heads=2, head_size=64,
                       block_size=32, past=[100, 5, 40], q_lens=[70, 3, 1])
    check(p, dict(q_norm_weight=_weights(p, 1.0, 2.0), k_norm_weight=_weights(p, 2.0, 1.0), eps=1e-6,
                  rotary_dim=0), route=route)
    check(p, dict(rotary_dim=32, theta=1e4), route=route)


def test_long_context_positions():
    # positions near 1.3e5: the fp32 rotary table and the fp64 one differ by ~1e-2 rad here
    p = w.make_problem(name="prep-long", seed=55, dtype="bf16", num_heads=8, kv_num_heads=2, head_size=128,
                       block_size=16, past=[131000, 90000], q_lens=[1, 1])
    check(p, dict(q_norm_weight=None, k_norm_weight=_weights(p, 0.8, 1.2), eps=1e-6, rotary_dim=128, theta=1e6))


# ---- the output gate ----

def _gate_bits(p, seed):
    g = w.uniform(seed, 1, p.num_tokens * p.num_heads * p.head_size) * 8.0 - 4.0
    g = oracle.double_to_bf16(g) if p.dtype == "bf16" else oracle.double_to_f16(g)
    return g.reshape(p.num_tokens, p.num_heads * p.head_size)


GATE_CASES = {
    "decode-splits": (lambda: w.make_problem(name="g-dec", seed=61, dtype="fp16", num_heads=32, kv_num_heads=8,
                                             head_size=128, block_size=64, past=[3000, 17, 600], q_lens=[1, 2, 4]),
                      {"decode_split_keys": 64}),
    "decode-auto-bf16": (lambda: w.make_problem(name="g-dec2", seed=62, dtype="bf16", num_heads=16, kv_num_heads=4,
                                                head_size=128, block_size=16, past=[4000, 1], q_lens=[1, 1]), {}),
    "prefill-bf16": (lambda: w.make_problem(name="g-pre", seed=63, dtype="bf16", num_heads=16, kv_num_heads=4,
                                            head_size=128, block_size=256, past=[0, 300], q_lens=[300, 129]), {}),
    "mixed-64": (lambda: w.make_problem(name="g-mix", seed=64, dtype="fp16", num_heads=8, kv_num_heads=2,
                                        head_size=64, block_size=32, past=[100, 5, 40], q_lens=[70, 3, 1]), {}),
}


@pytest.mark.parametrize("name", sorted(GATE_CASES))
def test_output_gate(name):
    make, opts = GATE_CASES[name]
    p = make()
    gb = _gate_bits(p, 70)
    ref = oracle.paged_attention(p, gate=gb)
    d = upload(p)
    gate = torch.from_numpy(gb.view(np.int16)).cuda().view(TORCH_DT[p.dtype])
    lse = torch.empty((p.num_tokens, p.num_heads), dtype=torch.float32, device="cuda")
    out = pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                             d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], d["slot_mapping"],
                             num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, scale=p.scale, lse=lse,
                             output_gate=gate, **opts)
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(d["key_cache"]), ref["key_cache"])
    assert_close(bits_of(out).reshape(p.num_tokens, p.num_heads, p.head_size), ref["out"], p.dtype, name)
    lg = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lg - ref["lse"]) <= 5e-4 + 1e-5 * np.abs(ref["lse"]))  # lse is not gated


def test_self_planned_decode_with_prep():
    # a decode-only call with the host bound and derived slots: no planner; the cache-write
    # kernel prepares Q and K, the decode kernel cuts its own share of the partition
    p = w.make_problem(name="prep-self", seed=56, dtype="fp16", num_heads=32, kv_num_heads=8, head_size=128,
                       block_size=16, past=[2900, 0, 17, 600, 1, 64], q_lens=[1, 2, 1, 4, 3, 1])
    n0 = pa.kernel_launch_count()
    check(p, dict(q_norm_weight=_weights(p, 0.5, 1.5), k_norm_weight=_weights(p, 1.2, 0.8), eps=1e-6,
                  rotary_dim=128, theta=1e6), max_query_len=int(p.q_lens.max()))
    assert pa.kernel_launch_count() - n0 == 3
