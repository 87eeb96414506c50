"""The exported log-sum-exp (pa_paged_attention_lse) against the oracle's.

lse of row i, head h = ln sum_t exp(scale * <q_ih, k_t>) over the keys the row attends: the
natural-log, scale-included value that the (out, lse) merge of context-parallel partials
consumes (WS2 CP-Aware Attention Contract, "Reduction Semantics"). The kernels form it in
fp32 from the running max and sum that normalise the output (scores accumulated in fp32,
the hardware base-2 exponential and logarithm with relative errors near 2^-22), so it
is checked to 5e-4 + 1e-5 |lse| against the oracle's fp64 value. The output is checked
at the same time: asking for lse must not change it.
"""
import numpy as np
import pytest
import torch

import oracle
import varlen_paged_kv_gb300 as pa
import workloads as w
from gpu_utils import assert_close, bits_of, make_workspace, upload
from helpers import bits_to_f64

pytestmark = pytest.mark.gpu

LSE_ATOL, LSE_RTOL = 5e-4, 1e-5


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is required for the gpu tests")
    from varlen_paged_kv_gb300 import build
    build.build()


def run_with_lse(p, **opts):
    d = upload(p)
    ws = make_workspace(p, opts.get("decode_split_keys", 0), opts.get("route", pa.ROUTE_AUTO))
    lse = torch.full((p.num_tokens, p.num_heads), float("nan"), dtype=torch.float32, device="cuda")
    out = pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                             d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"],
                             d["slot_mapping"], num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, scale=p.scale,
                             workspace=ws, lse=lse, **opts)
    assert pa.read_device_error(ws) == 0
    return bits_of(out), lse.cpu().numpy().astype(np.float64)


CASES = {
    "tiny": (lambda: w.config(1), {}),
    "tiny-prefill-kernel": (lambda: w.config(1), {"route": pa.ROUTE_ALL_PREFILL}),
    "tiny-forced-splits": (lambda: w.config(1), {"decode_split_keys": 64}),
    "decode-bf16-gqa4": (lambda: w.make_problem(name="d", seed=21, dtype="bf16", num_heads=32, kv_num_heads=8,
                                                head_size=128, block_size=16, past=[4000, 0, 17, 700],
                                                q_lens=[1, 3, 4, 2]), {}),
    "decode-splits": (lambda: w.make_problem(name="s", seed=22, dtype="fp16", num_heads=16, kv_num_heads=4,
                                             head_size=128, block_size=64, past=[3000, 1500], q_lens=[1, 1]),
                      {"decode_split_keys": 448}),
    "prefill-ragged-bf16": (lambda: w.make_problem(name="p", seed=23, dtype="bf16", num_heads=32, kv_num_heads=8,
                                                   head_size=128, block_size=256, past=[0, 0], q_lens=[300, 129]),
                            {}),
    "chunked-fp16-head64": (lambda: w.make_problem(name="c", seed=24, dtype="fp16", num_heads=8, kv_num_heads=2,
                                                   head_size=64, block_size=32, past=[1000, 5], q_lens=[200, 70]),
                            {}),
    "bf16-long-history-two-products": (lambda: w.make_problem(name="h", seed=25, dtype="bf16", num_heads=8,
                                                              kv_num_heads=2, head_size=128, block_size=128,
                                                              past=[2500], q_lens=[257]), {}),
    "mixed-packed": (lambda: w.make_problem(name="m", seed=26, dtype="fp16", num_heads=32, kv_num_heads=8,
                                            head_size=128, block_size=256, past=[0, 900, 50, 3000],
                                            q_lens=[130, 1, 40, 2], packed=True, slot_mode="explicit",
                                            drop_count=9), {}),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_lse_matches_the_oracle(name):
    make, opts = CASES[name]
    p = make()
    ref = oracle.paged_attention(p)
    out_bits, lse = run_with_lse(p, **opts)
    N, nh, hs = p.num_tokens, p.num_heads, p.head_size
    assert_close(out_bits.reshape(N, nh, hs), ref["out"], p.dtype, name)
    err = np.abs(lse - ref["lse"])
    bad = ~(err <= LSE_ATOL + LSE_RTOL * np.abs(ref["lse"]))
    assert not bad.any(), f"{name}: {bad.sum()} lse values off (max err {np.nanmax(err):.3g})"


def test_lse_of_a_single_key_is_its_scaled_score():
    # a sequence with no history and one token sees only itself: lse = scale * <q, k>
    p = w.make_problem(name="one", seed=27, dtype="fp16", num_heads=4, kv_num_heads=2, head_size=64, block_size=16,
                       past=[0], q_lens=[1])
    _, lse = run_with_lse(p)
    q = bits_to_f64(p.query, "fp16").reshape(1, 4, 64)
    k = bits_to_f64(p.key, "fp16").reshape(1, 2, 64)
    scale = p.scale if p.scale != 0 else 1 / np.sqrt(64)
    want = np.array([scale * q[0, h] @ k[0, h // 2] for h in range(4)])
    assert np.all(np.abs(lse[0] - want) <= LSE_ATOL + LSE_RTOL * np.abs(want))
