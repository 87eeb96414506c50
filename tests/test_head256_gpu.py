"""head_size 256: the decode kernel (one CTA per SM) and the 256-wide prefill kernel (one
head per unit, two S buffers in TMEM), through the C ABI against the oracle: decode-only
batches with and without forced splits, prefill and chunked prefill (fp16, bf16 with the
fp16 V copy and bf16 on the two-product path), packed rows with dropped slots, mixed
batches, lse, the Q/K preparation and the output gate.

Same bars as the other parity tests: caches bit for bit (prepared keys within one unit in
the last place), outputs within 2e-3 + 1e-2 |oracle|, lse within 5e-4 + 1e-5 |oracle|.
"""
import numpy as np
import pytest
import torch

import oracle
import varlen_paged_kv_gb300 as pa
import workloads as w
from gpu_utils import TORCH_DT, assert_close, bits_of, upload
from helpers import bits_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is required for the gpu tests")
    from varlen_paged_kv_gb300 import build
    build.build()


CASES = {
    # name: (dtype, nh, kvh, bs, past, q_lens)
    "gqa8-q-up-to-2": ("fp16", 16, 2, 64, [0, 5, 700, 3000], [1, 1, 2, 1]),
    "mha-q16": ("bf16", 4, 4, 16, [33, 1000], [16, 3]),
    "gqa16-long": ("bf16", 16, 1, 256, [4000, 0], [1, 1]),
    "gqa4-ragged": ("fp16", 8, 2, 32, [129, 63, 1], [4, 2, 1]),
    # 64 sequences, the most the 256-wide decode kernel plans itself, and 65, planned on the host
    "gqa8-b64": ("bf16", 16, 2, 16, [(37 * i) % 300 for i in range(64)], [1 + (i % 5 == 0) for i in range(64)]),
    "gqa8-b65": ("fp16", 16, 2, 16, [(41 * i) % 280 for i in range(65)], [1 + (i % 7 == 0) for i in range(65)]),
}


def _problem(name, seed=91):
    dt, nh, kvh, bs, past, q = CASES[name]
    return w.make_problem(name=name, seed=seed, dtype=dt, num_heads=nh, kv_num_heads=kvh, head_size=256,
                          block_size=bs, past=past, q_lens=q, packed=False, slot_mode="omitted", drop_count=0,
                          num_blocks=None)


def _workspace(p, split=0, prep=False):
    dims = pa.make_dims(p.num_tokens, p.batch_size, 256, p.num_blocks, p.block_size, p.max_blocks_per_sequence,
                        TORCH_DT[p.dtype], split, pa.ROUTE_AUTO, int(p.q_lens.max()), prep)
    n = pa.workspace_size(dims, p.num_heads, p.kv_num_heads)
    assert n > 0
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def _check_keys(kc, ref_kc, dtype, exact):
    if exact:
        assert np.array_equal(kc, ref_kc), "key cache differs"
        return
    diff = kc != ref_kc
    if diff.any():  # prepared keys: within one unit in the last place of T
        g, r = bits_to_f64(kc[diff], dtype), bits_to_f64(ref_kc[diff], dtype)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(r), 1e-30))) - (7 if dtype == "bf16" else 10))
        ulp = np.maximum(ulp, 2.0 ** (-133 if dtype == "bf16" else -24))
        assert np.all(np.abs(g - r) <= ulp * 1.0000001), "a prepared key is more than one ulp off"
        assert diff.mean() < 0.01


@pytest.mark.parametrize("split", [0, 64])
@pytest.mark.parametrize("name", sorted(CASES))
def test_head256_decode(name, split):
    p = _problem(name)
    ref = oracle.paged_attention(p)
    d = upload(p)
    ws = _workspace(p, split)
    lse = torch.empty((p.num_tokens, p.num_heads), dtype=torch.float32, device="cuda")
    out = pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                             d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], d["slot_mapping"],
                             num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, scale=p.scale,
                             decode_split_keys=split, workspace=ws, max_query_len=int(p.q_lens.max()), lse=lse)
    assert pa.read_device_error(ws) == 0
    _check_keys(bits_of(d["key_cache"]), ref["key_cache"], p.dtype, exact=True)
    assert np.array_equal(bits_of(d["value_cache"]), ref["value_cache"]), "value cache differs"
    assert_close(bits_of(out).reshape(p.num_tokens, p.num_heads, 256), ref["out"], p.dtype, name)
    lg = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lg - ref["lse"]) <= 5e-4 + 1e-5 * np.abs(ref["lse"])), "lse differs"


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_head256_prep_and_gate(dtype):
    # RMSNorm of both heads, rotary over the first 64 components, sigmoid output gate
    p = w.make_problem(name="h256-prep", seed=92, dtype=dtype, num_heads=16, kv_num_heads=2, head_size=256,
                       block_size=64, past=[100, 2000, 7], q_lens=[1, 2, 1], packed=False, slot_mode="omitted",
                       drop_count=0, num_blocks=None)
    to_t = oracle.double_to_bf16 if dtype == "bf16" else oracle.double_to_f16
    prep_bits = dict(q_norm_weight=to_t(np.linspace(0.5, 1.5, 256)), k_norm_weight=to_t(np.linspace(1.2, 0.8, 256)),
                     eps=1e-6, rotary_dim=64, theta=1.0e7)
    g = w.uniform(93, 1, p.num_tokens * p.num_heads * 256) * 8.0 - 4.0
    gate_bits = to_t(g).reshape(p.num_tokens, p.num_heads * 256)
    ref = oracle.paged_attention(p, prep=prep_bits, gate=gate_bits)
    d = upload(p)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(TORCH_DT[dtype])
    prep = dict(q_norm_weight=dev(prep_bits["q_norm_weight"]), k_norm_weight=dev(prep_bits["k_norm_weight"]),
                eps=1e-6, rotary_dim=64, theta=1.0e7)
    ws = _workspace(p, 0, prep=True)
    lse = torch.empty((p.num_tokens, p.num_heads), dtype=torch.float32, device="cuda")
    out = pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                             d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], d["slot_mapping"],
                             num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, scale=p.scale, workspace=ws,
                             max_query_len=int(p.q_lens.max()), lse=lse, qk_prep=prep, output_gate=dev(gate_bits))
    assert pa.read_device_error(ws) == 0
    _check_keys(bits_of(d["key_cache"]), ref["key_cache"], dtype, exact=False)
    assert np.array_equal(bits_of(d["value_cache"]), ref["value_cache"]), "value cache differs"
    assert_close(bits_of(out).reshape(p.num_tokens, p.num_heads, 256), ref["out"], dtype, "h256-prep")
    lg = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lg - ref["lse"]) <= 5e-4 + 1e-5 * np.abs(ref["lse"])), "lse differs"


PREFILL = {
    # name: (dtype, nh, kvh, bs, past, q_lens, packed, drops)
    "ragged-fp16": ("fp16", 8, 2, 256, [0, 0], [300, 129], False, 0),
    "chunked-bf16-copy": ("bf16", 16, 2, 64, [1000, 17, 255], [200, 64, 130], False, 0),
    "bf16-two-product": ("bf16", 4, 1, 128, [2500], [257], False, 0),
    "mixed-packed-drops": ("fp16", 8, 2, 32, [0, 900, 50, 3000], [130, 1, 40, 2], True, 9),
    "mha-pages16": ("bf16", 4, 4, 16, [5, 0], [140, 33], False, 0),
}


def _prefill_problem(name, seed=95):
    dt, nh, kvh, bs, past, q, packed, drops = PREFILL[name]
    return w.make_problem(name=name, seed=seed, dtype=dt, num_heads=nh, kv_num_heads=kvh, head_size=256,
                          block_size=bs, past=past, q_lens=q, packed=packed,
                          slot_mode="explicit" if drops else "omitted", drop_count=drops, num_blocks=None)


@pytest.mark.parametrize("route", [pa.ROUTE_AUTO, pa.ROUTE_ALL_PREFILL])
@pytest.mark.parametrize("name", sorted(PREFILL))
def test_head256_prefill(name, route):
    p = _prefill_problem(name)
    ref = oracle.paged_attention(p)
    d = upload(p)
    lse = torch.empty((p.num_tokens, p.num_heads), dtype=torch.float32, device="cuda")
    out = pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                             d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], d["slot_mapping"],
                             num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, scale=p.scale, route=route, lse=lse)
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(d["key_cache"]), ref["key_cache"]), "key cache differs"
    assert np.array_equal(bits_of(d["value_cache"]), ref["value_cache"]), "value cache differs"
    assert_close(bits_of(out).reshape(p.num_tokens, p.num_heads, 256), ref["out"], p.dtype, name)
    lg = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lg - ref["lse"]) <= 5e-4 + 1e-5 * np.abs(ref["lse"])), "lse differs"


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_head256_prefill_prep_and_gate(dtype):
    p = w.make_problem(name="h256-prep-pre", seed=96, dtype=dtype, num_heads=8, kv_num_heads=2, head_size=256,
                       block_size=64, past=[0, 300], q_lens=[260, 70], packed=False, slot_mode="omitted",
                       drop_count=0, num_blocks=None)
    to_t = oracle.double_to_bf16 if dtype == "bf16" else oracle.double_to_f16
    prep_bits = dict(q_norm_weight=to_t(np.linspace(0.5, 1.5, 256)), k_norm_weight=to_t(np.linspace(1.2, 0.8, 256)),
                     eps=1e-6, rotary_dim=64, theta=1.0e7)
    g = w.uniform(97, 1, p.num_tokens * p.num_heads * 256) * 8.0 - 4.0
    gate_bits = to_t(g).reshape(p.num_tokens, p.num_heads * 256)
    ref = oracle.paged_attention(p, prep=prep_bits, gate=gate_bits)
    d = upload(p)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(TORCH_DT[dtype])
    prep = dict(q_norm_weight=dev(prep_bits["q_norm_weight"]), k_norm_weight=dev(prep_bits["k_norm_weight"]),
                eps=1e-6, rotary_dim=64, theta=1.0e7)
    out = pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                             d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], d["slot_mapping"],
                             num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, scale=p.scale, qk_prep=prep,
                             output_gate=dev(gate_bits))
    torch.cuda.synchronize()
    _check_keys(bits_of(d["key_cache"]), ref["key_cache"], dtype, exact=False)
    assert np.array_equal(bits_of(d["value_cache"]), ref["value_cache"]), "value cache differs"
    assert_close(bits_of(out).reshape(p.num_tokens, p.num_heads, 256), ref["out"], dtype, "h256-prep-pre")
