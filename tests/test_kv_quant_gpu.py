"""INT8 / INT4 per-channel KV caches on both attention kernels, through the C ABI against
the oracle (oracle_quantize_rows, oracle_attention_q; pinned in test_oracle_quant_pins.py):
decode-only batches on the decode kernel, and chunked-prefill and mixed batches whose
prefill-class rows run on the tcgen05 prefill kernel (code tiles turned into fp16 in shared
memory).

The cache write quantizes this call's K and V rows with the same rule as the oracle (IEEE
fp32 quotient, rint half to even, clamp), so the code caches must match bit for bit. The
attention reads the codes as exact fp16 integers, folds the K scales into an fp16 copy of
the query rows (with a power-of-two row exponent) and the V scales into the output, so the
outputs must meet the usual bound |gpu - oracle| <= 2e-3 + 1e-2 |oracle|, and lse its
5e-4 + 1e-5 |oracle| widened by the scores' error bound of the fp16 scaled query rows
(score_error_bound: relative 2^-11 per product term).
"""
import numpy as np
import pytest
import torch

import oracle
import varlen_paged_kv_gb300 as pa
import workloads as w
from gpu_utils import TORCH_DT, assert_close, bits_of, cache_bytes, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is required for the gpu tests")
    from varlen_paged_kv_gb300 import build
    build.build()


CASES = {
    # name: (fmt, dtype, nh, kvh, hs, bs, past, q_lens, packed, drops)
    "int8-gqa4-fp16": ("int8", "fp16", 32, 8, 128, 256, [0, 5, 300, 1000], [1, 1, 2, 4], False, 0),
    "int8-gqa8-bf16-pages16": ("int8", "bf16", 16, 2, 128, 16, [4000, 17, 1], [1, 2, 1], False, 0),
    "int8-mha-q16-hs64": ("int8", "fp16", 8, 8, 64, 32, [100, 33], [16, 7], False, 0),
    "int8-hs256-bf16": ("int8", "bf16", 16, 2, 256, 64, [700, 3000, 0], [1, 2, 1], False, 0),
    "int8-packed-drops": ("int8", "fp16", 32, 8, 128, 64, [900, 50, 3000, 7], [1, 2, 4, 3], True, 3),
    "int4-gqa4-fp16": ("int4", "fp16", 32, 8, 128, 256, [0, 5, 300, 1000], [1, 1, 2, 4], False, 0),
    "int4-gqa16-bf16": ("int4", "bf16", 16, 1, 128, 64, [500, 1, 2500], [1, 1, 1], False, 0),
    "int4-hs256-fp16": ("int4", "fp16", 16, 2, 256, 32, [129, 63, 1], [2, 1, 1], False, 0),
    "int4-packed-drops-bf16": ("int4", "bf16", 32, 8, 128, 16, [60, 4, 2000], [2, 4, 1], True, 2),
    # at most 8 query rows per item (q_len * G <= 8): the decode kernel's narrow form
    "int8-narrow-gqa4-q2-fp16": ("int8", "fp16", 32, 8, 128, 64, [0, 5, 300, 1000, 4097], [1, 2, 1, 2, 1], False, 0),
    "int8-narrow-gqa8-hs256-bf16": ("int8", "bf16", 16, 2, 256, 32, [700, 3000, 0], [1, 1, 1], False, 0),
    "int8-narrow-mha-q8-hs64": ("int8", "fp16", 8, 8, 64, 32, [100, 33, 0], [8, 3, 1], False, 0),
    "int8-narrow-packed-drops": ("int8", "fp16", 32, 8, 128, 64, [900, 50, 3000, 7], [1, 2, 2, 1], True, 2),
    "int4-narrow-gqa4-q2-bf16": ("int4", "bf16", 32, 8, 128, 16, [60, 4, 2000, 0], [2, 1, 2, 1], False, 0),
    "int4-narrow-gqa2-q4-hs256": ("int4", "fp16", 8, 4, 256, 64, [129, 63, 1, 500], [4, 1, 3, 2], False, 0),
}


def _problem(name, seed=31):
    fmt, dt, nh, kvh, hs, bs, past, q, packed, drops = CASES[name]
    return w.make_problem(name=name, seed=seed, dtype=dt, num_heads=nh, kv_num_heads=kvh, head_size=hs,
                          block_size=bs, past=past, q_lens=q, packed=packed,
                          slot_mode="explicit" if drops else "omitted", drop_count=drops, kv_quant=fmt)


def _run(p, split=0, route=pa.ROUTE_AUTO, decode_sms=0, **kw):
    d = upload(p)
    lse = torch.empty((p.num_tokens, p.num_heads), dtype=torch.float32, device="cuda")
    dims = pa.make_dims(p.num_tokens, p.batch_size, p.head_size, p.num_blocks, p.block_size,
                        p.max_blocks_per_sequence, TORCH_DT[p.dtype], split, route, int(p.q_lens.max()),
                        "qk_prep" in kw, p.kv_quant, decode_sms)
    ws = torch.zeros(pa.workspace_size(dims, p.num_heads, p.kv_num_heads), dtype=torch.uint8, device="cuda")
    out = pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                             d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], d["slot_mapping"],
                             num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, scale=p.scale, workspace=ws,
                             decode_split_keys=split, max_query_len=int(p.q_lens.max()), lse=lse, route=route,
                             decode_sms=decode_sms, kv_quant=p.kv_quant, k_scale=d["k_scale"], v_scale=d["v_scale"],
                             **kw)
    assert pa.read_device_error(ws) == 0
    return d, out, lse


def _codes(raw, fmt, hs):
    """Integer codes (..., hs) of a code cache (..., row bytes)."""
    if fmt == "int8":
        return raw.view(np.int8).astype(np.float64)
    c = np.stack([raw & 15, raw >> 4], axis=-1).reshape(raw.shape[:-1] + (hs,)).astype(np.int64)
    return np.where(c >= 8, c - 16, c).astype(np.float64)


def score_error_bound(p, key_cache):
    """Per (row, head): the scores' error from the fp16 scaled query rows, an fp16 rounding
    (relative 2^-11) of every term q_c * s_c: scale * 2^-11 * max_t sum_c |q_c k_tc|."""
    nh, kvh, hs, bs = p.num_heads, p.kv_num_heads, p.head_size, p.block_size
    k = _codes(key_cache, p.kv_quant, hs).reshape(-1, kvh, hs) * p.k_scale[None].astype(np.float64)
    q = (oracle.bf16_to_double if p.dtype == "bf16" else oracle.f16_to_double)(p.query[:, :nh * hs])
    q = np.abs(q.reshape(-1, nh, hs))
    sc = p.scale if p.scale else 1.0 / np.sqrt(hs)
    out = np.zeros((p.num_tokens, nh))
    for b in range(p.batch_size):
        c0, past = int(p.cumulative_sequence_length[b]), int(p.past_seqlens[b])
        for j in range(int(p.q_lens[b])):
            keys = np.arange(past + j + 1)
            rows = p.block_table[b, keys // bs].astype(np.int64) * bs + keys % bs
            kk = np.abs(k[rows])  # (L, kvh, hs)
            for h in range(nh):
                out[c0 + j, h] = sc * 2.0 ** -11 * np.max(kk[:, h // (nh // kvh)] @ q[c0 + j, h])
    return out


def _check(p, ref, d, out, lse, exact_codes=True, prepared=None):
    kc, vc = cache_bytes(d["key_cache"]), cache_bytes(d["value_cache"])
    assert np.array_equal(vc, ref["value_cache"]), "value codes differ"
    if exact_codes:
        assert np.array_equal(kc, ref["key_cache"]), "key codes differ"
    assert_close(bits_of(out).reshape(p.num_tokens, p.num_heads, p.head_size), ref["out"], p.dtype, p.name)
    lg = lse.cpu().numpy().astype(np.float64)
    bound = 5e-4 + 1e-5 * np.abs(ref["lse"]) + score_error_bound(prepared or p, ref["key_cache"])
    assert np.all(np.abs(lg - ref["lse"]) <= bound), "lse differs"


@pytest.mark.parametrize("split", [0, 64])
@pytest.mark.parametrize("name", sorted(CASES))
def test_integer_cache_decode(name, split):
    p = _problem(name)
    ref = oracle.paged_attention(p)
    d, out, lse = _run(p, split)
    _check(p, ref, d, out, lse)


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_codes_at_and_next_to_ties(fmt):
    # a code is rint (ties to even) of the correctly rounded quotient value / scale: new K and
    # V values at exact half-integer multiples of power-of-two scales (past the saturation
    # too), and a third of them one fp16 unit in the last place away on either side
    p = w.make_problem(name="ties", seed=41, dtype="fp16", num_heads=8, kv_num_heads=2, head_size=128,
                       block_size=16, past=[20, 7, 300], q_lens=[40, 30, 1], kv_quant=fmt)
    qm = 127 if fmt == "int8" else 7
    rng = np.random.default_rng(5)
    kvh, hs, n = p.kv_num_heads, p.head_size, p.num_tokens
    p.k_scale = (2.0 ** rng.integers(-8, -3, size=(kvh, hs))).astype(np.float32)
    p.v_scale = (2.0 ** rng.integers(-8, -3, size=(kvh, hs))).astype(np.float32)

    def values(scale):
        half = rng.integers(-qm - 2, qm + 2, size=(n, kvh, hs)) + 0.5  # exact in fp16 times 2^-8..2^-4
        bits = oracle.double_to_f16(half * scale[None].astype(np.float64)).reshape(n, kvh * hs)
        step = rng.integers(-1, 2, size=bits.shape)  # one unit of the magnitude down, none, up
        return (bits.astype(np.int64) + step).astype(np.uint16)

    p.key = values(p.k_scale)
    p.value = values(p.v_scale)
    ref = oracle.paged_attention(p)
    d, out, lse = _run(p)
    assert np.array_equal(cache_bytes(d["key_cache"]), ref["key_cache"]), "key codes differ"
    assert np.array_equal(cache_bytes(d["value_cache"]), ref["value_cache"]), "value codes differ"


@pytest.mark.parametrize("q_lens", [[1, 2, 1], [1, 1, 1]])  # 16 rows per item at most; 8: the narrow form
@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_integer_cache_with_prep_and_gate(fmt, q_lens):
    p = w.make_problem(name="q-prep", seed=33, dtype="bf16", num_heads=16, kv_num_heads=2, head_size=128,
                       block_size=64, past=[100, 2000, 7], q_lens=q_lens, kv_quant=fmt)
    to_t = oracle.double_to_bf16
    prep_bits = dict(q_norm_weight=to_t(np.linspace(0.5, 1.5, 128)), k_norm_weight=to_t(np.linspace(1.2, 0.8, 128)),
                     eps=1e-6, rotary_dim=64, theta=1.0e6)
    gate_bits = to_t(w.uniform(34, 1, p.num_tokens * 16 * 128) * 8.0 - 4.0).reshape(p.num_tokens, 16 * 128)
    ref = oracle.paged_attention(p, prep=prep_bits, gate=gate_bits)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)
    prep = dict(q_norm_weight=dev(prep_bits["q_norm_weight"]), k_norm_weight=dev(prep_bits["k_norm_weight"]),
                eps=1e-6, rotary_dim=64, theta=1.0e6)
    d, out, lse = _run(p, qk_prep=prep, output_gate=dev(gate_bits))
    _check(p, ref, d, out, lse, exact_codes=False, prepared=oracle.apply_qk_prep(p, prep_bits))
    # prepared keys are computed in fp32 here and in fp64 by the oracle, then rounded to T:
    # where the two roundings differ the code may differ by one
    kc = cache_bytes(d["key_cache"]).reshape(-1)
    rk = ref["key_cache"].reshape(-1)
    if fmt == "int8":
        a, b = kc.view(np.int8).astype(int), rk.view(np.int8).astype(int)
    else:
        a = np.stack([(kc & 15), (kc >> 4)]).astype(int)
        b = np.stack([(rk & 15), (rk >> 4)]).astype(int)
        a, b = np.where(a >= 8, a - 16, a), np.where(b >= 8, b - 16, b)
    assert np.all(np.abs(a - b) <= 1) and np.mean(a != b) < 0.01


# prefill-class rows on integer caches: (fmt, dtype, nh, kvh, hs, bs, past, q_lens, packed, drops)
PREFILL_CASES = {
    "int8-chunked-fp16": ("int8", "fp16", 32, 8, 128, 256, [1000, 17, 255], [200, 64, 513], False, 0),
    "int8-mixed-packed-drops-bf16": ("int8", "bf16", 32, 8, 128, 64, [0, 900, 50, 3000], [130, 1, 40, 2], True, 9),
    "int8-hs64-pages16": ("int8", "fp16", 8, 2, 64, 16, [0, 5, 100], [70, 3, 300], False, 0),
    "int8-odd-group-bf16": ("int8", "bf16", 6, 2, 128, 32, [40, 0], [150, 129], False, 0),
    "int4-chunked-bf16": ("int4", "bf16", 16, 4, 128, 32, [0, 300, 2000], [300, 129, 17], False, 0),
    "int4-mixed-packed-drops-fp16": ("int4", "fp16", 32, 8, 128, 16, [60, 4, 2000, 0], [2, 40, 1, 129], True, 5),
    "int4-one-kv-head": ("int4", "fp16", 16, 1, 128, 64, [500, 0], [100, 20], False, 0),
    "int8-one-kv-head-hs64": ("int8", "bf16", 4, 1, 64, 16, [33, 0], [40, 200], False, 0),
    "int8-hs256-chunked-bf16": ("int8", "bf16", 16, 2, 256, 64, [700, 0, 129], [130, 300, 2], False, 0),
    "int4-hs256-packed-drops-fp16": ("int4", "fp16", 8, 2, 256, 32, [0, 2000, 63], [200, 1, 129], True, 4),
    "int4-hs256-one-kv-head": ("int4", "bf16", 8, 1, 256, 16, [10, 0], [50, 17], False, 0),
}


def _prefill_problem(name, seed=37):
    fmt, dt, nh, kvh, hs, bs, past, q, packed, drops = PREFILL_CASES[name]
    return w.make_problem(name=name, seed=seed, dtype=dt, num_heads=nh, kv_num_heads=kvh, head_size=hs,
                          block_size=bs, past=past, q_lens=q, packed=packed,
                          slot_mode="explicit" if drops else "omitted", drop_count=drops, kv_quant=fmt)


@pytest.mark.parametrize("route", [pa.ROUTE_AUTO, pa.ROUTE_ALL_PREFILL])
@pytest.mark.parametrize("name", sorted(PREFILL_CASES))
def test_integer_cache_prefill_rows(name, route):
    p = _prefill_problem(name)
    ref = oracle.paged_attention(p)
    d, out, lse = _run(p, route=route)
    _check(p, ref, d, out, lse)


@pytest.mark.parametrize("dsm", [1, 76])
def test_integer_cache_mixed_batch_on_split_sms(dsm):
    p = _prefill_problem("int8-mixed-packed-drops-bf16")
    ref = oracle.paged_attention(p)
    d, out, lse = _run(p, decode_sms=dsm, split=64)
    _check(p, ref, d, out, lse)


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_integer_cache_prefill_with_prep_and_gate(fmt):
    p = w.make_problem(name="q-prep-prefill", seed=38, dtype="fp16", num_heads=16, kv_num_heads=4, head_size=128,
                       block_size=32, past=[0, 700, 5], q_lens=[200, 1, 130], kv_quant=fmt)
    to_t = oracle.double_to_f16
    prep_bits = dict(q_norm_weight=to_t(np.linspace(0.5, 1.5, 128)), k_norm_weight=to_t(np.linspace(1.2, 0.8, 128)),
                     eps=1e-6, rotary_dim=128, theta=1.0e4)
    gate_bits = to_t(w.uniform(39, 1, p.num_tokens * 16 * 128) * 8.0 - 4.0).reshape(p.num_tokens, 16 * 128)
    ref = oracle.paged_attention(p, prep=prep_bits, gate=gate_bits)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(torch.float16)
    prep = dict(q_norm_weight=dev(prep_bits["q_norm_weight"]), k_norm_weight=dev(prep_bits["k_norm_weight"]),
                eps=1e-6, rotary_dim=128, theta=1.0e4)
    d, out, lse = _run(p, qk_prep=prep, output_gate=dev(gate_bits))
    _check(p, ref, d, out, lse, exact_codes=False, prepared=oracle.apply_qk_prep(p, prep_bits))


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_refused_self_planned_batch_writes_nothing(fmt):
    # a decode-only call with no planner: an inconsistent batch (the last offset one short of
    # the token count) must leave both code caches and the output untouched
    p = w.make_problem(name="q-refuse", seed=35, dtype="fp16", num_heads=16, kv_num_heads=4, head_size=128,
                       block_size=32, past=[40, 700, 3], q_lens=[1, 2, 1], kv_quant=fmt)
    p.cumulative_sequence_length = p.cumulative_sequence_length.copy()
    p.cumulative_sequence_length[-1] -= 1
    d = upload(p)
    before = cache_bytes(d["key_cache"]).copy(), cache_bytes(d["value_cache"]).copy()
    dims = pa.make_dims(p.num_tokens, p.batch_size, p.head_size, p.num_blocks, p.block_size,
                        p.max_blocks_per_sequence, TORCH_DT[p.dtype], 0, pa.ROUTE_AUTO, 2, False, fmt)
    ws = torch.zeros(pa.workspace_size(dims, p.num_heads, p.kv_num_heads), dtype=torch.uint8, device="cuda")
    out = torch.full((p.num_tokens, p.num_heads * p.head_size), 7.0, dtype=TORCH_DT[p.dtype], device="cuda")
    pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                       d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], None,
                       num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, output=out, workspace=ws,
                       max_query_len=2, kv_quant=fmt, k_scale=d["k_scale"], v_scale=d["v_scale"])
    assert pa.read_device_error(ws) & pa.DEVERR_BAD_BATCH
    assert np.array_equal(cache_bytes(d["key_cache"]), before[0])
    assert np.array_equal(cache_bytes(d["value_cache"]), before[1])
    assert torch.all(out == 7.0)


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_full_size_decode_batch_on_integer_caches(fmt):
    # the 64-sequence decode batch as bench.py times it: every code byte and every output
    # element against the oracle
    p = w.config_kv_quant(2, fmt)
    ref = oracle.paged_attention(p)
    d, out, lse = _run(p)
    _check(p, ref, d, out, lse)
