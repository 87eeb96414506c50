"""Pins of the oracle's integer KV caches (oracle_quantize_rows, oracle_scatter_codes,
oracle_attention_q) to facts other than the oracle itself.

Reading pinned: a value x of type T is stored as code = min(max(rint(fl32(x) / s), -Q), Q)
with the fp32 quotient correctly rounded and rint rounding half to even, Q = 127 (INT8) or
7 (INT4); INT4 codes are packed two per byte, channel 2i in the low nibble; attention reads
code * s with s the (KV head, channel) scale.
"""
import numpy as np
import pytest

import oracle
import workloads as w

QMAX = {"int8": 127, "int4": 7}


def _bits(x, dtype):
    x = np.asarray(x, dtype=np.float64)
    return oracle.double_to_bf16(x).reshape(x.shape) if dtype == "bf16" else oracle.double_to_f16(x).reshape(x.shape)


def _codes(x, dtype, fmt, scale):
    """oracle_quantize_rows on one row (kvh = 1); returns the integer codes per channel."""
    x = np.asarray(x, dtype=np.float64)
    hs = x.shape[-1]
    c = oracle.quantize_rows(_bits(x, dtype).reshape(1, hs), dtype, fmt, 1, hs, np.asarray(scale, np.float32).reshape(1, hs))
    return unpack(c[0], fmt, hs)


def unpack(row, fmt, hs):
    """Integer codes of one code row (the storage format stated in the docstring)."""
    row = np.asarray(row, dtype=np.uint8)
    if fmt == "int8":
        return row.view(np.int8).astype(np.int64)[:hs]
    lo = (row & 0x0F).astype(np.int64)
    hi = (row >> 4).astype(np.int64)
    out = np.empty(hs, dtype=np.int64)
    out[0::2], out[1::2] = lo, hi
    return np.where(out >= 8, out - 16, out)


@pytest.mark.parametrize("fmt", ["int8", "int4"])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_exact_multiples_give_their_integer(fmt, dtype):
    # x = k * s with s a power of two: the quotient is k exactly
    qm = QMAX[fmt]
    k = np.arange(-qm, qm + 1, dtype=np.float64)
    hs = len(k) + (len(k) % 2)
    k = np.concatenate([k, np.zeros(hs - len(k))])
    s = np.full(hs, 0.125)
    assert np.array_equal(_codes(k * 0.125, dtype, fmt, s), k.astype(np.int64))


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_halfway_values_round_to_even(fmt):
    # quotients 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, -3.5 with s = 0.25 (all exact in fp16)
    q = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, -3.5])
    s = np.full(8, 0.25)
    assert np.array_equal(_codes(q * 0.25, "fp16", fmt, s), [0, 2, 2, 0, -2, -2, 4, -4])


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_saturation_zero_and_nan(fmt):
    qm = QMAX[fmt]
    x = np.array([1000.0, -1000.0, 0.0, -0.0, np.inf, -np.inf, np.nan, 0.01])
    s = np.full(8, 0.5)
    assert np.array_equal(_codes(x, "fp16", fmt, s), [qm, -qm, 0, 0, qm, -qm, -qm, 0])


@pytest.mark.parametrize("fmt", ["int8", "int4"])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_quantization_matches_numpy_float32(fmt, dtype):
    # the definition through numpy's IEEE float32 division, rint and clip
    x_bits = w.normal_bits(3, 1, (64, 2 * 32), dtype)
    scale = (0.5 + w.uniform(3, 2, 64).reshape(2, 32)).astype(np.float32) / (QMAX[fmt] / 4)
    codes = oracle.quantize_rows(x_bits, dtype, fmt, 2, 32, scale)
    xf = (oracle.bf16_to_double(x_bits) if dtype == "bf16" else oracle.f16_to_double(x_bits)).astype(np.float32)
    want = np.clip(np.rint(xf.reshape(64, 2, 32) / scale[None]), -QMAX[fmt], QMAX[fmt]).astype(np.int64)
    got = np.stack([unpack(r, fmt, 64) for r in codes]).reshape(64, 2, 32)
    assert np.array_equal(got, want)
    # symmetric: -x gives -code
    neg = x_bits ^ np.uint16(0x8000)
    got_neg = np.stack([unpack(r, fmt, 64) for r in oracle.quantize_rows(neg, dtype, fmt, 2, 32, scale)])
    assert np.array_equal(got_neg.reshape(64, 2, 32), -want)


def test_int4_nibble_order_by_hand():
    # channel 0 -> low nibble, channel 1 -> high nibble, two's complement: 3 and -2 give 0xE3
    c = oracle.quantize_rows(_bits([3.0, -2.0, -7.0, 7.0], "fp16").reshape(1, 4), "fp16", "int4", 1, 4,
                             np.ones((1, 4), np.float32))
    assert c.tolist() == [[0xE3, 0x79]]


def test_int8_bytes_by_hand():
    c = oracle.quantize_rows(_bits([1.0, -1.0, 127.0, -127.0], "fp16").reshape(1, 4), "fp16", "int8", 1, 4,
                             np.ones((1, 4), np.float32))
    assert c.tolist() == [[0x01, 0xFF, 0x7F, 0x81]]


def _quant_problem(fmt, dtype, seed=5, **kw):
    args = dict(name="qpin", seed=seed, dtype=dtype, num_heads=4, kv_num_heads=2, head_size=32, block_size=16,
                past=[0, 7, 20], q_lens=[1, 3, 5])
    args.update(kw)
    return w.make_problem(kv_quant=fmt, **args)


@pytest.mark.parametrize("fmt", ["int8", "int4"])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_attention_equals_the_16bit_operator_on_exact_values(fmt, dtype):
    # power-of-two scales make every code * s exact in T: the integer-cache operator must
    # then be the plain operator on a T cache holding those values (pinned elsewhere)
    p = _quant_problem(fmt, dtype)
    kvh, hs = p.kv_num_heads, p.head_size
    p.k_scale = (2.0 ** -(3 + (np.arange(kvh * hs) % 4))).astype(np.float32).reshape(kvh, hs)
    p.v_scale = (2.0 ** -(2 + (np.arange(kvh * hs) % 3))).astype(np.float32).reshape(kvh, hs)
    r = oracle.paged_attention(p)
    # the same operator on T caches: K/V rows and caches replaced by their exact values
    kr, vr = oracle.kv_rows(p)
    kq = oracle.quantize_rows(kr, dtype, fmt, kvh, hs, p.k_scale)
    vq = oracle.quantize_rows(vr, dtype, fmt, kvh, hs, p.v_scale)

    def values(code_rows, scale):  # (n, rb) code rows -> T bits of code * s
        n = code_rows.shape[0]
        c = np.stack([unpack(row, fmt, kvh * hs) for row in code_rows.reshape(n, -1)]) if n else np.zeros((0, kvh * hs))
        return _bits(c.reshape(n, kvh, hs) * scale[None].astype(np.float64), dtype).reshape(n, kvh * hs)

    t = p.copy()
    t.kv_quant = None
    nb = p.num_blocks * p.block_size
    t.key_cache = values(p.key_cache.reshape(nb, -1), p.k_scale).reshape(p.num_blocks, p.block_size, kvh, hs)
    t.value_cache = values(p.value_cache.reshape(nb, -1), p.v_scale).reshape(p.num_blocks, p.block_size, kvh, hs)
    t.key = values(kq, p.k_scale)
    t.value = values(vq, p.v_scale)
    ref = oracle.paged_attention(t)
    assert np.array_equal(r["out"], ref["out"])
    assert np.array_equal(r["lse"], ref["lse"])
    assert np.array_equal(r["out_bits"], ref["out_bits"])


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_one_key_returns_its_dequantized_value(fmt):
    # a single token without history attends only itself: out = code(v) * s_v, per KV head
    p = _quant_problem(fmt, "fp16", past=[0], q_lens=[1], num_heads=4, kv_num_heads=2)
    r = oracle.paged_attention(p)
    kr, vr = oracle.kv_rows(p)
    codes = unpack(oracle.quantize_rows(vr, "fp16", fmt, 2, 32, p.v_scale)[0], fmt, 64).reshape(2, 32)
    want = codes * p.v_scale.astype(np.float64)
    for h in range(4):
        assert np.array_equal(r["out"][0, h], want[h // 2])


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_scores_use_the_k_scale_of_each_channel(fmt):
    # two keys, one query: with s = k_scale the score difference is scale * <q, (c1 - c0) * s>
    p = _quant_problem(fmt, "fp16", past=[1], q_lens=[1], num_heads=1, kv_num_heads=1)
    r = oracle.paged_attention(p)
    kc = r["key_cache"].reshape(p.num_blocks * p.block_size, -1)
    rows = [p.block_table[0, 0] * p.block_size + t for t in range(2)]
    c = [unpack(kc[i], fmt, 32) * p.k_scale[0].astype(np.float64) for i in rows]
    vc = r["value_cache"].reshape(p.num_blocks * p.block_size, -1)
    v = [unpack(vc[i], fmt, 32) * p.v_scale[0].astype(np.float64) for i in rows]
    q = oracle.f16_to_double(p.query[0])
    s = [np.dot(q, ci) / np.sqrt(32) for ci in c]
    a = 1.0 / (1.0 + np.exp(s[0] - s[1]))  # weight of key 1
    assert np.allclose(r["out"][0, 0], (1 - a) * v[0] + a * v[1], rtol=1e-12, atol=1e-14)
    assert np.isclose(r["lse"][0, 0], max(s) + np.log(np.exp(s[0] - max(s)) + np.exp(s[1] - max(s))), rtol=1e-12)


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_cache_write_places_code_rows_and_skips_dropped_slots(fmt):
    p = _quant_problem(fmt, "bf16", past=[3, 0], q_lens=[4, 6], slot_mode="explicit", drop_count=3, packed=True)
    r = oracle.paged_attention(p)
    kr, vr = oracle.kv_rows(p)
    kvh, hs = p.kv_num_heads, p.head_size
    kq = oracle.quantize_rows(kr, "bf16", fmt, kvh, hs, p.k_scale)
    kc0 = p.key_cache.reshape(p.num_blocks * p.block_size, -1)
    kc1 = r["key_cache"].reshape(p.num_blocks * p.block_size, -1)
    written = set()
    for i, slot in enumerate(p.slot_mapping):
        if slot >= 0:
            assert np.array_equal(kc1[slot], kq[i])
            written.add(int(slot))
    for slot in range(kc0.shape[0]):
        if slot not in written:
            assert np.array_equal(kc1[slot], kc0[slot])
