"""GPU parity: the CUDA path through the C ABI against the oracle.

Caches must match bit for bit (the write is a copy); outputs must satisfy
|gpu - oracle| <= 2e-3 + 1e-2 |oracle| elementwise, the oracle taken in fp64 before
rounding. Every case, the full-size workloads included, is checked on every cache byte
and every output element.
"""
import numpy as np
import pytest
import torch

import oracle
import varlen_paged_kv_gb300 as pa
import workloads as w
from gpu_utils import assert_close, bits_of, make_workspace, run_gpu, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is required for the gpu tests")
    from varlen_paged_kv_gb300 import build
    build.build()


def check(p, **opts):
    ref = oracle.paged_attention(p)
    r = run_gpu(p, **opts)
    assert r["err"] == 0, f"device error bits {r['err']}"
    assert np.array_equal(r["key_cache"], ref["key_cache"]), "key cache differs"
    assert np.array_equal(r["value_cache"], ref["value_cache"]), "value cache differs"
    N, nh, hs = p.num_tokens, p.num_heads, p.head_size
    assert_close(r["out_bits"].reshape(N, nh, hs), ref["out"], p.dtype, p.name)
    return r, ref


# ---- the tiny workload ----------------------------------------------------------------

def test_tiny_workload_auto_route():
    check(w.config(1))


def test_tiny_workload_on_the_prefill_kernel():
    check(w.config(1), route=pa.ROUTE_ALL_PREFILL)


def test_tiny_workload_forced_splits():
    check(w.config(1), decode_split_keys=64)


# ---- shapes spanning tiles, ragged tails, page sizes and routes --------------------------

CASES = {
    # name: (dtype, nh, kvh, hs, bs, past, q_lens, packed, explicit_slots_with_drops)
    "decode-single-split": ("fp16", 32, 8, 128, 256, [0, 5, 300, 1000], [1, 1, 1, 1], False, 0),
    "decode-q-up-to-4": ("bf16", 32, 8, 128, 16, [4000, 0, 17], [1, 3, 4], False, 0),
    "decode-mha-q16": ("fp16", 8, 8, 64, 32, [100, 33], [16, 7], False, 0),
    "decode-gqa16": ("bf16", 16, 1, 128, 64, [500, 1], [1, 1], False, 0),
    "prefill-ragged": ("bf16", 32, 8, 128, 256, [0, 0], [300, 129], False, 0),
    "chunked-prefill": ("fp16", 32, 8, 128, 256, [1000, 17, 255], [200, 64, 513], False, 0),
    "mixed-packed-drops": ("fp16", 32, 8, 128, 256, [0, 900, 50, 3000], [130, 1, 40, 2], True, 9),
    "head64-pages16": ("fp16", 4, 2, 64, 16, [0, 5, 20, 100], [70, 3, 7, 1], False, 0),
    "pages48": ("bf16", 8, 2, 128, 48, [100, 0], [50, 1], False, 0),
    "pages512": ("fp16", 16, 4, 128, 512, [700], [300], False, 0),
    "empty-sequences": ("fp16", 8, 2, 128, 32, [5, 0, 10, 7], [0, 9, 0, 1], False, 0),
    "gqa8-q2": ("bf16", 32, 4, 128, 16, [60], [2], False, 0),
    "rows-over-16-go-prefill": ("fp16", 32, 8, 128, 32, [40], [5], True, 0),
    "bf16-long-history-chunk": ("bf16", 8, 2, 128, 128, [2500], [257], False, 0),
    # explicit slots with drops: the fp16 V copy is made by its own kernel after the cache write
    "bf16-prefill-explicit-slots": ("bf16", 16, 4, 128, 64, [300, 0, 70], [200, 129, 1], False, 7),
}


def _case(name, seed=7):
    dt, nh, kvh, hs, bs, past, q, packed, drops = CASES[name]
    return w.make_problem(name=name, seed=seed, dtype=dt, num_heads=nh, kv_num_heads=kvh, head_size=hs,
                          block_size=bs, past=past, q_lens=q, packed=packed,
                          slot_mode="explicit" if drops else "omitted", drop_count=drops, num_blocks=None)


@pytest.mark.parametrize("name", sorted(CASES))
def test_cases_auto_route(name):
    check(_case(name))


@pytest.mark.parametrize("name", sorted(CASES))
def test_cases_prefill_route(name):
    check(_case(name), route=pa.ROUTE_ALL_PREFILL)


@pytest.mark.parametrize("split", [64, 128, 448])
@pytest.mark.parametrize("name", ["decode-q-up-to-4", "decode-single-split", "decode-gqa16", "mixed-packed-drops"])
def test_decode_split_lengths(name, split):
    check(_case(name), decode_split_keys=split)


def test_scale_attribute_including_negative():
    for scale in (0.05, -0.3):
        p = _case("chunked-prefill")
        p.scale = scale
        check(p)
        p = _case("decode-q-up-to-4")
        p.scale = scale
        check(p)


# ---- invariants on the GPU ------------------------------------------------------------------

def test_bitwise_deterministic():
    for name in ("mixed-packed-drops", "chunked-prefill"):
        p = _case(name)
        a = run_gpu(p, decode_split_keys=128)
        b = run_gpu(p, decode_split_keys=128)
        assert np.array_equal(a["out_bits"], b["out_bits"])


def test_physical_page_permutation_is_bitwise_invisible():
    p = _case("chunked-prefill")
    perm = np.random.default_rng(3).permutation(p.num_blocks)
    q = p.copy()
    q.key_cache = np.empty_like(p.key_cache)
    q.value_cache = np.empty_like(p.value_cache)
    q.key_cache[perm] = p.key_cache
    q.value_cache[perm] = p.value_cache
    q.block_table = np.where(p.block_table >= 0, perm[np.maximum(p.block_table, 0)], -1).astype(np.int32)
    a = run_gpu(p)
    b = run_gpu(q)
    assert np.array_equal(a["out_bits"], b["out_bits"])


def test_packed_qkv_bitwise_equals_separate():
    p = _case("chunked-prefill")
    q = p.copy()
    q.query = np.concatenate([p.query, p.key, p.value], axis=1)
    q.key = q.value = None
    a = run_gpu(p)
    b = run_gpu(q)
    assert np.array_equal(a["out_bits"], b["out_bits"])
    assert np.array_equal(a["key_cache"], b["key_cache"]) and np.array_equal(a["value_cache"], b["value_cache"])


def test_single_token_without_history_returns_its_own_v_bitwise():
    p = w.make_problem(name="t", seed=5, dtype="bf16", num_heads=8, kv_num_heads=2, head_size=128, block_size=16,
                       past=[0, 0, 0], q_lens=[1, 1, 1])
    for route in (pa.ROUTE_AUTO, pa.ROUTE_ALL_PREFILL):
        r = run_gpu(p, route=route)
        out = r["out_bits"].reshape(3, 8, 128)
        v = p.value.reshape(3, 2, 128)
        for h in range(8):
            assert np.array_equal(out[:, h], v[:, h // 4])


# ---- full-size workloads: every cache byte and every output element ------------------------
# Each of the four full-size workloads runs in the launch configuration bench.py times (the
# caller's bound on new tokens per sequence, max_query_len, passed as the bench passes it:
# the decode-only batches then take the self-planned decode kernel) and, for the decode-only
# ones, also without the bound (planner, cache-write and decode kernels). The oracle computes
# the whole workload once per module.

_FULL_REF = {}


def _full_ref(k):
    if k not in _FULL_REF:
        _FULL_REF[k] = oracle.paged_attention(w.config(k))
    return _FULL_REF[k]


@pytest.mark.parametrize("k,bounded", [(2, True), (2, False), (3, True), (4, True), (5, True), (5, False)])
def test_full_size_workload(k, bounded):
    p = w.config(k)
    ref = _full_ref(k)
    r = run_gpu(p, max_query_len=int(p.q_lens.max()) if bounded else 0)
    assert r["err"] == 0, f"device error bits {r['err']}"
    assert np.array_equal(r["key_cache"], ref["key_cache"]), "key cache differs"
    assert np.array_equal(r["value_cache"], ref["value_cache"]), "value cache differs"
    N, nh, hs = p.num_tokens, p.num_heads, p.head_size
    assert_close(r["out_bits"].reshape(N, nh, hs), ref["out"], p.dtype, p.name)


def test_max_query_len_hint_skips_prefill_and_is_checked():
    p = _case("decode-q-up-to-4")  # q_len <= 4, G = 4: every sequence decode-class
    ref = oracle.paged_attention(p)
    d = upload(p)
    ws = make_workspace(p)
    n0 = pa.kernel_launch_count()
    out = pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                             d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], None,
                             num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, workspace=ws, max_query_len=4)
    assert pa.read_device_error(ws) == 0
    assert pa.kernel_launch_count() - n0 == 2  # the counters' reset, the self-planned decode kernel
    assert_close(bits_of(out).reshape(p.num_tokens, p.num_heads, p.head_size), ref["out"], p.dtype, "hint")
    # a bound below the real q_len is refused on the device, nothing written
    d = upload(p)
    pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                       d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], None,
                       num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, workspace=ws, max_query_len=2)
    assert pa.read_device_error(ws) & pa.DEVERR_BAD_BATCH
    assert np.array_equal(bits_of(d["key_cache"]), p.key_cache)


def test_balanced_partition_splits_long_units_across_ctas():
    # two sequences with long histories and many short ones: the long units are cut across
    # several CTAs and merged by the last one; results must not depend on the cut
    past = [60000, 5, 17, 33000, 300, 1, 2, 3]
    p = w.make_problem(name="skew", seed=9, dtype="bf16", num_heads=16, kv_num_heads=4, head_size=128,
                       block_size=16, past=past, q_lens=[1, 2, 1, 3, 1, 4, 1, 1])
    check(p)
    a = run_gpu(p)
    b = run_gpu(p)
    assert np.array_equal(a["out_bits"], b["out_bits"])


# A whole call with prefill-class and decode-class rows runs the two attention kernels at the
# same time on SMs the planner splits between them (pa_dims.decode_sms fixes the decode share).
# Results must not depend on the split, from one decode SM to all but one.
MIXED = {
    "mixed-packed-drops": lambda: _case("mixed-packed-drops"),
    "mixed-long-decode-bf16": lambda: w.make_problem(
        name="mixed-long-decode-bf16", seed=13, dtype="bf16", num_heads=32, kv_num_heads=8, head_size=128,
        block_size=16, past=[9000, 0, 4000, 700, 12000, 33], q_lens=[1, 300, 2, 1, 4, 129]),
    "mixed-head64": lambda: w.make_problem(
        name="mixed-head64", seed=14, dtype="fp16", num_heads=8, kv_num_heads=2, head_size=64,
        block_size=32, past=[2000, 10, 0], q_lens=[1, 200, 3]),
}


@pytest.mark.parametrize("dsm", [0, 1, 5, 76, 151, 4096])
@pytest.mark.parametrize("name", sorted(MIXED))
def test_mixed_batches_on_split_sms(name, dsm):
    check(MIXED[name](), decode_sms=dsm)


def test_split_sms_are_bitwise_deterministic():
    p = MIXED["mixed-long-decode-bf16"]()
    a = run_gpu(p)
    b = run_gpu(p)
    assert np.array_equal(a["out_bits"], b["out_bits"])


# ---- device-side error reporting (no faults) ----------------------------------------------------

def test_out_of_range_block_is_reported_and_read_as_zeros():
    p = _case("decode-q-up-to-4")
    p.block_table = p.block_table.copy()
    p.block_table[0, 0] = 10 ** 6
    r = run_gpu(p)
    assert r["err"] & pa.DEVERR_BAD_BLOCK


def test_errors_of_a_copy_beside_the_planner_are_kept():
    # fp16 bit copies run beside this call's planner, which resets the error word: their
    # bad-block and bad-slot bits are added only after it
    p = _case("chunked-prefill")
    p.block_table = p.block_table.copy()
    p.block_table[1, 0] = 10 ** 6
    assert run_gpu(p)["err"] & pa.DEVERR_BAD_BLOCK
    q = _case("mixed-packed-drops")
    q.slot_mapping = q.slot_mapping.copy()
    live = int(np.flatnonzero(q.slot_mapping >= 0)[0])
    q.slot_mapping[live] = q.num_blocks * q.block_size + 5
    assert run_gpu(q)["err"] & pa.DEVERR_BAD_SLOT


@pytest.mark.parametrize("name", ["chunked-prefill", "bf16-long-history-chunk"])
def test_inconsistent_batch_is_refused_without_writes(name):
    # (fp16: the bit copy beside the planner; bf16 with derived slots: the one that also
    # makes the fp16 V copy)
    p = _case(name)
    p.cumulative_sequence_length = p.cumulative_sequence_length.copy()
    p.cumulative_sequence_length[-1] -= 1  # does not end at num_tokens
    d = upload(p)
    before = bits_of(d["key_cache"]).copy()
    before_v = bits_of(d["value_cache"]).copy()
    ws = make_workspace(p)
    out = torch.full((p.num_tokens, p.num_heads * p.head_size), 7.0, dtype=d["query"].dtype, device="cuda")
    pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                       d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], None,
                       num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, output=out, workspace=ws)
    assert pa.read_device_error(ws) & pa.DEVERR_BAD_BATCH
    assert np.array_equal(bits_of(d["key_cache"]), before)
    assert np.array_equal(bits_of(d["value_cache"]), before_v)
    assert torch.all(out == 7.0)


# ---- bf16 V outside fp16's range, and unwritten cache rows --------------------------------

def _scale_bf16_rows(bits, rows, exp_shift):
    """Replaces the bf16 values v of the given rows by |v| * 2**exp_shift, exactly (sign bit
    and exponent field)."""
    out = bits.copy()
    sel = out[rows].astype(np.int32) & 0x7FFF
    nonzero = (sel & 0x7F80) != 0
    sel = np.where(nonzero, sel + (exp_shift << 7), sel)
    assert np.all((sel & 0x7F80) < 0x7F80) and np.all(sel >= 0)  # stays finite, no sign flip
    out[rows] = sel.astype(np.uint16)
    return out


def test_bf16_values_beyond_fp16_range():
    # sequence 0 has three 128-key tiles; six of its tokens in the middle tile get values
    # 2^17 |N(0,1)|, mostly beyond fp16's largest finite value, while the other tiles stay
    # small, so one unit mixes both kinds of tile. The large values are all positive: with
    # both signs the outputs would be small differences of terms near 1e5, and no fp32
    # computation meets a tolerance relative to such a difference.
    p = _case("prefill-ragged")
    assert p.dtype == "bf16"
    p.value = _scale_bf16_rows(p.value, np.arange(130, 136), 17)
    check(p)
    check(p, route=pa.ROUTE_ALL_PREFILL)


def _poison_unread_cache_rows(p, bits):
    """Sets every cache row no sequence reads (past its length, or in pages it does not
    own) to the 16-bit pattern `bits` in both caches."""
    used = np.zeros((p.num_blocks, p.block_size), bool)
    for b in range(p.batch_size):
        keys = np.arange(int(p.kv_lens[b]))
        used[p.block_table[b, keys // p.block_size], keys % p.block_size] = True
    p.key_cache = p.key_cache.copy()
    p.value_cache = p.value_cache.copy()
    p.key_cache[~used] = bits
    p.value_cache[~used] = bits


@pytest.mark.parametrize("name", ["prefill-ragged", "chunked-prefill", "pages48", "head64-pages16"])
def test_nan_in_unread_cache_rows_does_not_leak(name):
    # the last KV tile of a sequence reaches past its length into cache rows that may never
    # have been written; P is 0 there, but 0 * NaN is NaN, so those rows must not reach P V
    p = _case(name)
    _poison_unread_cache_rows(p, 0x7FC0 if p.dtype == "bf16" else 0x7E00)
    check(p)
    check(p, route=pa.ROUTE_ALL_PREFILL)


# ---- shared-prefix pages: several block_table rows point at the same physical pages ----

def _share_prefix(p, seqs, n_pages):
    """Makes sequences `seqs` read their first n_pages logical pages from seqs[0]'s physical
    pages (a read-only shared prefix; every sequence's history must cover those pages, so
    this call's writes land in pages of its own)."""
    bt = p.block_table.copy()
    for b in seqs:
        assert int(p.past_seqlens[b]) >= n_pages * p.block_size
        bt[b, :n_pages] = bt[seqs[0], :n_pages]
    p.block_table = bt
    return p


@pytest.mark.parametrize("route", [pa.ROUTE_AUTO, pa.ROUTE_ALL_PREFILL])
def test_shared_prefix_pages_decode(route):
    p = w.make_problem(name="shared-decode", seed=31, dtype="fp16", num_heads=32, kv_num_heads=8, head_size=128,
                       block_size=64, past=[600, 700, 640, 1000], q_lens=[1, 2, 1, 4])
    check(_share_prefix(p, [0, 1, 2, 3], 9), route=route)
    check(p, decode_split_keys=128)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_shared_prefix_pages_chunked_prefill(dtype):
    # three chunks continuing one 512-token prompt prefix held once in the pool
    p = w.make_problem(name="shared-prefill", seed=32, dtype=dtype, num_heads=16, kv_num_heads=4, head_size=128,
                       block_size=256, past=[512, 512, 768], q_lens=[100, 200, 17])
    check(_share_prefix(p, [0, 1, 2], 2))


# ---- decode-only batches run with the max_query_len bound ----

def _run_hinted(p, split=0, ws=None):
    d = upload(p)
    ws = make_workspace(p, split) if ws is None else ws
    out = pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                             d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], d["slot_mapping"],
                             num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, scale=p.scale,
                             decode_split_keys=split, workspace=ws, max_query_len=int(p.q_lens.max()))
    return d, out, ws


@pytest.mark.parametrize("split", [0, 64])
@pytest.mark.parametrize("name", ["decode-single-split", "decode-q-up-to-4", "decode-gqa16", "gqa8-q2"])
def test_decode_only_batches_with_the_query_bound(name, split):
    # max_query_len <= 4 proves these batches decode-only (no prefill launch)
    p = _case(name)
    assert int(p.q_lens.max()) <= 4 and p.slot_mapping is None
    ref = oracle.paged_attention(p)
    d, out, ws = _run_hinted(p, split)
    assert pa.read_device_error(ws) == 0
    assert np.array_equal(bits_of(d["key_cache"]), ref["key_cache"]), "key cache differs"
    assert np.array_equal(bits_of(d["value_cache"]), ref["value_cache"]), "value cache differs"
    assert_close(bits_of(out).reshape(p.num_tokens, p.num_heads, p.head_size), ref["out"], p.dtype, name)


def test_refused_batch_runs_no_stale_plan():
    # a workspace left holding a valid plan must not let a refused batch write or compute
    p = _case("decode-q-up-to-4")
    _, _, ws = _run_hinted(p)
    bad = _case("decode-q-up-to-4")
    bad.cumulative_sequence_length = bad.cumulative_sequence_length.copy()
    bad.cumulative_sequence_length[-1] -= 1
    d = upload(bad)
    before = bits_of(d["key_cache"]).copy(), bits_of(d["value_cache"]).copy()
    out = torch.full((bad.num_tokens, bad.num_heads * bad.head_size), 7.0, dtype=d["query"].dtype, device="cuda")
    pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                       d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], None,
                       num_heads=bad.num_heads, kv_num_heads=bad.kv_num_heads, output=out, workspace=ws,
                       max_query_len=int(bad.q_lens.max()))
    assert pa.read_device_error(ws) & pa.DEVERR_BAD_BATCH
    assert np.array_equal(bits_of(d["key_cache"]), before[0]) and np.array_equal(bits_of(d["value_cache"]), before[1])
    assert torch.all(out == 7.0)


# ---- decode-only batches the decode kernel plans itself -------------------------------------
# A whole call whose host bound proves every sequence decode-class, with derived slots and at
# most 256 sequences, runs no planner and no cache-write kernel: each decode CTA cuts its share
# of the partition from the batch description and writes the new K/V rows of the tiles it loads.
SELF = {
    "self-gqa4-pages16": dict(dtype="fp16", num_heads=32, kv_num_heads=8, head_size=128, block_size=16,
                              past=list(range(0, 4000, 100)), q_lens=[1 + (i % 4) for i in range(40)]),
    "self-mha-q16-hs64": dict(dtype="bf16", num_heads=8, kv_num_heads=8, head_size=64, block_size=32,
                              past=[0, 31, 32, 500, 1023], q_lens=[16, 1, 16, 7, 2]),
    "self-gqa8-empty-seqs": dict(dtype="bf16", num_heads=16, kv_num_heads=2, head_size=128, block_size=64,
                                 past=[5, 0, 300, 0, 63, 1000], q_lens=[0, 1, 2, 0, 1, 2]),
    "self-skewed-long": dict(dtype="fp16", num_heads=32, kv_num_heads=8, head_size=128, block_size=16,
                             past=[60000, 3, 100000, 0, 17, 5000], q_lens=[1, 1, 2, 1, 1, 1]),
    "self-256-seqs": dict(dtype="fp16", num_heads=16, kv_num_heads=2, head_size=128, block_size=256,
                          past=[(37 * i) % 2000 for i in range(256)], q_lens=[1] * 256),
}


@pytest.mark.parametrize("name", sorted(SELF))
def test_self_planned_decode_only_batches(name):
    p = w.make_problem(name=name, seed=21, **SELF[name])
    ref = oracle.paged_attention(p)
    d = upload(p)
    ws = make_workspace(p)
    lse = torch.empty((p.num_tokens, p.num_heads), dtype=torch.float32, device="cuda")
    n0 = pa.kernel_launch_count()
    out = pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                             d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], None,
                             num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, workspace=ws,
                             max_query_len=int(p.q_lens.max()), lse=lse)
    assert pa.kernel_launch_count() - n0 == 2
    assert pa.read_device_error(ws) == 0
    assert np.array_equal(bits_of(d["key_cache"]), ref["key_cache"]), "key cache differs"
    assert np.array_equal(bits_of(d["value_cache"]), ref["value_cache"]), "value cache differs"
    assert_close(bits_of(out).reshape(p.num_tokens, p.num_heads, p.head_size), ref["out"], p.dtype, name)
    lg = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lg - ref["lse"]) <= 5e-4 + 1e-5 * np.abs(ref["lse"])), "lse differs"


def test_self_planned_calls_repeat_bitwise():
    # the merge counters are reset by each call: a second call on the same workspace gives the
    # same bits
    p = w.make_problem(name="self-skewed-long", seed=22, **SELF["self-skewed-long"])
    d = upload(p)
    ws = make_workspace(p)
    outs = []
    for _ in range(3):
        outs.append(bits_of(pa.paged_attention(
            d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"], d["cumulative_sequence_length"],
            d["past_seqlens"], d["block_table"], None, num_heads=p.num_heads, kv_num_heads=p.kv_num_heads,
            workspace=ws, max_query_len=int(p.q_lens.max()))))
    assert pa.read_device_error(ws) == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


# ---- batches larger than one planner round (1024 sequences) and than the tile sort ----

def test_many_sequences_mixed_across_planner_rounds():
    # 2600 sequences: decode rows with short histories plus prefill-class chunks spread over
    # all three planner rounds (carries of the scans, item indices, the V-copy layout)
    B = 2600
    past = w.uniform_int(41, 1, B, 0, 200)
    q = np.where(np.arange(B) % 97 == 5, 40, 1).astype(np.int64)
    p = w.make_problem(name="many-mixed", seed=41, dtype="bf16", num_heads=8, kv_num_heads=2, head_size=64,
                       block_size=16, past=past, q_lens=q)
    check(p)


def test_more_prefill_tiles_than_the_sort_holds():
    # 4200 prefill-class sequences (q_len 5, 4 query heads per KV head: 20 rows) make 4200
    # query tiles, past the planner's 4096-entry sort: the tiles run in list order
    B = 4200
    past = w.uniform_int(42, 1, B, 0, 40)
    p = w.make_problem(name="many-tiles", seed=42, dtype="fp16", num_heads=8, kv_num_heads=2, head_size=64,
                       block_size=16, past=past, q_lens=np.full(B, 5, np.int64))
    check(p)


# ---- a call split into stage groups runs the whole call's program ----------------------------

@pytest.mark.parametrize("name,max_q,groups", [
    ("decode-q-up-to-4", 4, [pa.STAGE_PLAN | pa.STAGE_CACHE_WRITE, pa.STAGE_DECODE]),  # self-planned
    ("decode-q-up-to-4", 4, [pa.STAGE_PLAN, pa.STAGE_CACHE_WRITE, pa.STAGE_PREFILL, pa.STAGE_DECODE]),
    ("mixed-packed-drops", 0, [pa.STAGE_PLAN | pa.STAGE_CACHE_WRITE, pa.STAGE_PREFILL | pa.STAGE_DECODE]),
    ("mixed-packed-drops", 0, [pa.STAGE_PLAN, pa.STAGE_CACHE_WRITE, pa.STAGE_PREFILL, pa.STAGE_DECODE]),
    ("bf16-long-history-chunk", 0, [pa.STAGE_PLAN | pa.STAGE_CACHE_WRITE, pa.STAGE_PREFILL, pa.STAGE_DECODE]),
])
def test_stage_split_calls_match_the_whole_call(name, max_q, groups):
    p = _case(name)
    whole = run_gpu(p, max_query_len=max_q)
    d = upload(p)
    ws = make_workspace(p, 0, pa.ROUTE_AUTO, max_q)
    out = torch.empty((p.num_tokens, p.num_heads * p.head_size), dtype=d["query"].dtype, device="cuda")
    for st in groups:
        pa.paged_attention(d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"],
                           d["cumulative_sequence_length"], d["past_seqlens"], d["block_table"], d["slot_mapping"],
                           num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, scale=p.scale, output=out,
                           workspace=ws, max_query_len=max_q, stages=st)
    assert pa.read_device_error(ws) == 0
    assert np.array_equal(bits_of(d["key_cache"]), whole["key_cache"])
    assert np.array_equal(bits_of(d["value_cache"]), whole["value_cache"])
    # the split-SM program of a mixed batch runs its two attention kernels side by side only
    # when one call launches both; the partition and the arithmetic are the same either way
    assert np.array_equal(bits_of(out), whole["out_bits"])
