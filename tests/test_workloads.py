"""The seeded generator: determinism, distributions, and the page-table invariants the
WS2 CP-Aware Attention Contract states for decode caches ("Mode-Specific Metadata":
trailing padding, ceil(kv_len / page_size) active pages, no physical page repeated
within a sequence, no page shared across sequences)."""
import numpy as np
import pytest

import workloads as w


def test_streams_are_deterministic_and_independent():
    a = w.u64(5, 1, 100)
    assert np.array_equal(a, w.u64(5, 1, 100))
    assert not np.array_equal(a, w.u64(5, 2, 100))
    assert not np.array_equal(a, w.u64(6, 1, 100))
    assert np.array_equal(w.u64(5, 1, 50, offset=50), a[50:])


def test_normal_and_uniform_moments():
    x = w.normal_f64(1, 1, 400001)
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1) < 0.01
    assert abs(((x - x.mean()) ** 4).mean() / x.var() ** 2 - 3) < 0.05
    u = w.uniform(1, 2, 200000)
    assert u.min() >= 0 and u.max() < 1 and abs(u.mean() - 0.5) < 0.005
    i = w.uniform_int(1, 3, 100000, 512, 4096)
    assert i.min() == 512 and i.max() == 4096


def test_rounded_bits_match_numpy_rounding_of_the_deviates():
    x = w.normal_f64(9, 4, 1001)
    b16 = w.normal_bits(9, 4, (1001,), "fp16")
    assert np.array_equal(b16, x.astype(np.float32).astype(np.float16).view(np.uint16))
    bb = w.normal_bits(9, 4, (1001,), "bf16")
    import torch
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bb, ref)


def _check_pages(p):
    bs = p.block_size
    pages = (p.kv_lens + bs - 1) // bs
    used = []
    for b in range(p.batch_size):
        row = p.block_table[b]
        act = row[: pages[b]]
        assert np.all(act >= 0) and np.all(act < p.num_blocks)
        assert len(set(act.tolist())) == len(act)
        used.extend(act.tolist())
    assert len(set(used)) == len(used)  # no page shared across sequences


@pytest.mark.parametrize("k", [1, 3])
def test_small_configs_shapes_and_pages(k):
    p = w.config(k)
    _check_pages(p)
    if k == 1:
        assert p.num_tokens == 10 and p.num_blocks == 16 and p.block_table.shape == (2, 8)
        assert sorted(p.block_table.ravel().tolist()) == list(range(16))
        q = p.query.view(np.float16).astype(np.float64)
        assert q.min() >= -1 and q.max() <= 1
    if k == 3:
        assert p.num_tokens == 8192 and p.dtype == "bf16" and p.num_blocks == 32
        assert np.all(p.block_table >= 0)


def test_padding_is_trailing_minus_one():
    p = w.make_problem(name="t", seed=1, dtype="fp16", num_heads=4, kv_num_heads=2, head_size=64,
                       block_size=16, past=[0, 40, 3], q_lens=[5, 1, 0], max_blocks_per_sequence=6)
    _check_pages(p)
    pages = (p.kv_lens + 15) // 16
    for b in range(3):
        assert np.all(p.block_table[b, pages[b]:] == -1)


def test_explicit_slots_with_drops():
    p = w.make_problem(name="t", seed=2, dtype="fp16", num_heads=2, kv_num_heads=1, head_size=64,
                       block_size=16, past=[3, 17], q_lens=[20, 10], slot_mode="explicit", drop_count=3)
    assert (p.slot_mapping == -1).sum() == 3
    kept = p.slot_mapping[p.slot_mapping >= 0]
    assert len(set(kept.tolist())) == len(kept)
    assert kept.max() < p.num_blocks * 16
