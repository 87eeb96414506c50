"""Host-side logic of bench.py that needs no GPU.

The DRAM traffic a bench line reports comes from one ncu capture per (kernel, workload),
kept with a hash of the kernel's sources at capture time; it is reported only while the
sources hash the same. The hash leaves out line comments and trailing blanks: a comment
edit keeps the counters, a code edit drops them.
"""
import os
import shutil

import bench


def _copy_sources(tmp_path):
    src = os.path.join(bench.ROOT, "varlen_paged_kv_gb300", "csrc")
    dst = tmp_path / "varlen_paged_kv_gb300" / "csrc"
    shutil.copytree(src, dst)
    return dst


def test_comment_edits_keep_the_hash_code_edits_change_it(tmp_path, monkeypatch):
    before = {k: bench.source_hash(k) for k in bench.KERNEL_SOURCES}
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert {k: bench.source_hash(k) for k in bench.KERNEL_SOURCES} == before
    p = dst / "decode.cu"
    text = p.read_text()
    p.write_text("// a note\n" + text.replace("\n", "  // note\n", 3) + "\n\n")
    assert bench.source_hash("decode_kernel_self") == before["decode_kernel_self"]
    assert bench.source_hash("prefill_kernel") == before["prefill_kernel"]
    p.write_text(text.replace("kDecTile", "kDecTile ", 1) + "int unused_marker;\n")
    assert bench.source_hash("decode_kernel_self") != before["decode_kernel_self"]
    assert bench.source_hash("prefill_kernel") == before["prefill_kernel"]  # (another kernel's files)


def test_traffic_is_dropped_when_the_sources_change(tmp_path, monkeypatch):
    key = next(iter(bench.NCU_TRAFFIC))
    kernel, name = key
    bytes_, digest = bench.NCU_TRAFFIC[key]
    monkeypatch.setitem(bench.NCU_TRAFFIC, key, (bytes_, bench.source_hash(kernel)))
    assert bench.ncu_traffic(kernel, name) == bytes_
    monkeypatch.setitem(bench.NCU_TRAFFIC, key, (bytes_, "0" * 16))
    assert bench.ncu_traffic(kernel, name) is None
    assert bench.ncu_traffic(kernel, "no-such-workload") is None
