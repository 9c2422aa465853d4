"""bench.py reports a kernel's DRAM traffic from a committed ncu summary only
while that summary was taken on the current kernel source: the source hash
ignores comments and blank space, and any change to the code voids it."""

import os
import shutil

import bench

FILES = ("decode.cu", "decode_fp16.cu", "pa_internal.cuh")


def _tree(tmp_path):
    csrc = tmp_path / "paged_kv_attention_prepare_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in FILES:
        shutil.copy(os.path.join(bench.ROOT, "paged_kv_attention_prepare_gb300", "csrc", name),
                    csrc / name)
    (tmp_path / "profiles").mkdir()
    return csrc


def test_hash_ignores_comments_and_blank_space(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    p = csrc / "decode.cu"
    text = p.read_text()
    p.write_text("// a new comment line\n" + text.replace("\n", "\n\n", 3) + "\n/* block\ncomment */\n")
    assert bench.kernel_source_hash() == h0


def test_hash_changes_with_the_code(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    p = csrc / "pa_internal.cuh"
    p.write_text(p.read_text() + "\nconstexpr int kProbe = 1;\n")
    assert bench.kernel_source_hash() != h0


def test_recorded_traffic_only_for_the_current_source(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    prof = tmp_path / "profiles" / "paged_decode_kernel_probe.txt"
    prof.write_text(f"kernel_source_hash: {bench.kernel_source_hash()}  (comments removed)\n"
                    "dram_bytes_per_launch: 123456789\n")
    assert bench.recorded_traffic("probe") == 123456789.0
    assert bench.recorded_traffic("absent") is None
    p = csrc / "decode.cu"
    p.write_text(p.read_text() + "\nstatic int probe_variable = 0;\n")
    assert bench.recorded_traffic("probe") is None


def test_committed_summaries_name_hash_and_bytes():
    # every committed split-K summary carries the two lines bench.py reads
    pdir = os.path.join(bench.ROOT, "profiles")
    names = [n for n in os.listdir(pdir) if n.startswith("paged_decode_kernel_")]
    assert names
    for n in names:
        text = open(os.path.join(pdir, n)).read()
        assert "kernel_source_hash:" in text and "dram_bytes_per_launch:" in text, n
