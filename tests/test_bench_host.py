"""Host-side logic of bench.py that needs no GPU: the per-kernel source hashes that gate the
ncu traffic figure, and the lookup of that figure in a profile table."""
import os

import bench


def test_kernel_sources_exist():
    csrc = os.path.join(bench.ROOT, "forget_gated_softmax_gb300", "csrc")
    for kernel, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(csrc, f)), (kernel, f)


def test_kernel_source_hash_is_per_kernel_and_stable():
    hf, hb = bench.kernel_source_hash("attn_fwd"), bench.kernel_source_hash("attn_bwd")
    assert len(hf) == 12 and len(hb) == 12 and int(hf, 16) >= 0 and int(hb, 16) >= 0
    assert hf != hb
    assert hf == bench.kernel_source_hash("attn_fwd")


def test_code_only_ignores_comments_and_layout():
    a = "int x = 1;  // one\n/* block\n comment */\nint  y=2;\n"
    b = "int x = 1;\n\nint  y=2;   // two\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only("int x = 2;\nint y = 2;\n")


def test_ncu_traffic_only_for_matching_source(tmp_path, monkeypatch):
    h = bench.kernel_source_hash("attn_bwd")
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "ncu_traffic.md").write_text(
        "| kernel | workload | dram bytes per launch | source hash |\n|---|---|---|---|\n"
        f"| attn_bwd | wl | 123456 | {h} |\n| attn_fwd | wl | 777 | 000000000000 |\n"
    )
    # the lookup reads profiles/ under ROOT; the sources' hashes are pinned to the table's
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: {"attn_bwd": h}.get(k, "x"))
    assert bench.ncu_traffic("attn_bwd", "wl") == 123456.0
    assert bench.ncu_traffic("attn_fwd", "wl") is None  # taken on other code
    assert bench.ncu_traffic("attn_bwd", "other") is None
