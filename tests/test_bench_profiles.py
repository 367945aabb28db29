"""The benchmark's use of committed ncu summaries, on CPU: a DRAM traffic figure counts
only while every kernel source its summary was taken on is unchanged."""
import os

import bench


def _tree(tmp_path):
    csrc = tmp_path / "latent_moe_layer_rmsnorm_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cuh").write_text("// kernel a\n")
    (csrc / "b.cuh").write_text("// kernel b\n")
    (tmp_path / "profiles").mkdir()
    return csrc


def _summary(tmp_path, line):
    (tmp_path / "profiles" / "k_w.md").write_text(
        "# summary\n\ntraffic_bytes_per_launch: 1.5e9\n" + line + "\n")


def test_scoped_hash_follows_only_its_files(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_sha(["a.cuh"])
    _summary(tmp_path, f"kernel_source_sha: {h} (a.cuh)")
    assert bench.recorded_traffic("w", "k") == 1.5e9
    (csrc / "b.cuh").write_text("// kernel b, changed\n")     # not covered: still valid
    assert bench.recorded_traffic("w", "k") == 1.5e9
    (csrc / "a.cuh").write_text("// kernel a, changed\n")     # covered: stale
    assert bench.recorded_traffic("w", "k") is None


def test_unscoped_hash_covers_every_file(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _summary(tmp_path, f"kernel_source_sha: {bench.kernel_source_sha()}")
    assert bench.recorded_traffic("w", "k") == 1.5e9
    (csrc / "b.cuh").write_text("// kernel b, changed\n")
    assert bench.recorded_traffic("w", "k") is None


def test_missing_or_unknown_files(tmp_path, monkeypatch):
    _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("w", "k") is None                  # no summary
    _summary(tmp_path, "kernel_source_sha: 0123456789abcdef (gone.cuh)")
    assert bench.recorded_traffic("w", "k") is None                  # file removed


def test_committed_summaries_name_existing_files():
    text = open(os.path.join(os.path.dirname(bench.__file__), "profiles",
                             "gemm1_gate_up_swiglu_prefill_bf16.md")).read()
    line = [ln for ln in text.splitlines() if ln.startswith("kernel_source_sha:")][0]
    files = line[line.index("(") + 1: line.index(")")].split()
    csrc = os.path.join(os.path.dirname(bench.__file__), "latent_moe_layer_rmsnorm_gb300",
                        "csrc")
    assert files and all(os.path.exists(os.path.join(csrc, f)) for f in files)
