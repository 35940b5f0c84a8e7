"""Host logic of bench.py on CPU: the DRAM traffic records and the attention byte model.

A traffic record (DRAM bytes per launch from an ncu capture) may only be reported while
the kernel source it was taken on is unchanged; the byte model is the per-unit figure
the roofline divides by (K and V rows read, Q read, output written).
"""
import hashlib
import json
import os

import bench
from speculative_decoding_draft_dflash_gb300 import synth


def _tree(tmp_path, source_text, recorded_hash=None, run="serve_b32/bf16/contiguous"):
    src = tmp_path / "kernel.cu"
    src.write_text(source_text)
    h = recorded_hash or hashlib.sha256(source_text.encode()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    rec = {"runs": {run: {"attention": {"bytes_per_launch": 123.0, "source": "kernel.cu",
                                        "sha256_16": h}}}}
    (tmp_path / "profiles" / "traffic_serve_b32.json").write_text(json.dumps(rec))
    return src


def test_traffic_record_used_while_source_unchanged(tmp_path, monkeypatch):
    _tree(tmp_path, "// kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC_RUN", "serve_b32/bf16/contiguous")
    assert bench.measured_traffic("attention") == 123.0


def test_traffic_record_dropped_after_source_change(tmp_path, monkeypatch):
    src = _tree(tmp_path, "// kernel v1\n")
    src.write_text("// kernel v2\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC_RUN", "serve_b32/bf16/contiguous")
    assert bench.measured_traffic("attention") is None


def test_traffic_record_keyed_by_run_and_kernel(tmp_path, monkeypatch):
    _tree(tmp_path, "// kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC_RUN", "serve_b32/fp8/contiguous")   # other cache type
    assert bench.measured_traffic("attention") is None
    monkeypatch.setattr(bench, "TRAFFIC_RUN", "serve_b32/bf16/contiguous")
    assert bench.measured_traffic("gemm_fc") is None                         # no record


def test_committed_traffic_records_name_existing_sources():
    with open(os.path.join(bench.ROOT, "profiles", "traffic_serve_b32.json")) as f:
        runs = json.load(f)["runs"]
    for run, kernels in runs.items():
        for name, t in kernels.items():
            assert os.path.exists(os.path.join(bench.ROOT, t["source"])), (run, name)
            assert t["bytes_per_launch"] > 0 and len(t["sha256_16"]) == 16


def test_attention_bytes_worked_example():
    """Three sequences of the serving shape (n_kv 8, d_h 128, 32 query heads, block 16) whose
    blocks start at 100, 0 and 5000. Full attention reads keys [0, start + 16): 116 + 16 +
    5016 = 5148 rows at 4096 bytes (K and V, bf16), with a window of 64 keys [start - 63,
    start + 16): 79 + 16 + 79 = 174 rows; Q read and output written are 3 x 16 x 32 x 128
    x 2 bytes each. An fp8 cache halves the K / V bytes only."""
    w = synth.WORKLOADS["serve_b32"].replace(batch=3)
    starts = [100, 0, 5000]
    qo = 2 * 3 * 16 * 32 * 128 * 2                       # 786432
    assert bench.attention_bytes(w, starts) == 5148 * 4096 + qo == 21872640
    assert bench.attention_bytes(w, starts, 64) == 174 * 4096 + qo == 1499136
    assert bench.attention_bytes(w.replace(kv="fp8"), starts) == 5148 * 2048 + qo == 11329536


def test_gemm_roofline_uses_the_burst_peak():
    """A projection GEMM above the ridge point is reported against the burst bf16 peak (its
    launches last tens of microseconds at the maximum clock), with the sustained fraction
    alongside; 85.9 GFLOP in 50 us is 1718 TFLOP/s."""
    pk = {"hbm_gbs": 6784.5, "bf16_tflops": 1954.5, "bf16_tflops_sustained": 1739.5,
          "source": "measured"}
    fl, by = bench.gemm_cost(512, 5 * 4096, 4096)
    kernels = {"gemm_fc": {"avg_us": 50.0}}
    r = bench.roofline_for("gemm_fc", kernels, {"gemm_fc": (fl, by)}, 0, pk)
    assert r["bound"] == "tensor" and r["peak"] == 1954.5
    assert abs(r["achieved"] - fl / 50e-6 / 1e12) < 1e-9
    assert abs(r["frac"] - r["achieved"] / 1954.5) < 1e-12
    assert abs(r["frac_of_sustained"] - r["achieved"] / 1739.5) < 1e-12
    # a weight-streaming GEMM (M = 16) sits below the ridge: HBM-bound
    fl, by = bench.gemm_cost(16, 5 * 4096, 4096)
    r = bench.roofline_for("gemm_fc", {"gemm_fc": {"avg_us": 30.0}}, {"gemm_fc": (fl, by)}, 0, pk)
    assert r["bound"] == "hbm" and r["peak"] == 6784.5
