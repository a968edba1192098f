"""bench.py's JSON line (CPU: the oracle arm on the tiny workload) and its host helpers."""
import json
import subprocess
import sys
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--tokens", "16", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_layer_work_counts():
    from mixture_experts_layer_05_gb300 import configs
    w = configs.MIXTRAL
    work = bench.layer_work(w, 4096, 8)
    assert work["flops_w13"] == 4.0 * 4096 * 2 * 4096 * 14336
    assert work["flops"] == 6.0 * 4096 * 2 * 4096 * 14336
    assert work["bytes"] > 8 * 3 * 4096 * 14336 * 2          # at least every weight once


def test_traffic_lookup_needs_matching_source():
    assert bench.kernel_traffic("gemm_w13", "no-such-workload", 1) is None


def test_source_digest_ignores_comments_not_code(tmp_path, monkeypatch):
    """The traffic digest keys on code: a comment-only edit keeps it, a code edit changes it."""
    csrc = tmp_path / "mixture_experts_layer_05_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src_dir = os.path.join(ROOT, "mixture_experts_layer_05_gb300", "csrc")
    for name in bench.KERNEL_SOURCES["gemm.cu"]:
        (csrc / name).write_text(open(os.path.join(src_dir, name)).read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d0 = bench.source_digest("gemm.cu")
    common = csrc / "common.cuh"
    text = common.read_text()
    common.write_text("// a new comment line\n" + text.replace("\n", "  // trailing note\n", 1))
    assert bench.source_digest("gemm.cu") == d0
    common.write_text(text + "\nconstexpr int kDigestProbe = 1;\n")
    assert bench.source_digest("gemm.cu") != d0


def test_roofline_picks_the_binding_bound():
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    # 1.9 TFLOP and 1 GB in 2 ms: tensor time 1 ms > HBM time 0.147 ms -> tensor, frac 0.5
    r = bench.roofline_of({"flops_w13": 1.9e12, "bytes_w13": 1e9}, 2e-3, peaks, "measured",
                          "none", "k")
    assert r["bound"] == "tensor" and abs(r["frac"] - 0.5) < 1e-9
    assert abs(r["tensor_frac_of_sustained"] - 950.0 / 1700.0) < 1e-4
    assert abs(r["ridge_frac"] - 0.5) < 1e-9
    # 1.9 GFLOP and 13.6 GB in 4 ms: HBM time 2 ms -> hbm, frac 0.5
    r = bench.roofline_of({"flops_w13": 1.9e9, "bytes_w13": 13.6e9}, 4e-3, peaks, "measured",
                          "none", "k")
    assert r["bound"] == "hbm" and abs(r["frac"] - 0.5) < 1e-9
    # e4m3: the tensor peak doubles
    r = bench.roofline_of({"flops_w13": 3.8e12, "bytes_w13": 1e9}, 2e-3, peaks, "measured",
                          "fp8", "k")
    assert r["bound"] == "tensor" and abs(r["frac"] - 0.5) < 1e-9
    # nvfp4: six times the bf16 peak (13.5 / 2.25 nominal)
    r = bench.roofline_of({"flops_w13": 11.4e12, "bytes_w13": 1e9}, 2e-3, peaks, "measured",
                          "nvfp4", "k")
    assert r["bound"] == "tensor" and abs(r["frac"] - 0.5) < 1e-9
