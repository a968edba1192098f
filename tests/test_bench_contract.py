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
