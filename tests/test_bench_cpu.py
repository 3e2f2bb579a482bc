"""bench.py's reference arm on one rank, CPU only: the JSON line carries every
key the benchmark line needs, with the oracle's own figures in value,
cpu_baseline and e2e (no host-device copies)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_line_has_every_key():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
           "--warmup", "3", "--workload", "f32_b1_h1_t256_k64_v64"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["n_gpus"] == 1
    assert d["steps"] == 3 and d["warmup"] >= 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["data"] == "synthetic"
    assert d["config"]["workload"] == "f32_b1_h1_t256_k64_v64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert isinstance(cb["sample"], str) and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_step_statistics_and_roofline_arithmetic():
    """The headline uses the median step; p10/p90 bracket it; the pipeline
    roofline fraction is max(flops / peak, bytes / HBM) over the step time."""
    sys.path.insert(0, ROOT)
    import bench
    from gated_delta_rule_35_gb300.inputs import WORKLOADS

    st = bench.step_stats([5.0, 1.0, 2.0, 4.0, 3.0, 100.0, 2.5, 3.5, 4.5, 1.5, 2.2])
    assert st["median_ms"] == 3.0 and st["steps"] == 11
    assert st["p10_ms"] <= st["median_ms"] <= st["p90_ms"] < 100.0
    assert st["min_ms"] == 1.0 and st["max_ms"] == 100.0
    w = WORKLOADS["bf16_b8_h64_t8192_k128_v128"]
    peaks = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "_source": "test"}
    r = bench.pipeline_roofline(w, 2e-3, peaks, False)
    units = w.B * w.T * w.H
    nbytes = 1032 * units + w.B * w.H * w.K * w.V * 4
    assert r["bytes"] == nbytes and r["bound"] == "hbm"
    assert abs(r["frac"] - nbytes / 6800e9 / 2e-3) < 1e-12


def test_dominant_kernel_of_a_split_forward():
    """With the forward split over the wide and the 64-column kernel, the two
    count as one launch; given the unmarked steps' total, the pair's time is
    that total minus the other kernels' marked time when that is the smaller
    (the marker between the pair removes their overlap)."""
    sys.path.insert(0, ROOT)
    import bench

    kernels = ["gdn_wy_tc_kernel", "gdn_wide_tc_kernel", "gdn_fused_tc_kernel"]
    name, t = bench.dominant(kernels, [6.0, 10.5, 2.4])
    assert name == "gdn_wide_tc_kernel+gdn_fused_tc_kernel" and abs(t - 12.9) < 1e-12
    name, t = bench.dominant(kernels, [6.0, 10.5, 2.4], 18.7)
    assert abs(t - 12.7) < 1e-12
    # never longer than the marked sum
    assert abs(bench.dominant(kernels, [6.0, 10.5, 2.4], 20.0)[1] - 12.9) < 1e-12
    # an unsplit step: the longest kernel, untouched by the total
    assert bench.dominant(["gdn_wy_tc_kernel", "gdn_fused_tc_kernel"], [3.0, 7.0], 9.0) == ("gdn_fused_tc_kernel", 7.0)


def test_design_traffic_from_the_committed_records():
    """The pipeline line adds the bytes the design moves per step (the ncu
    records of every kernel of the step, when all are current) to the
    compulsory bytes; a kernel without a current record leaves it null."""
    sys.path.insert(0, ROOT)
    import bench
    from gated_delta_rule_35_gb300.inputs import WORKLOADS

    w = WORKLOADS["bf16_b8_h64_t8192_k128_v128"]
    peaks = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "_source": "test"}
    ks = ["gdn_wy_tc_kernel", "gdn_wide_tc_kernel", "gdn_fused_tc_kernel"]
    r = bench.pipeline_roofline(w, 2e-3, peaks, False, ks)
    recs = [bench.ncu_traffic(k, w.name) for k in ks]
    if any(x is None for x in recs):
        assert r["design_traffic"] is None
    else:
        assert r["design_traffic"] == sum(recs)
        assert abs(r["design_traffic_over_compulsory"] - sum(recs) / r["bytes"]) < 1e-12
        assert abs(r["design_traffic_frac_of_hbm"] - sum(recs) / 2e-3 / 6800e9) < 1e-12
    assert bench.pipeline_roofline(w, 2e-3, peaks, False, ["no_such_kernel"])["design_traffic"] is None
    assert "design_traffic" not in bench.pipeline_roofline(w, 2e-3, peaks, False)


def test_traffic_records_by_workload_and_source(tmp_path, monkeypatch):
    """A kernel's ncu records may be one object or a list, one per workload:
    the bench takes the record of its workload, and none once the kernel's
    source no longer has the recorded hash."""
    sys.path.insert(0, ROOT)
    import bench

    src = tmp_path / "k.cu"
    src.write_text("// kernel source\n")
    sha = bench.hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps({
        "one": {"workload": "w1", "source_sha": sha, "dram_bytes_per_launch": 5},
        "many": [{"workload": "w1", "source_sha": sha, "dram_bytes_per_launch": 7},
                 {"workload": "w2", "source_sha": sha, "dram_bytes_per_launch": 11}],
        "stale": {"workload": "w1", "source_sha": "0" * 16, "dram_bytes_per_launch": 13}}))
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    monkeypatch.setattr(bench, "KERNEL_SOURCE", {"one": "k.cu", "many": "k.cu", "stale": "k.cu"})
    assert bench.ncu_traffic("one", "w1") == 5 and bench.ncu_traffic("one", "w2") is None
    assert bench.ncu_traffic("many", "w1") == 7 and bench.ncu_traffic("many", "w2") == 11
    assert bench.ncu_traffic("many", "w3") is None
    assert bench.ncu_traffic("stale", "w1") is None
    assert bench.ncu_traffic("one+many", "w1") == 12
    assert bench.ncu_traffic("one+many", "w2") is None
    assert bench.ncu_traffic("absent", "w1") is None
