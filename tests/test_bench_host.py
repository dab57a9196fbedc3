"""Host-side logic of the benchmark, checked without a GPU: the workload table
(shapes and algorithmic work), the robust mean of the sweep, the clock-record
summary that decides the peak, the guard that drops stale ncu traffic, and the
reference arm (the oracle on host cores) and its JSON line."""
import json
import os
import statistics

import pytest

import bench
from tensor_gemm_reduction_gb300 import inputs as gi


def test_workload_table_has_the_pages_projection_shapes():
    names = {w.name: w for w in gi.ALL_WORKLOADS}
    # AG-GEMM page, microbenchmark tables: KDA (N = 6288) and MLA (N = 3648)
    # projections at K = 7168 on TP8, global M = 8 x local M.
    for local in (256, 384, 448, 512, 1024, 2048, 4096):
        for kind, n in (("kda", 6288), ("mla", 3648)):
            w = names[f"ag_{kind}_m{8 * local}"]
            assert (w.mode, w.N, w.K, w.R, w.M) == ("ag", n, 7168, 8, 8 * local)
            assert w.shard_sizes() == [local] * 8
    # GEMM-RS/AR page, o_proj: N = K = 7168, K split over 8 ranks.
    for m in (1, 16, 64, 128, 129, 256, 1000, 4096, 32768):
        w = names[f"ar_oproj_m{m}"]
        assert (w.mode, w.N, w.K, w.R, w.M) == ("ar", 7168, 7168, 8, m)
        assert w.shard_sizes() == [896] * 8
    for r in (2, 4, 8, 16):
        w = names[f"rs_r{r}"]
        assert w.shard_sizes() == [7168 // r] * r and w.M == 32768
        # RS shares its inputs with AR o_proj M = 32768.
        assert w.seed == gi.default_seed(32768, 7168)
    assert names["ar_tiny"].seed == 0


def test_algorithmic_work_closed_forms():
    w = bench.workload_by_name("ag_kda_m32768")
    assert w.flops == 2 * 32768 * 6288 * 7168            # 2.95 TFLOP
    assert round(w.flops / 1e12, 2) == 2.95
    assert w.bytes == 2 * (32768 * 7168 + 6288 * 7168 + 32768 * 6288)
    ar = bench.workload_by_name("ar_oproj_m32768")
    assert round(ar.flops / 1e12, 2) == 3.37
    # W alone at N = K = 7168 is 102.8 MB: the whole cost of a decode step.
    small = bench.workload_by_name("ar_oproj_m128")
    assert small.bytes - 2 * (128 * 7168 * 2) == 2 * 7168 * 7168
    assert round(2 * 7168 * 7168 / 1e6, 1) == 102.8
    # Packed gather: the kept rows of every state read once, P written once.
    p = gi.PACK_SP
    assert p.bytes == 2 * 2 * (8 * 4096 - 5) * 4 * 7168


def test_decode_layer_rows_stream_more_weights_than_the_l2_holds():
    # The decode-step rows run without an L2 flush. A weight set is used again
    # only after the three others (3 x 103 MB) have streamed through the L2,
    # so every call reads its W from HBM.
    w = bench.workload_by_name("ar_oproj_m1")
    assert (bench.DECODE_LAYERS - 1) * 2 * w.N * w.K > bench.L2_BYTES


def test_decode_layer_rows_cover_the_small_m_o_proj_shapes():
    assert [w.M for w in bench.decode_layer_workloads()] == [1, 16, 64, 128, 129, 256]
    assert {w.K for w in bench.decode_layer_workloads()} == {7168}
    assert [w.M for w in bench.decode_layer_workloads(["ar_oproj_m129", "ag_kda_m2048"])] == [129]
    assert [w.M for w in bench.decode_layer_workloads(["ar_oproj_m1_layers4"])] == [1]
    assert bench.decode_layer_workloads(["ar_oproj_m1000"]) == []


def test_unknown_workload_is_rejected():
    with pytest.raises(SystemExit):
        bench.workload_by_name("no_such_workload")


def test_describe_workload_names_the_shard_sizes():
    d = bench.describe_workload(bench.workload_by_name("ag_mla_m3584"))
    assert d == {"workload": "ag_mla_m3584", "mode": "ag", "R": 8, "M": 3584, "N": 3648,
                 "K": 7168, "M_r": 448}
    d = bench.describe_workload(bench.workload_by_name("rs_r16"))
    assert d["K_r"] == 448 and "M_r" not in d


def test_trimmed_mean_drops_both_tails():
    xs = [10.0] * 8 + [1000.0, 0.001, 10.5, 9.5]
    assert bench.trimmed_mean(xs) == pytest.approx(10.0)
    assert bench.trimmed_mean([3.0]) == 3.0
    assert bench.trimmed_mean([1.0, 2.0]) == 1.5


def _clock_rows(path, rows):
    with open(path, "w") as f:
        for sm, mx, pw, flags in rows:
            f.write(f"0, {sm}, {mx}, {pw}, 0x0, " + ", ".join(flags) + "\n")


def test_clock_summary_uses_loaded_samples_and_collects_reasons(tmp_path):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    s.proc = object()              # as if nvidia-smi had run
    idle = ("Not Active",) * 4
    capped = ("Not Active", "Not Active", "Not Active", "Active")
    _clock_rows(s.path, [(2070, 2070, 200.0, idle)] * 5 +
                        [(1400, 2070, 1390.0, capped)] * 3 + [(1450, 2070, 1300.0, idle)] * 2)
    out = s.summary()
    assert out["sm_mhz"] == 1400                 # median of the five loaded samples
    assert out["sm_max_mhz"] == 2070
    assert out["samples"] == 5
    assert out["reasons"] == ["sw_power_cap"]
    assert not os.path.exists(s.path)


def test_clock_summary_without_nvidia_smi():
    s = bench.ClockSampler(0)
    assert s.summary()["reasons"] == ["nvidia-smi unavailable"]


def test_peaks_fall_back_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks()["source"] == "fallback"
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"hbm_gbs": 7000.0, "bf16_tflops": 1800.0}))
    pk = bench.peaks()
    assert pk["source"] == "measured"
    assert pk["bf16_sustained"] == pk["bf16_burst"] == 1800.0


def test_ncu_traffic_is_dropped_once_the_kernel_changes(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"ag_kda_m32768": {"kernel_hash": "aaaa", "dram_bytes_per_launch": 123}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "aaaa")
    assert bench.ncu_traffic("ag_kda_m32768") == 123
    assert bench.ncu_traffic("ag_mla_m2048") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "bbbb")
    assert bench.ncu_traffic("ag_kda_m32768") is None


def _bench(args, env_extra=None):
    import subprocess
    import sys
    env = dict(os.environ, **(env_extra or {}))
    return subprocess.run([sys.executable, os.path.join(os.path.dirname(bench.__file__), "bench.py")]
                          + args, capture_output=True, text=True, timeout=300, env=env)


def test_reference_arm_prints_one_contract_line():
    r = _bench(["--impl", "reference", "--workload", "ar_tiny", "--steps", "3", "--warmup", "3"])
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["steps"] == 3 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "ar_tiny"


def test_reference_arm_other_ranks_exit_quietly():
    r = _bench(["--impl", "reference", "--workload", "ar_tiny", "--steps", "3", "--warmup", "3"],
               {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_bench_rejects_fewer_than_three_warmup_steps():
    r = _bench(["--impl", "reference", "--workload", "ar_tiny", "--steps", "3", "--warmup", "2"])
    assert r.returncode != 0 and "--warmup" in r.stderr


def test_both_arms_share_the_config_object():
    w = bench.workload_by_name("ag_kda_m32768")
    c = bench.bench_config(w, 1)
    assert c["workload"] == "ag_kda_m32768" and c["seed"] == 2000 + 32768 + 7168
    assert c["parallelism"] == "single" and bench.bench_config(w, 8)["parallelism"] == "replicas"
    assert bench.bench_config(bench.workload_by_name("ar_tiny"), 1)["seed"] == 0
    r = _bench(["--impl", "reference", "--workload", "ar_tiny", "--steps", "3", "--warmup", "3"])
    assert json.loads(r.stdout)["config"] == bench.bench_config(bench.workload_by_name("ar_tiny"), 1)


def test_config_states_whether_the_inputs_exceed_l2():
    assert bench.bench_config(bench.workload_by_name("ag_kda_m32768"), 1)["l2"].startswith(
        "inputs larger than L2: 560 MB")
    assert "fit in L2" in bench.bench_config(bench.workload_by_name("ar_tiny"), 1)["l2"]


def test_plan_options_parse_and_are_recorded():
    from tensor_gemm_reduction_gb300 import binding as B
    opts = bench.parse_options(["schedule=5", "BLOCK_N=192", "raster_n=0x4"])
    assert opts == {"GSR_OPT_SCHEDULE": 5, "GSR_OPT_BLOCK_N": 192, "GSR_OPT_RASTER_N": 4}
    assert all(hasattr(B, k) for k in opts)
    w = bench.workload_by_name("ag_mla_m2048")
    assert bench.bench_config(w, 1, opts)["options"] == {"schedule": 5, "block_n": 192, "raster_n": 4}
    assert "options" not in bench.bench_config(w, 1, {})
    for bad in (["nosuch=1"], ["schedule"], ["schedule=fast"]):
        with pytest.raises(SystemExit):
            bench.parse_options(bad)
    r = _bench(["--impl", "reference", "--workload", "ar_tiny", "--steps", "3", "--warmup", "3",
                "--option", "split_k=2"])
    assert json.loads(r.stdout)["config"]["options"] == {"split_k": 2}


def test_nvml_sampler_summary_keeps_only_the_timed_region():
    """The in-process clock sampler's summary: samples outside the marked
    region are dropped, the median SM clock and the power come from the
    samples inside it, and the event-reason bits decode to their names."""
    s = bench.NvmlClockSampler(0)
    s.max_mhz = 2070.0
    s.t0, s.t1 = 10.0, 10.05
    s.samples = [(9.99, 700.0, 150.0, 0x1)] + \
        [(10.0 + 0.001 * i, 1900.0 + i, 900.0 + i, 0x4 if i == 7 else 0) for i in range(40)] + \
        [(10.2, 600.0, 140.0, 0x8)]
    c = s.summary()
    assert c["samples"] == 40
    assert c["sm_mhz"] == statistics.median(1900.0 + i for i in range(40))
    assert c["sm_mhz_min"] == 1900.0 and c["sm_max_mhz"] == 2070.0
    assert c["power_w_max"] == 939.0
    assert c["reasons"] == ["sw_power_cap"]          # hw_slowdown fell outside the region
    e = bench.NvmlClockSampler(0)
    assert e.summary()["reasons"] == ["no samples"]
