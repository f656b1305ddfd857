"""bench.py's JSON contract, checked on CPU through the reference arm (the fp64
oracle timed on the host cores) and the host-side helpers of the GPU arm."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
             "vs_baseline", "dtype", "data", "config"}


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert BASE_KEYS <= set(line), set(line) ^ BASE_KEYS
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["higher_is_better"] is True and line["steps"] == 1 and line["warmup"] == 1
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0

    import bench

    # both arms report the same workload
    assert line["config"] == bench.arm_config(1, bench.DEFAULT_SPLITS)
    assert line["metric"] == bench.METRIC


def test_traffic_table_has_every_leg():
    import bench

    traffic = bench._profile_traffic()
    for tag in ("fwd_kernel_128_llama3_8b_prefill", "decode_split_kernel_128_decode_32k",
                "bwd_kernel_128_llama3_8b_prefill", "decode_gqa_split_kernel_128_decode_gqa8_32k",
                "fwd_kernel_128_fp8_llama3_8b_prefill", "fwd_kernel_128_sparse_llama3_8b_bigbird"):
        assert tag in traffic and traffic[tag] > 0, tag


def test_peaks_are_read():
    import bench

    peaks = bench._peaks()
    assert peaks["hbm_gbs"] > 1000 and peaks["bf16_tflops"] > 500


def test_one_core_oracle_leg_restores_the_thread_count():
    import bench
    import oracle

    before = oracle.set_threads(0)
    out = bench.oracle_one_core()
    assert set(out) == {"C1_pr1", "C2a_gpt2_small", "C2b_gpt2_small_causal"}
    assert all(v["value"] > 0 and v["seconds"] > 0 and v["sample"] for v in out.values())
    assert oracle.set_threads(0) == before


def test_clock_windows():
    """Each leg's clocks come from the samples inside its own host time window
    (the nearest one when the window is shorter than the sampling period)."""
    import bench

    s = bench.ClockSampler("0")
    idle = ["1000", "2070", "100", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]
    busy = ["2070", "2070", "900", "0x0", "Not Active", "Not Active", "Not Active", "Active"]
    s.rows = [(10.0, idle), (10.2, busy), (10.4, busy), (10.6, idle), (20.0, idle)]
    w = s.summary(10.15, 10.45)
    assert w["sm_mhz"] == 2070 and w["samples"] == 2 and w["reasons"] == ["sw_power_cap"]
    near = s.summary(19.9, 19.95)
    assert near["samples"] == 1 and near["sm_mhz"] == 1000 and near["reasons"] == []
