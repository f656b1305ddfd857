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
