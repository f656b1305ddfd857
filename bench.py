"""Benchmark of the exact-attention hot path on GB300.

One step = one pass over every stage of the path on one synthetic batch:
  * prefill: fused attention forward on the Llama-3-8B-shaped workload
    (B=2, H=32, N=4096, d=128, causal, bf16), stages a1-a7;
  * decode: Flash-Decoding split + merge on B=16, H=32, L=32768, d=128
    (bf16 KV cache of 8.6 GB), stages a8-a9.
The headline ``value`` is the prefill's TFLOP/s (matmul FLOPs 4 B H N^2 d,
halved for causal, over the summed device time of the prefill launches);
the decode's KV-read GB/s is reported beside it under ``decode``.

Prints one JSON line (rank 0). ``--impl reference`` times the fp64 CPU
oracle on a bounded sample of the same workload instead.

Multi-GPU (torchrun, one rank per GPU): every rank runs its own batch (weak
scaling, no collective on the data path); value = all ranks' FLOPs over the
max time across ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s (% of GB300 BF16 peak); decode KV-read GB/s (% of HBM)"
PREFILL_NAME = "llama3_8b_prefill"
NOMINAL_BF16_TFLOPS = 2250.0  # GB300 dense bf16 tensor peak (nominal)
NOMINAL_HBM_GBS = 7900.0      # GB300 HBM3e bandwidth (nominal)
DECODE_NAME = "decode_32k"
DEFAULT_SPLITS = 16
GQA_NAME = "decode_gqa8_32k"
GQA_SPLITS = 8
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": FALLBACK_BF16_TFLOPS_SUSTAINED, "source": "fallback"}


def _profile_traffic():
    """DRAM bytes per launch from the committed ncu summary, keyed by kernel tag."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    out = {}
    if not os.path.exists(path):
        return out
    for line in open(path):
        parts = [p.strip() for p in line.strip().strip("|").split("|")]
        if len(parts) >= 4 and parts[0].startswith("traffic:"):
            try:
                out[parts[0][len("traffic:"):]] = float(parts[3])
            except ValueError:
                pass
    return out


class ClockSampler:
    """Samples SM clocks, power and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "start":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        """Stop sampling; returns the summary of the window between mark("start") and mark("end")."""
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            self.rows.append((ts, parts))
        return self.summary(self.t0, self.t1)

    def summary(self, t0, t1):
        """Median SM clock, maximum clock and throttle reasons seen between host
        times t0 and t1 (the nearest sample when the window is shorter than the
        sampling period)."""
        rows = getattr(self, "rows", None)
        if not rows or t0 is None:
            return None
        t1 = t1 or t0
        inside = [r for ts, r in rows if t0 - 0.06 <= ts <= t1 + 0.06]
        if not inside:
            mid = (t0 + t1) / 2
            inside = [min(rows, key=lambda r: abs(r[0] - mid))[1]]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[0]) for r in inside if num(r[0]) is not None]
        smax = [num(r[1]) for r in inside if num(r[1]) is not None]
        reasons = set()
        for r in inside:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 r[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(values, world):
    """Element-wise max of a list of floats over all ranks (no-op when world == 1)."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist

    backend = dist.get_backend()
    dev = "cuda" if backend == "nccl" else "cpu"
    t = torch.tensor(values, dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.cpu().tolist()


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_oracle_sample(n_heads: int, seed: int = 0):
    """Time the fp64 oracle on the first n_heads (b, h) of the prefill workload
    (every row of each head); returns (tflops, seconds, flops, description)."""
    import numpy as np

    import oracle
    from exact_attention_29_gb300 import perfmodel
    from exact_attention_29_gb300 import workloads as wl

    c = wl.PREFILL[PREFILL_NAME]
    q, k, v = wl.prefill_inputs(c.B, c.H, c.N, c.d, seed=seed)
    heads = [(b, h) for b in range(c.B) for h in range(c.H)][:n_heads]
    qs = [(q[b, h].double().numpy(), k[b, h].double().numpy(), v[b, h].double().numpy()) for b, h in heads]
    oracle.build()
    pos = np.arange(c.N)
    t0 = time.perf_counter()
    for qq, kk, vv in qs:
        oracle.attention_rows(qq, pos, kk, vv, c.causal, c.scale)
    dt = time.perf_counter() - t0
    flops = perfmodel.fwd_flops(1, len(heads), c.N, c.d, c.causal)
    return flops / dt / 1e12, dt, flops, f"{len(heads)} of {c.B * c.H} heads of {PREFILL_NAME}, all {c.N} rows each"


def arm_config(world: int, splits: int) -> dict:
    """The workload both arms report (the same dict in the GPU and the reference line)."""
    from exact_attention_29_gb300 import workloads as wl

    pc, dc = wl.PREFILL[PREFILL_NAME], wl.DECODE[DECODE_NAME]
    return {"workload": f"{PREFILL_NAME} + {DECODE_NAME}",
            "prefill": {"B": pc.B, "H": pc.H, "N": pc.N, "d": pc.d, "causal": pc.causal},
            "decode": {"B": dc.B, "H": dc.H, "L": dc.L, "d": dc.d, "num_splits": splits},
            "l2": "inputs larger than L2 (prefill q/k/v/o 268 MB, decode KV 8.6 GB); no flush",
            "parallelism": f"replicas x{world}"}


def run_reference(args, world, rank):
    """The reference arm: the fp64 CPU oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    heads = 2
    for _ in range(args.warmup):
        cpu_oracle_sample(1)
    times, flops_total = [], 0.0
    desc = ""
    for _ in range(args.steps):
        _, dt, fl, desc = cpu_oracle_sample(heads)
        times.append(dt)
        flops_total += fl
    total = sum(times)
    value = flops_total / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": arm_config(world, args.splits),
        "sample_per_step": desc + " (value is the prefill's TFLOP/s, as in the GPU line; the oracle times no decode)",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


L2_BYTES = 129 * 2 ** 20  # GB300 L2 (126 MiB usable of 129 MB nominal; inputs above this stream from HBM)


def time_leg(fn, iters, stream, flush=None):
    """Device time of `iters` calls of fn() on `stream`, in ms per call, after 3
    warm-up calls. With `flush` (a callable that writes a buffer larger than
    L2), every call is timed alone between two events after a flush, so each
    starts with its inputs out of L2; without it the calls run back to back
    (inputs larger than L2)."""
    import torch

    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    if flush is None:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / iters
    total = 0.0
    pairs = []
    for _ in range(iters):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize()
    for a, b in pairs:
        total += a.elapsed_time(b)
    return total / iters


# Per-configuration legs: (name, prefill workload or decode workload, splits, calls timed)
PREFILL_LEGS = (("C1_pr1", "pr1", 200), ("C2a_gpt2_small", "gpt2_small", 100),
                ("C2b_gpt2_small_causal", "gpt2_small_causal", 100),
                ("C3_llama3_8b_prefill_noncausal", "llama3_8b_prefill_noncausal", 50),
                ("C4_long_16k", "long_16k", 20), ("C4_long_64k", "long_64k", 4))
DECODE_LEGS = tuple((f"C5_{name}_S{s}", name, s, 20) for name in ("decode_32k", "decode_32k_ragged")
                    for s in (8, 16, 32))


def run_config_legs(fa, wl, perfmodel, dev, stream, peaks, tag, dec_cache):
    """Every synthetic configuration timed on its own: absolute time, throughput
    and fraction of the measured and of the nominal peak; each leg keeps its host
    time window, for the clocks sampled while it ran. Inputs smaller than L2 are
    flushed out of it before each call."""
    import torch

    legs = {}
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.fill_(1.0)

    for leg, name, iters in PREFILL_LEGS:
        c = wl.PREFILL[name]
        q, k, v = wl.prefill_inputs(c.B, c.H, c.N, c.d, seed=0, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((c.B, c.H, c.N), dtype=torch.float32, device=dev)
        small = 4 * q.numel() * q.element_size() < L2_BYTES

        def call():
            fa.fa_fwd(q, k, v, causal=c.causal, o=o, lse=lse, stream=stream)

        t0 = time.time()
        ms = time_leg(call, iters, stream, flush if small else None)
        t1 = time.time()
        fa.fa_check_device_error(stream)
        flops = perfmodel.fwd_flops(c.B, c.H, c.N, c.d, c.causal)
        tf = flops / (ms * 1e-3) / 1e12
        legs[leg] = {"ms": ms, "value": tf, "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                     "frac_of_nominal": tf / NOMINAL_BF16_TFLOPS, "calls": iters,
                     "l2": "flushed before each call" if small else "inputs larger than L2",
                     "shape": f"B{c.B} H{c.H} N{c.N} d{c.d} {'causal' if c.causal else 'non-causal'}",
                     "window": (t0, t1)}
        del q, k, v, o, lse
    dq, kc, vc = dec_cache
    for leg, name, splits, iters in DECODE_LEGS:
        c = wl.DECODE[name]
        sl_host = wl.decode_seqlens(c.B, c.L, seed=0, ragged=c.ragged)
        sl = sl_host.to(dev)
        o = torch.empty_like(dq)
        lse = torch.empty((c.B, c.H), dtype=torch.float32, device=dev)

        def call():
            fa.fa_decode(dq, kc, vc, sl, splits, o=o, lse=lse, stream=stream)

        t0 = time.time()
        ms = time_leg(call, iters, stream)
        t1 = time.time()
        fa.fa_check_device_error(stream)
        kv = perfmodel.decode_kv_bytes(c.H, c.d, sl_host.tolist())
        alg = perfmodel.decode_algorithmic_bytes(c.B, c.H, c.d, sl_host.tolist())
        gbs = alg / (ms * 1e-3) / 1e9
        legs[leg] = {"ms": ms, "value": gbs, "unit": "GB/s", "kv_gbs": kv / (ms * 1e-3) / 1e9,
                     "frac": gbs / peaks["hbm_gbs"], "frac_of_nominal": gbs / NOMINAL_HBM_GBS, "calls": iters,
                     "l2": "inputs larger than L2", "shape": f"B{c.B} H{c.H} L{c.L} d{c.d} splits {splits}"
                     + (" ragged" if c.ragged else ""), "window": (t0, t1)}
    del flush_buf
    for leg in legs.values():
        leg["peak_kind"] = ("burst bf16 " if leg["unit"] == "TFLOP/s" else "copy ") + tag
    return legs


def oracle_one_core():
    """The oracle on one host core (OpenMP threads = 1): all of C1 and two heads
    of each GPT-2-shaped configuration, every row; TFLOP/s under the GPU's FLOP
    convention (causal halved), then the thread count restored."""
    import oracle
    from exact_attention_29_gb300 import perfmodel
    from exact_attention_29_gb300 import workloads as wl

    oracle.build()
    before = oracle.set_threads(0)
    out = {}
    try:
        oracle.set_threads(1)
        for leg, name, heads in (("C1_pr1", "pr1", 1), ("C2a_gpt2_small", "gpt2_small", 2),
                                 ("C2b_gpt2_small_causal", "gpt2_small_causal", 2)):
            c = wl.PREFILL[name]
            q, k, v = wl.prefill_inputs(c.B, c.H, c.N, c.d, seed=0)
            qs = q.reshape(-1, c.N, c.d)[:heads].unsqueeze(0)
            ks = k.reshape(-1, c.N, c.d)[:heads].unsqueeze(0)
            vs = v.reshape(-1, c.N, c.d)[:heads].unsqueeze(0)
            t0 = time.perf_counter()
            oracle.attention(qs, ks, vs, c.causal, c.scale)
            dt = time.perf_counter() - t0
            flops = perfmodel.fwd_flops(1, heads, c.N, c.d, c.causal)
            out[leg] = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "seconds": dt,
                        "sample": f"{heads} of {c.B * c.H} heads, all {c.N} rows"}
    finally:
        oracle.set_threads(before)
    return out


def run_gpu(args, world, rank, local):
    import torch

    import exact_attention_29_gb300 as fa
    from exact_attention_29_gb300 import build as fa_build
    from exact_attention_29_gb300 import perfmodel
    from exact_attention_29_gb300 import workloads as wl

    fa_build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    pc = wl.PREFILL[PREFILL_NAME]
    dc = wl.DECODE[DECODE_NAME]
    splits = args.splits
    q, k, v = wl.prefill_inputs(pc.B, pc.H, pc.N, pc.d, seed=rank, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((pc.B, pc.H, pc.N), dtype=torch.float32, device=dev)
    dq, kc, vc, seqlens = wl.decode_inputs(dc.B, dc.H, dc.L, dc.d, seed=rank, device=dev)
    do_ = torch.empty_like(dq)
    dlse = torch.empty((dc.B, dc.H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        fa.fa_fwd(q, k, v, causal=pc.causal, o=o, lse=lse, stream=stream)
        if evs is not None:
            evs[1].record(stream)
        fa.fa_decode(dq, kc, vc, seqlens, splits, o=do_, lse=dlse, stream=stream)
        if evs is not None:
            evs[2].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    fa.fa_check_device_error(stream)
    torch.cuda.synchronize(dev)

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", local))
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) > 8:
        gpu_id = "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id)
    if rank == 0:
        sampler.start()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.mark("start")
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark("end")
    if world > 1:
        dist.barrier()
    fa.fa_check_device_error(stream)

    total_ms = t_start.elapsed_time(t_end)
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in evs)
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in evs)
    total_ms, fwd_ms, dec_ms = reduce_max([total_ms, fwd_ms, dec_ms], world)

    fwd_flops = perfmodel.fwd_flops(pc.B, pc.H, pc.N, pc.d, pc.causal)
    kv_bytes = perfmodel.decode_kv_bytes(dc.H, dc.d, seqlens.tolist())
    dec_bytes = perfmodel.decode_algorithmic_bytes(dc.B, dc.H, dc.d, seqlens.tolist())
    value = world * fwd_flops * args.steps / (fwd_ms * 1e-3) / 1e12
    dec_gbs = world * kv_bytes * args.steps / (dec_ms * 1e-3) / 1e9

    # backward (gradients of the same prefill), timed on its own after the step loop
    bwd_steps = max(1, min(args.steps, 50))
    gdo = wl.backward_inputs(pc.B, pc.H, pc.N, pc.d, seed=rank, device=dev)
    gq, gk, gv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)

    def bwd_step():
        fa.fa_bwd(q, k, v, o, lse, gdo, causal=pc.causal, dq=gq, dk=gk, dv=gv, stream=stream)

    for _ in range(3):
        bwd_step()
    torch.cuda.synchronize(dev)
    b0 = torch.cuda.Event(enable_timing=True)
    b1 = torch.cuda.Event(enable_timing=True)
    w_bwd = [time.time()]
    b0.record(stream)
    for _ in range(bwd_steps):
        bwd_step()
    b1.record(stream)
    torch.cuda.synchronize(dev)
    w_bwd.append(time.time())
    fa.fa_check_device_error(stream)
    bwd_ms = reduce_max([b0.elapsed_time(b1)], world)[0]
    bwd_flops = perfmodel.bwd_flops(pc.B, pc.H, pc.N, pc.d, pc.causal)
    bwd_value = world * bwd_flops * bwd_steps / (bwd_ms * 1e-3) / 1e12

    # FP8 forward on the same prefill (e4m3 inputs quantized once, outside the timing)
    gsign = torch.Generator().manual_seed(1)
    signs = (torch.randint(0, 2, (pc.d,), generator=gsign) * 2 - 1).float().to(dev)
    q8, qsc = fa.fa_quantize_fp8(q, signs)
    k8, ksc = fa.fa_quantize_fp8(k, signs)
    vt8, vsc = fa.fa_quantize_fp8(v, None, per_head=True, transpose=True)
    o8 = torch.empty_like(o)
    l8 = torch.empty_like(lse)
    for _ in range(3):
        fa.fa_fwd_fp8(q8, k8, vt8, qsc, ksc, vsc, causal=pc.causal, o=o8, lse=l8, stream=stream)
    torch.cuda.synchronize(dev)
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    fp8_steps = max(1, min(args.steps, 100))
    w_fp8 = [time.time()]
    f0.record(stream)
    for _ in range(fp8_steps):
        fa.fa_fwd_fp8(q8, k8, vt8, qsc, ksc, vsc, causal=pc.causal, o=o8, lse=l8, stream=stream)
    f1.record(stream)
    torch.cuda.synchronize(dev)
    w_fp8.append(time.time())
    fa.fa_check_device_error(stream)
    fp8_ms = reduce_max([f0.elapsed_time(f1)], world)[0]
    fp8_value = world * fwd_flops * fp8_steps / (fp8_ms * 1e-3) / 1e12
    del q8, k8, vt8

    # block-sparse forward on the non-causal twin of the prefill under the band + global + random mask
    sc = wl.SPARSE_PREFILL
    smask = wl.block_mask_bigbird(sc.N // 128, heads=sc.H, seed=rank)
    s_allowed, s_computed = fa.fa_fwd_sparse_plan(smask, sc.B, sc.H, sc.N, sc.causal)
    smask_d = smask.to(dev)
    for _ in range(3):
        fa.fa_fwd_sparse(q, k, v, smask_d, causal=sc.causal, o=o8, lse=l8, stream=stream)
    torch.cuda.synchronize(dev)
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    sparse_steps = max(1, min(args.steps, 100))
    w_sparse = [time.time()]
    s0.record(stream)
    for _ in range(sparse_steps):
        fa.fa_fwd_sparse(q, k, v, smask_d, causal=sc.causal, o=o8, lse=l8, stream=stream)
    s1.record(stream)
    torch.cuda.synchronize(dev)
    w_sparse.append(time.time())
    fa.fa_check_device_error(stream)
    sparse_ms = reduce_max([s0.elapsed_time(s1)], world)[0]
    sparse_flops = 4.0 * 128 * 128 * sc.d * s_allowed
    sparse_value = world * sparse_flops * sparse_steps / (sparse_ms * 1e-3) / 1e12

    # GQA decode (64 query heads over 8 K/V heads), timed on its own after the step loop
    gc = wl.DECODE_GQA[GQA_NAME]
    gq, gkc, gvc, gsl = wl.decode_gqa_inputs(gc.B, gc.Hq, gc.Hkv, gc.L, gc.d, seed=rank, device=dev)
    go = torch.empty_like(gq)
    glse = torch.empty((gc.B, gc.Hq), dtype=torch.float32, device=dev)
    for _ in range(3):
        fa.fa_decode_gqa(gq, gkc, gvc, gsl, GQA_SPLITS, o=go, lse=glse, stream=stream)
    torch.cuda.synchronize(dev)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    gqa_steps = max(1, min(args.steps, 50))
    w_gqa = [time.time()]
    g0.record(stream)
    for _ in range(gqa_steps):
        fa.fa_decode_gqa(gq, gkc, gvc, gsl, GQA_SPLITS, o=go, lse=glse, stream=stream)
    g1.record(stream)
    torch.cuda.synchronize(dev)
    w_gqa.append(time.time())
    fa.fa_check_device_error(stream)
    gqa_ms = reduce_max([g0.elapsed_time(g1)], world)[0]
    gqa_kv = perfmodel.decode_kv_bytes(gc.Hkv, gc.d, gsl.tolist())
    gqa_gbs = world * gqa_kv * gqa_steps / (gqa_ms * 1e-3) / 1e9
    del gkc, gvc

    # every synthetic configuration on its own (C1-C5; C3 causal is the step's prefill above)
    peaks = _peaks()
    tag = "of measured" if peaks["source"] == "measured" else "of fallback"
    legs = run_config_legs(fa, wl, perfmodel, dev, stream, peaks, tag, (dq, kc, vc))

    # end to end through the C ABI with host buffers: every step is one
    # fa_fwd_host call, which uploads q, k, v from pinned host memory, runs the
    # forward and downloads o and lse, all inside the timed region. Steps go
    # round-robin over three streams, as a serving pipeline would issue them,
    # so step s+1's upload and step s-1's download overlap step s's kernel.
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    e2e_streams = [torch.cuda.Stream(dev) for _ in range(3)]
    hosts_out = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(), torch.empty(lse.shape, dtype=lse.dtype).pin_memory())
                 for _ in range(3)]
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_run(steps, e_start=None, e_end=None):
        s0 = e2e_streams[0]
        if e_start is not None:
            e_start.record(s0)
            for st in e2e_streams[1:]:
                st.wait_stream(s0)
        for s in range(steps):
            ho, hl = hosts_out[s % 3]
            fa.fa_fwd_host(hq, hk, hv, causal=pc.causal, o=ho, lse=hl, stream=e2e_streams[s % 3])
        if e_end is not None:
            for st in e2e_streams[1:]:
                s0.wait_stream(st)
            e_end.record(s0)

    e2e_run(3)
    torch.cuda.synchronize(dev)
    # three timed trials of e2e_steps calls each; the median trial is reported
    # and every trial is listed (a trial now and then runs far slower while the
    # link measured alone does not, so one trial alone is not a stable figure)
    trial_ms = []
    for _ in range(3):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e2e_run(e2e_steps, e0, e1)
        torch.cuda.synchronize(dev)
        trial_ms.append(e0.elapsed_time(e1))
    for st in e2e_streams:
        fa.fa_check_device_error(st)
    trial_ms = reduce_max(trial_ms, world)
    e2e_ms = sorted(trial_ms)[1]
    e2e_value = world * fwd_flops * e2e_steps / (e2e_ms * 1e-3) / 1e12
    e2e_trials = [world * fwd_flops * e2e_steps / (t * 1e-3) / 1e12 for t in trial_ms]
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()

    # the host link alone: one step's uploads and downloads, at the same time on
    # the same two streams, no kernel; the pipeline above cannot beat this
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    d_in = tuple(torch.empty_like(t) for t in (q, k, v))
    d_out = (torch.empty_like(o), torch.empty_like(lse))

    def link_step(i):
        with torch.cuda.stream(s_in):
            for dst, src in zip(d_in, (hq, hk, hv)):
                dst.copy_(src, non_blocking=True)
        with torch.cuda.stream(s_out):
            hosts_out[i % 3][0].copy_(d_out[0], non_blocking=True)
            hosts_out[i % 3][1].copy_(d_out[1], non_blocking=True)

    link_step(0)
    torch.cuda.synchronize(dev)
    l0 = torch.cuda.Event(enable_timing=True)
    l1 = torch.cuda.Event(enable_timing=True)
    l0.record(s_in)
    s_out.wait_stream(s_in)
    for i in range(6):
        link_step(i)
    s_out.wait_stream(s_in)
    l1.record(s_out)
    torch.cuda.synchronize(dev)
    link_ms = l0.elapsed_time(l1) / 6
    del d_in, d_out

    if rank != 0:
        return
    clocks = sampler.stop()
    for leg in legs.values():
        leg["clocks"] = sampler.summary(*leg.pop("window"))
    leg_clocks = {name: sampler.summary(*w) for name, w in
                  (("backward", w_bwd), ("fwd_fp8", w_fp8), ("fwd_sparse", w_sparse), ("decode_gqa", w_gqa))}
    long_region = total_ms > 1000.0
    tflops_peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    traffic = _profile_traffic()
    fwd_avg_ms = fwd_ms / args.steps
    dec_avg_ms = dec_ms / args.steps
    fwd_roof = {"bound": "tensor", "achieved": fwd_flops / (fwd_avg_ms * 1e-3) / 1e12, "peak": tflops_peak,
                "unit": "TFLOP/s", "traffic": traffic.get("fwd_kernel_128_llama3_8b_prefill"),
                "kernel": "fwd_kernel<128>", "peak_kind": ("sustained " if long_region else "burst ") + tag}
    fwd_roof["frac"] = fwd_roof["achieved"] / fwd_roof["peak"]
    # the metric's own denominators: GB300 nominal dense bf16 and HBM3e bandwidth
    fwd_roof["frac_of_nominal"] = fwd_roof["achieved"] / NOMINAL_BF16_TFLOPS
    dec_roof = {"bound": "hbm", "achieved": dec_bytes / (dec_avg_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "traffic": traffic.get("decode_split_kernel_128_decode_32k"),
                "kernel": "decode_split_kernel<128> + decode_merge_kernel<128>", "peak_kind": "copy " + tag}
    dec_roof["frac"] = dec_roof["achieved"] / dec_roof["peak"]
    dec_roof["frac_of_nominal"] = dec_roof["achieved"] / NOMINAL_HBM_GBS
    dominant = dec_roof if dec_avg_ms >= fwd_avg_ms else fwd_roof

    def leg_roof(bound, achieved, peak, unit, traffic_tag, kernel, peak_kind):
        return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                "traffic": traffic.get(traffic_tag), "kernel": kernel, "peak_kind": peak_kind}

    # GQA algorithmic bytes: K/V of the shared heads, plus q, o and lse of every query head
    gqa_bytes = perfmodel.decode_algorithmic_bytes(gc.B, gc.Hq, gc.d, gsl.tolist()) - \
        perfmodel.decode_kv_bytes(gc.Hq, gc.d, gsl.tolist()) + gqa_kv
    leg_roofs = {
        "backward": leg_roof("tensor", bwd_value / world, peaks["bf16_tflops"], "TFLOP/s",
                             "bwd_kernel_128_llama3_8b_prefill", "bwd_kernel<128> (+ prep, convert)",
                             "burst " + tag),
        "fwd_fp8": leg_roof("tensor", fp8_value / world, 2 * peaks["bf16_tflops"], "TFLOP/s",
                            "fwd_kernel_128_fp8_llama3_8b_prefill", "fwd_kernel<128, e4m3>",
                            "2x burst bf16 " + tag + " (nominal e4m3/bf16 ratio)"),
        "fwd_sparse": leg_roof("tensor", sparse_value / world, peaks["bf16_tflops"], "TFLOP/s",
                               "fwd_kernel_128_sparse_llama3_8b_bigbird", "fwd_kernel<128, block-sparse>",
                               "burst " + tag),
        "decode_gqa": leg_roof("hbm", gqa_bytes / (gqa_ms / gqa_steps * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s",
                               "decode_gqa_split_kernel_128_decode_gqa8_32k",
                               "decode_gqa_split_kernel<128> + decode_merge_kernel<128>", "copy " + tag),
    }

    c_tflops, c_dt, _, c_desc = cpu_oracle_sample(args.cpu_heads)
    one_core = oracle_one_core()
    for name, lc in leg_clocks.items():
        leg_roofs[name]["clocks"] = lc

    def row(ms, val, unit, frac, frac_nom, clk):
        return [float(f"{ms:.4g}"), float(f"{val:.4g}"), unit, round(frac, 3), round(frac_nom, 3),
                (clk or {}).get("sm_mhz")]

    summary = {"fields": "ms per call, value, unit (TF = TFLOP/s, GB = GB/s), frac of measured peak, "
                         "frac of nominal (2.25 PF bf16, 7.9 TB/s), median SM MHz"}
    for name in ("C1_pr1", "C2a_gpt2_small", "C2b_gpt2_small_causal"):
        g = legs[name]
        summary[name] = row(g["ms"], g["value"], "TF", g["frac"], g["frac_of_nominal"], g["clocks"])
    summary["C3_llama3_8b_prefill"] = row(fwd_avg_ms, value / world, "TF", value / world / peaks["bf16_tflops"],
                                          value / world / NOMINAL_BF16_TFLOPS, clocks)
    for name, g in legs.items():
        if name not in summary:
            summary[name] = row(g["ms"], g["value"], "TF" if g["unit"] == "TFLOP/s" else "GB", g["frac"],
                                g["frac_of_nominal"], g["clocks"])
    summary["backward"] = row(bwd_ms / bwd_steps, bwd_value / world, "TF", leg_roofs["backward"]["frac"],
                              bwd_value / world / NOMINAL_BF16_TFLOPS, leg_clocks["backward"])
    summary["fwd_fp8"] = row(fp8_ms / fp8_steps, fp8_value / world, "TF", leg_roofs["fwd_fp8"]["frac"],
                             fp8_value / world / (2 * NOMINAL_BF16_TFLOPS), leg_clocks["fwd_fp8"])
    summary["fwd_sparse_kept"] = row(sparse_ms / sparse_steps, sparse_value / world, "TF",
                                     leg_roofs["fwd_sparse"]["frac"], sparse_value / world / NOMINAL_BF16_TFLOPS,
                                     leg_clocks["fwd_sparse"])
    summary["fwd_sparse_computed_over_kept"] = round(s_computed / max(1, s_allowed), 3)
    summary["decode_gqa"] = row(gqa_ms / gqa_steps, leg_roofs["decode_gqa"]["achieved"], "GB",
                                leg_roofs["decode_gqa"]["frac"], leg_roofs["decode_gqa"]["achieved"] / NOMINAL_HBM_GBS,
                                leg_clocks["decode_gqa"])
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": arm_config(world, splits),
        "decode": {"value": dec_gbs, "unit": "GB/s (KV read)", "frac_of_hbm": dec_gbs / peaks["hbm_gbs"],
                   "ms_per_step": dec_avg_ms},
        "prefill_ms_per_step": fwd_avg_ms,
        "fwd_fp8": {"roofline": leg_roofs["fwd_fp8"], "value": fp8_value, "unit": "TFLOP/s", "ms_per_call": fp8_ms / fp8_steps, "steps": fp8_steps,
                    "frac_of_fp8_peak": fp8_value / world / (2 * peaks["bf16_tflops"]),
                    "peak_note": "fp8 peak taken as 2x the measured bf16 burst (the nominal dense ratio)",
                    "what": "fa_fwd_fp8 on e4m3 inputs of the prefill workload (quantized once, outside the timing)"},
        "fwd_sparse": {"roofline": leg_roofs["fwd_sparse"], "value": sparse_value, "unit": "TFLOP/s (kept block pairs, 4*128*128*d each)",
                       "ms_per_call": sparse_ms / sparse_steps, "steps": sparse_steps,
                       "pairs_kept": s_allowed, "pairs_computed": s_computed,
                       "pairs_all": sc.B * sc.H * (sc.N // 128) ** 2,
                       "what": f"fa_fwd_sparse on {sc.name} (B{sc.B} H{sc.H} N{sc.N} d{sc.d}, non-causal) under the "
                               "band + global + random block mask, one per head"},
        "decode_gqa": {"roofline": leg_roofs["decode_gqa"], "value": gqa_gbs, "unit": "GB/s (KV read)", "ms_per_call": gqa_ms / gqa_steps,
                       "steps": gqa_steps, "frac_of_hbm": gqa_gbs / peaks["hbm_gbs"],
                       "what": f"fa_decode_gqa on {GQA_NAME} (B{gc.B} Hq{gc.Hq} Hkv{gc.Hkv} L{gc.L} d{gc.d}), "
                               f"{GQA_SPLITS} splits, timed after the step loop"},
        "backward": {"roofline": leg_roofs["backward"], "value": bwd_value, "unit": "TFLOP/s (10 N^2 d per head, halved causal)",
                     "ms_per_call": bwd_ms / bwd_steps, "steps": bwd_steps,
                     "frac_of_bf16_peak": bwd_value / world / peaks["bf16_tflops"],
                     "what": "fa_bwd on the prefill workload (dQ zeroing, D, main kernel, dQ conversion), "
                             "timed after the step loop"},
        "prefill_frac_of_bf16_peak": value / world / tflops_peak,
        "roofline": dominant,
        "rooflines": {"fwd": fwd_roof, "decode": dec_roof},
        "cpu_baseline": {"value": c_tflops, "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
                         "sample": c_desc, "seconds": c_dt, "one_core": one_core},
        "configs": legs,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "trials": e2e_trials,
                "link": {"ms_per_step": link_ms, "h2d_gbs": h2d / (link_ms * 1e-3) / 1e9,
                         "frac": link_ms / (e2e_ms / e2e_steps),
                         "what": "one step's uploads and downloads alone (same streams, no kernel): the host "
                                 "link's bound on a step; frac = that time / the pipelined step time"},
                "what": "prefill through the C-ABI call fa_fwd_host with pinned host buffers; every step's call "
                        "uploads q/k/v, runs the forward and downloads o/lse inside the timed region; steps go "
                        "round-robin over three streams (upload of step s+1 and download of step s-1 overlap "
                        "step s); three trials of `steps` calls, value = the median trial"},
        "gpu_launches": 3 * args.steps,
        "summary": summary,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--splits", type=int, default=DEFAULT_SPLITS)
    ap.add_argument("--cpu-heads", type=int, default=48)
    args = ap.parse_args()
    world, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    run_gpu(args, world, rank, local)


if __name__ == "__main__":
    main()
