"""Run one named workload a few times on cuda:0 (for profilers such as ncu).

    python -m exact_attention_29_gb300.run_case --workload llama3_8b_prefill --iters 3
    python -m exact_attention_29_gb300.run_case --workload decode_32k --batch 4 --splits 16 --iters 3
    python -m exact_attention_29_gb300.run_case --workload llama3_8b_prefill --bwd --iters 3

``--batch`` overrides B (to keep a profiled case small); inputs are drawn by
the seeded generators of ``workloads.py``. Prints the device time per
iteration measured with CUDA events.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch

    import exact_attention_29_gb300 as fa
    from exact_attention_29_gb300 import build
    from exact_attention_29_gb300 import workloads as wl

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", required=True,
                    choices=sorted(list(wl.PREFILL) + list(wl.DECODE) + list(wl.DECODE_GQA)))
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--batch", type=int, default=0)
    ap.add_argument("--splits", type=int, default=16)
    ap.add_argument("--n", type=int, default=0, help="override the sequence length of a prefill workload")
    ap.add_argument("--bwd", action="store_true", help="time fa_bwd (after one fa_fwd) on a prefill workload")
    ap.add_argument("--fp8", action="store_true", help="time fa_fwd_fp8 on e4m3 inputs of a prefill workload")
    ap.add_argument("--sparse", action="store_true",
                    help="time fa_fwd_sparse under the band + global + random block mask (one per head)")
    args = ap.parse_args()
    build.build()
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev)
    if args.workload in wl.PREFILL:
        c = wl.PREFILL[args.workload]
        if args.n:
            c = wl.Prefill(c.name, c.B, c.H, args.n, c.d, c.causal)
        B = args.batch or c.B
        q, k, v = wl.prefill_inputs(B, c.H, c.N, c.d, seed=0, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, c.H, c.N), dtype=torch.float32, device=dev)

        def run():
            fa.fa_fwd(q, k, v, causal=c.causal, o=o, lse=lse, stream=stream)

        if args.sparse:
            mask = wl.block_mask_bigbird((c.N + 127) // 128, heads=c.H, seed=0)
            allowed, computed = fa.fa_fwd_sparse_plan(mask, B, c.H, c.N, c.causal)
            mask_d = mask.to(dev)

            def run():
                fa.fa_fwd_sparse(q, k, v, mask_d, causal=c.causal, o=o, lse=lse, stream=stream)

        if args.fp8:
            g = torch.Generator().manual_seed(1)
            signs = (torch.randint(0, 2, (c.d,), generator=g) * 2 - 1).float().to(dev)
            q8, qs = fa.fa_quantize_fp8(q, signs)
            k8, ks = fa.fa_quantize_fp8(k, signs)
            vt8, vs = fa.fa_quantize_fp8(v, None, per_head=True, transpose=True)

            def run():
                fa.fa_fwd_fp8(q8, k8, vt8, qs, ks, vs, causal=c.causal, o=o, lse=lse, stream=stream)

        if args.bwd:
            run()
            do = wl.backward_inputs(B, c.H, c.N, c.d, seed=0, device=dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)

            def run():
                fa.fa_bwd(q, k, v, o, lse, do, causal=c.causal, dq=dq, dk=dk, dv=dv, stream=stream)
    elif args.workload in wl.DECODE:
        c = wl.DECODE[args.workload]
        B = args.batch or c.B
        q, kc, vc, sl = wl.decode_inputs(B, c.H, c.L, c.d, seed=0, ragged=c.ragged, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, c.H), dtype=torch.float32, device=dev)

        def run():
            fa.fa_decode(q, kc, vc, sl, args.splits, o=o, lse=lse, stream=stream)
    else:
        c = wl.DECODE_GQA[args.workload]
        B = args.batch or c.B
        q, kc, vc, sl = wl.decode_gqa_inputs(B, c.Hq, c.Hkv, c.L, c.d, seed=0, ragged=c.ragged, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, c.Hq), dtype=torch.float32, device=dev)

        def run():
            fa.fa_decode_gqa(q, kc, vc, sl, args.splits, o=o, lse=lse, stream=stream)

    torch.cuda.synchronize(dev)
    times = []
    for _ in range(args.iters):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1))
    fa.fa_check_device_error(stream)
    extra = ""
    if args.workload in wl.PREFILL:
        from exact_attention_29_gb300 import perfmodel

        flops = (perfmodel.bwd_flops if args.bwd else perfmodel.fwd_flops)(B, c.H, c.N, c.d, c.causal)
        if args.sparse:
            # the two products on the block pairs the mask keeps (4 * 128 * 128 * d each)
            flops = 4.0 * 128 * 128 * c.d * allowed
            extra = f" (kept {allowed} of {B * c.H * ((c.N + 127) // 128) ** 2} pairs, computed {computed})"
        else:
            extra = ""
        extra = f" best {flops / min(times) / 1e9:.1f} TFLOP/s" + extra
    else:
        from exact_attention_29_gb300 import perfmodel

        kv = perfmodel.decode_kv_bytes(c.Hkv if hasattr(c, "Hkv") else c.H, c.d, sl.tolist())
        extra = f" best {kv / min(times) / 1e6:.0f} GB/s of K/V"
    what = "bwd" if args.bwd else ("fwd_fp8" if args.fp8 else ("fwd_sparse" if args.sparse else "fwd"))
    print(f"{args.workload} {what if args.workload in wl.PREFILL else ''} B={B}: "
          + " ".join(f"{t:.3f}ms" for t in times) + extra)


if __name__ == "__main__":
    main()
