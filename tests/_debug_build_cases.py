"""Run a spread of library calls and save their outputs (a helper of
test_gpu_debug_build.py, run as a child process so that FA_LIBRARY picks the
library build). After every call the device error word is checked: a protocol
check of an FA_DEBUG build that fails raises FaError(FA_ERR_CHECK)."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import exact_attention_29_gb300 as fa  # noqa: E402
from exact_attention_29_gb300 import workloads as wl  # noqa: E402


def main(out_path):
    out = {}

    def keep(name, *ts):
        fa.fa_check_device_error()
        for i, t in enumerate(ts):
            out[f"{name}_{i}"] = t.detach().float().cpu().numpy()

    for N, d, causal in ((1000, 128, True), (333, 64, False), (1, 128, True), (700, 64, True), (1300, 128, False)):
        q, k, v = wl.prefill_inputs(2, 3, N, d, seed=N + d, device="cuda")
        keep(f"fwd_{N}_{d}_{int(causal)}", *fa.fa_fwd(q, k, v, causal=causal))
        dout = wl.backward_inputs(2, 3, N, d, seed=N + d, device="cuda")
        o, lse = fa.fa_fwd(q, k, v, causal=causal)
        dq, dk, dv = fa.fa_bwd(q, k, v, o, lse, dout, causal=causal)
        keep(f"bwd_{N}_{d}_{int(causal)}", dk, dv)  # dQ sums atomic additions in any order
        T = (N + 127) // 128
        mask = (torch.rand((3, T, T), generator=torch.Generator().manual_seed(N)) < 0.5).to(torch.uint8).cuda()
        keep(f"sparse_{N}_{d}_{int(causal)}", *fa.fa_fwd_sparse(q, k, v, mask, causal=causal))
    # backward over several waves of CTAs (80 heads x 6 K/V tiles)
    for d, causal in ((128, True), (64, False)):
        q, k, v = wl.prefill_inputs(4, 20, 700, d, seed=d + 2, device="cuda")
        dout = wl.backward_inputs(4, 20, 700, d, seed=d + 2, device="cuda")
        o, lse = fa.fa_fwd(q, k, v, causal=causal)
        dq, dk, dv = fa.fa_bwd(q, k, v, o, lse, dout, causal=causal)
        keep(f"bwd_items_{d}_{int(causal)}", dk, dv)
    # block-sparse over 32 tiles: band + global + random rows, some block rows
    # keeping everything and some nothing (uneven private runs within a pair)
    for d, causal in ((128, False), (64, True)):
        q, k, v = wl.prefill_inputs(1, 3, 4000, d, seed=d, device="cuda")
        mask = wl.block_mask_bigbird(32, heads=3, seed=d)
        mask[:, 5::7, :] = 1
        mask[:, 9::11, :] = 0
        keep(f"sparse_mixed_{d}_{int(causal)}", *fa.fa_fwd_sparse(q, k, v, mask.cuda(), causal=causal))
    for N, causal in ((1000, True), (777, False)):
        q, k, v = wl.prefill_inputs(1, 2, N, 128, seed=N, device="cuda")
        signs = (torch.randint(0, 2, (128,), generator=torch.Generator().manual_seed(N)) * 2 - 1).float().cuda()
        q8, qs = fa.fa_quantize_fp8(q, signs)
        k8, ks = fa.fa_quantize_fp8(k, signs)
        vt8, vs = fa.fa_quantize_fp8(v, None, per_head=True, transpose=True)
        keep(f"fp8_{N}_{int(causal)}", *fa.fa_fwd_fp8(q8, k8, vt8, qs, ks, vs, causal=causal))
    q, kc, vc, _ = wl.decode_inputs(3, 4, 1500, 128, seed=5, device="cuda")
    sl = torch.tensor([1500, 700, 3], dtype=torch.int32, device="cuda")
    keep("decode", *fa.fa_decode(q, kc, vc, sl, 5))
    for g, d in ((8, 128), (4, 64)):
        q, kc, vc, _ = wl.decode_gqa_inputs(2, 2 * g, 2, 1500, d, seed=g + d, device="cuda")
        sl = torch.tensor([1500, 260], dtype=torch.int32, device="cuda")
        keep(f"gqa_{g}_{d}", *fa.fa_decode_gqa(q, kc, vc, sl, 3))
    np.savez(out_path, **out)
    print("cases", len(out), "library", fa.LIB_PATH)


if __name__ == "__main__":
    main(sys.argv[1])
