"""The C ABI library on the CPU: it builds, loads, exports every declared symbol,
and rejects bad arguments before touching the GPU. No compute calls here."""
import ctypes
import json
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    from exact_attention_29_gb300 import build

    build.build()
    import exact_attention_29_gb300 as fa

    return fa.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:fa_status|int|const\s+char\s*\*)\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("fa_fwd", "fa_decode", "fa_status_string", "fa_check_device_error", "fa_last_error_site"):
        assert required in names
    # the error check takes the stream alone; the failing site has a call of its own
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    assert re.search(r"fa_status\s+fa_check_device_error\s*\(\s*fa_stream_t\s+stream\s*\)\s*;", text)


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert names
    for name in names:
        assert hasattr(lib, name), f"libfa.so does not export {name}"


def test_status_strings(lib):
    for code in range(6):
        s = lib.fa_status_string(code)
        assert s and s.startswith(b"FA_")
    assert lib.fa_status_string(99) == b"unknown fa_status"


def _fwd(lib, q=16, k=16, v=16, o=16, lse=16, B=1, H=1, N=128, d=64, causal=0, scale=0.125):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, None)


def test_fwd_rejects_bad_arguments(lib):
    import exact_attention_29_gb300 as fa

    assert _fwd(lib, q=None) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, lse=None) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, k=24) == fa.FA_ERR_INVALID_ARG  # not 16-byte aligned
    assert _fwd(lib, N=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, B=-1) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("inf")) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, causal=2) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, d=96) == fa.FA_ERR_UNSUPPORTED
    assert _fwd(lib, d=256) == fa.FA_ERR_UNSUPPORTED
    assert _fwd(lib, N=65536 * 256 + 1) == fa.FA_ERR_INVALID_ARG  # more Q-tile pairs than the grid allows
    # work items (batch x heads x Q-tile pairs) are counted in 32 bits
    assert _fwd(lib, B=32768, H=32768, N=512) == fa.FA_ERR_INVALID_ARG
    assert b"bh * pairs" in lib.fa_last_error_string()


def test_host_buffer_fwd_rejects_bad_arguments(lib):
    """Argument checks run before any CUDA call, so they need no GPU."""
    import exact_attention_29_gb300 as fa

    def fwd_host(q=16, k=16, v=16, o=16, lse=16, B=1, H=1, N=128, d=64, causal=0, scale=0.125):
        return lib.fa_fwd_host(q, k, v, o, lse, B, H, N, d, causal, scale, None)

    assert fwd_host(v=None) == fa.FA_ERR_INVALID_ARG
    assert fwd_host(o=None) == fa.FA_ERR_INVALID_ARG
    assert fwd_host(q=8) == fa.FA_ERR_INVALID_ARG  # host pointers are held to 16 bytes too
    assert fwd_host(lse=2) == fa.FA_ERR_INVALID_ARG
    assert fwd_host(H=0) == fa.FA_ERR_INVALID_ARG
    assert fwd_host(scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert fwd_host(causal=-1) == fa.FA_ERR_INVALID_ARG
    assert fwd_host(d=32) == fa.FA_ERR_UNSUPPORTED


def test_host_buffer_binding_rejects_device_or_strided_tensors():
    import exact_attention_29_gb300 as fa

    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_fwd_host(q.float(), q, q)
    with pytest.raises(ValueError):
        fa.fa_fwd_host(q, q.transpose(2, 3).contiguous(), q)
    with pytest.raises(ValueError):
        fa.fa_fwd_host(q.transpose(2, 3), q, q)
    with pytest.raises(ValueError):
        fa.fa_fwd_host(q, q, q, o=torch.zeros(1, 1, 8, 64), lse=torch.zeros(1, 1, 8))


@pytest.mark.parametrize("entry", ["fa_decode", "fa_decode_noalloc"])
def test_decode_rejects_bad_arguments(lib, entry):
    """Both decode entry points run the same checks, before any CUDA call, and
    leave the failed check's text for fa_last_error_string."""
    import exact_attention_29_gb300 as fa

    call = getattr(lib, entry)

    def dec(num_splits=8, d=128, L=64, seqlens=16, q=16, B=1, H=1):
        return call(q, 16, 16, seqlens, 16, 16, B, H, L, d, num_splits, None)

    assert dec(num_splits=0) == fa.FA_ERR_INVALID_ARG
    assert b"num_splits" in lib.fa_last_error_string()
    assert dec(num_splits=65) == fa.FA_ERR_INVALID_ARG
    assert dec(seqlens=None) == fa.FA_ERR_INVALID_ARG
    assert b"seqlens" in lib.fa_last_error_string()
    assert dec(q=8) == fa.FA_ERR_INVALID_ARG
    assert b"aligned16(q)" in lib.fa_last_error_string()
    assert dec(L=0) == fa.FA_ERR_INVALID_ARG
    assert dec(B=70000) == fa.FA_ERR_INVALID_ARG
    assert dec(d=80) == fa.FA_ERR_UNSUPPORTED
    assert b"d != 64" in lib.fa_last_error_string()


def test_noalloc_size_limit_is_checked_on_the_host(lib):
    """16 * 32 * 64 * 129 fp32 values exceed the 4,194,304 of the static array:
    rejected before any CUDA call, with the sizes in the text."""
    import exact_attention_29_gb300 as fa

    st = lib.fa_decode_noalloc(16, 16, 16, 16, 16, 16, 16, 32, 64, 128, 64, None)
    assert st == fa.FA_ERR_INVALID_ARG
    assert b"static workspace" in lib.fa_last_error_string()


def test_every_rejection_says_why(lib):
    """A rejected call always leaves its reason, not an earlier call's text."""
    import exact_attention_29_gb300 as fa

    assert lib.fa_decode_noalloc(16, 16, 16, 16, 16, 16, 16, 32, 64, 128, 64, None) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, causal=2) == fa.FA_ERR_INVALID_ARG
    assert b"causal" in lib.fa_last_error_string()
    assert lib.fa_bwd_plan(0, 64, 128, 0, None) == fa.FA_ERR_INVALID_ARG
    assert b"N < 1" in lib.fa_last_error_string()
    assert lib.fa_selftest_wait_timeout(0, None) == fa.FA_ERR_INVALID_ARG
    assert b"timeout_us" in lib.fa_last_error_string()
    assert lib.fa_last_error_site() == 0


def test_selftests_reject_bad_arguments(lib):
    import exact_attention_29_gb300 as fa

    assert lib.fa_selftest_wait_timeout(0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_selftest_wait_timeout(10_000_000, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_selftest_mma(6, 16, 16, 16, 128, 128, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_selftest_mma(-1, 16, 16, 16, 128, 128, None) == fa.FA_ERR_INVALID_ARG


def test_causal_block_plan_matches_the_page(lib):
    """CMU 15-779 Lecture 5 notes §6.2 and Exercise 5: T(T+1)/2 of T^2 block pairs
    are computed; T = 4 gives 10/16 and K/V bytes 524,288 -> 327,680; T = 8 gives
    36/64; T = 32 gives 51.6 %."""
    import exact_attention_29_gb300 as fa

    g = json.load(open(os.path.join(GOLDEN, "causal_block_counts.json")))
    for case in g["cases"]:
        tot, done = fa.fa_fwd_plan(case["N"], case["block"], causal=True)
        assert tot == case["T"] ** 2
        if "pairs_computed" in case:
            assert done == case["pairs_computed"] and tot == case["pairs_total"]
        if "kv_bytes_all" in case:
            per_pair = 2 * case["block"] * case["d"] * case["elem_bytes"]
            assert tot * per_pair == case["kv_bytes_all"] and done * per_pair == case["kv_bytes_computed"]
        if "fraction_percent" in case:
            assert round(100 * done / tot, 1) == case["fraction_percent"]
        tot_nc, done_nc = fa.fa_fwd_plan(case["N"], case["block"], causal=False)
        assert tot_nc == done_nc == tot


def test_plan_ragged_and_tiny(lib):
    import exact_attention_29_gb300 as fa

    assert fa.fa_fwd_plan(1, 128, True) == (1, 1)
    assert fa.fa_fwd_plan(129, 128, True) == (4, 3)
    assert fa.fa_fwd_plan(129, 128, False) == (4, 4)
    with pytest.raises(fa.FaError):
        fa.fa_fwd_plan(0, 128, False)


def test_io_model_matches_the_page():
    """Lecture 5 notes Exercise 4: 2Nd + 2Nd N/B_r + N = 34.6 M elements for
    N = 4096, d = 128, B_r = 128, of which about 97 % are K/V re-reads."""
    from exact_attention_29_gb300 import perfmodel

    g = json.load(open(os.path.join(GOLDEN, "io_counts.json")))
    total = perfmodel.fwd_hbm_elements_tiled(g["N"], g["d"], g["B_r"])
    assert total == sum(g["terms"].values())
    assert round(total / 1e6, 1) == g["total_millions_printed"]
    assert round(100 * g["terms"]["kv_rereads"] / total) == g["kv_share_percent_printed"]


def test_flop_model():
    from exact_attention_29_gb300 import perfmodel

    # Llama-3-8B-shaped prefill: 2 * 32 * 4096^2 * 128 * 2 (causal half of 4 N^2 d per head)
    assert perfmodel.fwd_flops(2, 32, 4096, 128, True) == 2 * 32 * 4096 ** 2 * 128 * 2
    assert perfmodel.fwd_flops(1, 1, 10, 8, False) == 4 * 100 * 8
    assert perfmodel.decode_kv_bytes(32, 128, [32768] * 16) == 16 * 32 * 32768 * 128 * 2 * 2


def test_package_import_does_not_need_the_library(monkeypatch):
    """Importing the binding is cheap; a missing library fails loudly on first use."""
    import importlib

    import exact_attention_29_gb300._lib as L

    monkeypatch.setattr(L, "LIB_PATH", "/nonexistent/libfa.so")
    monkeypatch.setattr(L, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        L.load_library()
    importlib.reload(L)


def test_bwd_atomic_plan_matches_the_page(lib):
    """Lecture 5 notes §7.4: ceil(N/B_c) * N * d dQ additions, 67,200 at N = 300, d = 32, B_c = 48."""
    import exact_attention_29_gb300 as fa

    g = json.load(open(os.path.join(GOLDEN, "bwd_atomics.json")))
    assert fa.fa_bwd_plan(g["N"], g["d"], g["B_c"], causal=False) == g["dq_atomic_adds"]
    # under the causal mask K/V tile j is seen by Q tiles j.. only
    assert fa.fa_bwd_plan(256, 8, 128, causal=True) == (256 + 128) * 8


def test_bwd_rejects_bad_arguments(lib):
    import exact_attention_29_gb300 as fa

    def bwd(q=16, d=128, N=128, scale=0.1, causal=0):
        return lib.fa_bwd(q, 16, 16, 16, 16, 16, 16, 16, 16, 1, 1, N, d, causal, scale, None)

    assert bwd(q=None) == fa.FA_ERR_INVALID_ARG
    assert bwd(q=8) == fa.FA_ERR_INVALID_ARG
    assert bwd(N=0) == fa.FA_ERR_INVALID_ARG
    assert bwd(scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert bwd(causal=3) == fa.FA_ERR_INVALID_ARG
    assert bwd(d=96) == fa.FA_ERR_UNSUPPORTED


def test_decode_gqa_rejects_bad_arguments(lib):
    import exact_attention_29_gb300 as fa

    def dec(Hq=8, Hkv=2, num_splits=4, d=128, L=64, q=16):
        return lib.fa_decode_gqa(q, 16, 16, 16, 16, 16, 1, Hq, Hkv, L, d, num_splits, None)

    assert dec(Hq=6, Hkv=4) == fa.FA_ERR_INVALID_ARG
    assert dec(Hkv=0) == fa.FA_ERR_INVALID_ARG
    assert dec(num_splits=0) == fa.FA_ERR_INVALID_ARG
    assert dec(num_splits=65) == fa.FA_ERR_INVALID_ARG
    assert dec(q=None) == fa.FA_ERR_INVALID_ARG
    assert dec(L=0) == fa.FA_ERR_INVALID_ARG
    assert dec(d=96) == fa.FA_ERR_UNSUPPORTED


def test_fp8_calls_reject_bad_arguments(lib):
    import exact_attention_29_gb300 as fa

    def quant(d=128, N=300, per_head=0, transpose=0, pitch=0, x=16):
        return lib.fa_quantize_fp8(x, None, 16, 16, 1, 1, N, d, per_head, transpose, pitch, None)

    assert quant(x=None) == fa.FA_ERR_INVALID_ARG
    assert quant(N=0) == fa.FA_ERR_INVALID_ARG
    assert quant(per_head=2) == fa.FA_ERR_INVALID_ARG
    assert quant(transpose=1, pitch=296) == fa.FA_ERR_INVALID_ARG  # below N
    assert quant(transpose=1, pitch=308) == fa.FA_ERR_INVALID_ARG  # not a multiple of 16
    assert quant(d=64) == fa.FA_ERR_UNSUPPORTED

    def fwd(d=128, N=300, pitch=304, scale=0.1, causal=0):
        return lib.fa_fwd_fp8(16, 16, 16, 16, 16, 16, 16, 16, 1, 1, N, d, causal, scale, pitch, None)

    assert fwd(pitch=296) == fa.FA_ERR_INVALID_ARG
    assert fwd(pitch=300) == fa.FA_ERR_INVALID_ARG
    assert fwd(scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert fwd(causal=5) == fa.FA_ERR_INVALID_ARG
    assert fwd(d=64) == fa.FA_ERR_UNSUPPORTED


def test_sparse_plan_matches_the_pages_counts(lib):
    """All-ones mask: every pair; under the causal rule T(T+1)/2 of T^2 (Lecture 5
    notes §6.2); a mask keeping 1/s of the blocks keeps 1/s of the pairs (the
    block-sparse extension: IO shrinks with the density)."""
    import numpy as np

    import exact_attention_29_gb300 as fa

    T, N = 8, 8 * 128
    ones = np.ones((T, T), np.uint8)
    assert fa.fa_fwd_sparse_plan(ones, 2, 3, N) == (2 * 3 * T * T, 2 * 3 * T * T)
    allowed, computed = fa.fa_fwd_sparse_plan(ones, 1, 1, N, causal=True)
    assert allowed == T * (T + 1) // 2 == 36
    # each Q tile computes exactly the pairs its mask (and the causal rule) keeps
    assert computed == allowed
    quarter = np.zeros((T, T), np.uint8)
    quarter[:, ::4] = 1
    allowed, _ = fa.fa_fwd_sparse_plan(quarter, 1, 1, N)
    assert allowed * 4 == T * T


def test_sparse_rejects_bad_arguments(lib):
    import exact_attention_29_gb300 as fa

    def sp(mask=16, mask_heads=1, H=2, d=128, scale=0.1, N=300):
        return lib.fa_fwd_sparse(16, 16, 16, mask, mask_heads, 16, 16, 1, H, N, d, 0, scale, None)

    assert sp(mask=None) == fa.FA_ERR_INVALID_ARG
    # step lists hold a K/V tile index + 1 in 16 bits: at most 65535 tiles of 128 keys
    assert sp(N=65535 * 128 + 1) == fa.FA_ERR_INVALID_ARG
    assert b"tiles_ll > 65535" in lib.fa_last_error_string()
    # work items (batch x heads x Q-tile pairs) are counted in 32 bits
    assert lib.fa_fwd_sparse(16, 16, 16, 16, 1, 16, 16, 32768, 32768, 512, 128, 0, 0.1, None) == fa.FA_ERR_INVALID_ARG
    assert b"bh * ((tiles_ll + 1) / 2)" in lib.fa_last_error_string()
    assert sp(mask_heads=3) == fa.FA_ERR_INVALID_ARG
    assert sp(scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert sp(d=96) == fa.FA_ERR_UNSUPPORTED
