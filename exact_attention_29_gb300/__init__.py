"""Exact attention on one GB300 (sm_103a): fused prefill forward and Flash-Decoding.

The compute path is ``libfa.so`` (hand-written CUDA: tcgen05 tensor cores,
TMEM accumulators, TMA pipelines); this package is its thin Python binding.
Importing the package does not load the library; the first call does, and
fails loudly if it has not been built.
"""
from ._lib import (  # noqa: F401
    FA_ERR_CHECK,
    FA_ERR_CUDA,
    FA_ERR_INVALID_ARG,
    FA_ERR_TIMEOUT,
    FA_ERR_UNSUPPORTED,
    FA_OK,
    LIB_PATH,
    FaError,
    fa_bwd,
    fa_bwd_plan,
    fa_check_device_error,
    fa_decode,
    fa_decode_gqa,
    fa_decode_noalloc,
    fa_fwd,
    fa_fwd_fp8,
    fa_fwd_host,
    fa_fwd_sparse,
    fa_fwd_sparse_plan,
    fa_last_error_site,
    fa_quantize_fp8,
    fa_fwd_plan,
    fa_selftest_mma,
    fa_selftest_wait_timeout,
    load_library,
)
