"""GPU self-tests of the kernels' building blocks through the C ABI."""
import numpy as np
import pytest
import torch

from parity import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("k", [64, 128])
def test_mma_qk_k_major(k):
    """D = A B^T with both operands K-major in swizzled shared memory (the S = Q K^T product)."""
    import exact_attention_29_gb300 as fa

    a, b = _rand((128, k), 1), _rand((128, k), 2)
    d = fa.fa_selftest_mma(0, a.cuda(), b.cuda(), 128, k)
    fa.fa_check_device_error()
    ref = a.double() @ b.double().T
    err = (d.double().cpu() - ref).abs().max().item()
    assert err <= 1e-3, err


@pytest.mark.parametrize("n", [64, 128])
def test_mma_pv_tmem_a_mn_major_b(n):
    """D = A B with A (bf16 pairs) in tensor memory and B MN-major in shared memory (O += P V)."""
    import exact_attention_29_gb300 as fa

    a, b = _rand((128, 128), 3), _rand((128, n), 4)
    d = fa.fa_selftest_mma(1, a.cuda(), b.cuda(), n, 128)
    fa.fa_check_device_error()
    ref = a.double() @ b.double()
    err = (d.double().cpu() - ref).abs().max().item()
    assert err <= 1e-3, err


def _rand_e4m3(shape, seed):
    """e4m3 codes (uint8) and their values, from torch's float8_e4m3fn."""
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(shape, generator=g) * 8).to(torch.float8_e4m3fn)
    return x.view(torch.uint8), x.float().double()


@pytest.mark.parametrize("mode", [2, 3])
def test_mma_e4m3(mode):
    """D = A B^T with e4m3 operands (kind::f8f6f4): mode 2 both K-major in shared
    memory (S = Q K^T), mode 3 A in tensor memory, four values per column, and B
    K-major in shared memory (O += P V with V transposed)."""
    import exact_attention_29_gb300 as fa

    (a, av), (b, bv) = _rand_e4m3((128, 128), 5 + mode), _rand_e4m3((128, 128), 7 + mode)
    d = fa.fa_selftest_mma(mode, a.cuda(), b.cuda(), 128, 128)
    fa.fa_check_device_error()
    ref = av @ bv.T
    err = (d.double().cpu() - ref).abs().max().item()
    # products of e4m3 values are exact in fp32; 128-term fp32 sums of |terms| <= 448^2
    assert err <= 1e-6 * ref.abs().max().item() + 1e-3, err


@pytest.mark.parametrize("mode", [4, 5])
def test_mma_cta_pair(mode):
    """A cluster of two CTAs computes one M = 256 product (tcgen05 .cta_group::2):
    mode 4 D = A B^T with B K-major (S = Q K^T), mode 5 D = A B with B MN-major
    (O += P V with P in shared memory). Each CTA holds half of B and gets its
    128 rows of D; both see the same TMEM base address."""
    import exact_attention_29_gb300 as fa

    a, b = _rand((256, 128), 11 + mode), _rand((128, 128), 13 + mode)
    out = fa.fa_selftest_mma(mode, a.cuda(), b.cuda(), 128, 128)
    fa.fa_check_device_error()
    out = out.cpu()
    d = out[: 256 * 128].reshape(256, 128).double()
    bases = out[256 * 128:].view(torch.int32).tolist()
    ref = a.double() @ (b.double().T if mode == 4 else b.double())
    err = (d - ref).abs().max().item()
    assert err <= 1e-3, (err, bases)
    assert bases[0] == bases[1], bases


def test_bounded_wait_times_out_and_context_survives():
    """A wait on a barrier nothing arrives at gives up after its limit, the host
    reads FA_ERR_TIMEOUT, the word is cleared, and the GPU keeps working."""
    import exact_attention_29_gb300 as fa

    fa.fa_check_device_error()  # start clean
    fa.fa_selftest_wait_timeout(20_000)
    with pytest.raises(fa.FaError) as exc:
        fa.fa_check_device_error()
    assert exc.value.status == fa.FA_ERR_TIMEOUT and exc.value.site == 100
    assert fa.fa_last_error_site() == 100 and "site 100" in str(exc.value)
    assert fa.fa_check_device_error() == 0 and fa.fa_last_error_site() == 0
    x = torch.ones(1024, device="cuda")
    assert float(x.sum().item()) == 1024.0
