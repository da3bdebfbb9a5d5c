"""GPU self-test of the tcgen05 operand layouts (K-major / MN-major 128-byte
swizzled tiles, TMA-staged tiles, negated A) against a host matmul.  The fused
kernel builds every one of its MMAs from these layouts."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_chunked_gdn_gb300 import binding
    lib = binding.load()
    lib.gdn_selftest_umma.argtypes = [ctypes.c_int] + [ctypes.c_void_p] * 5
    lib.gdn_selftest_umma.restype = ctypes.c_int
    return lib


VARIANTS = [v for v in range(64) if not ((v >> 5) & 1 and v & 1)]


@pytest.mark.parametrize("variant", VARIANTS)
def test_umma_layout(lib, variant):
    N = 128 if variant & 4 else 64
    Kd = 128 if variant & 8 else 64
    gen = torch.Generator(device="cpu").manual_seed(1000 + variant)
    A = torch.randn(128, Kd, generator=gen).to(torch.bfloat16)
    B = torch.randn(Kd, N, generator=gen).to(torch.bfloat16)
    dA, dB = A.cuda(), B.cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    ws = torch.zeros(64, dtype=torch.int32, device="cuda")
    st = lib.gdn_selftest_umma(variant, dA.data_ptr(), dB.data_ptr(), D.data_ptr(), ws.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(ws[0]) == 0
    ref = A.double() @ B.double()
    if variant & 16:
        ref = -ref
    err = (D.double().cpu() - ref).abs().max().item()
    assert err < 1e-3 * max(1.0, ref.abs().max().item()), err


def test_fast_exp_against_cuda_expf(lib):
    """The fused kernel's e^x (2^{x log2 e} on ex2.approx) against CUDA's expf
    (torch.exp on the GPU) over the argument range of the decay factors: the
    relative error stays within 1e-5, results below the normal fp32 range
    flush to zero."""
    lib.gdn_selftest_exp.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    lib.gdn_selftest_exp.restype = ctypes.c_int
    x = torch.cat([torch.linspace(-87.0, 0.0, 200001), torch.linspace(-1e-3, 0.0, 1001),
                   torch.tensor([-103.0, -88.5, -200.0])]).cuda()
    y = torch.empty_like(x)
    assert lib.gdn_selftest_exp(x.data_ptr(), y.data_ptr(), x.numel(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    ref = torch.exp(x)
    normal = ref >= torch.finfo(torch.float32).tiny
    rel = ((y[normal].double() - ref[normal].double()).abs() / ref[normal].double()).max().item()
    assert rel < 1e-5, rel
    assert torch.all(y[~normal] <= ref[~normal] * 1.0001 + 1e-38)
    assert torch.all(y >= 0)
