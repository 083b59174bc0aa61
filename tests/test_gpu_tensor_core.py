"""The tcgen05 MMA path (shared-memory descriptors, A from shared or tensor
memory, bounded completion wait) against an fp64 matmul of the same bf16
operands (GPU)."""
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from sparse_attention_kv_skv_gb300 import skv


@pytest.mark.parametrize("a_tmem", [0, 1])
@pytest.mark.parametrize("mn_major", [0, 1])
@pytest.mark.parametrize("n,k", [(16, 16), (32, 64), (64, 128), (128, 32), (256, 128), (48, 80), (256, 32)])
def test_selftest_mma_matches_matmul(n, k, mn_major, a_tmem):
    g = torch.Generator(device="cuda").manual_seed(n * 1000 + k)
    a = torch.randn(128, k, device="cuda", generator=g).to(torch.bfloat16)
    b = torch.randn(n, k, device="cuda", generator=g).to(torch.bfloat16)
    src = b.t().contiguous() if mn_major else b          # [k][n] when staged MN-major
    d = torch.full((128, n), float("nan"), device="cuda")
    skv.check(skv.skv_selftest_mma(a.data_ptr(), src.data_ptr(), d.data_ptr(), n, k, mn_major | (2 * a_tmem),
                                   torch.cuda.current_stream().cuda_stream), "skv_selftest_mma")
    ref = a.double() @ b.double().t()
    # products of bf16 values are exact in fp32; only the fp32 sum order differs
    assert torch.allclose(d.double(), ref, rtol=1e-5, atol=1e-4 * k ** 0.5), (d - ref).abs().max()
