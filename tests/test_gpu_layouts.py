"""tcgen05 operand-layout self-test (GPU): one M=128 x N x K bf16 MMA per
combination of K-major / MN-major A and B, compared with an fp32 matmul of
the same bf16 operands."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K", [(16, 128), (32, 128), (48, 128), (64, 128), (128, 128),
                                 (32, 64), (64, 64), (128, 64), (256, 16)])
def test_tcgen05_layouts(kda_lib, N, K):
    import gated_delta_rule_30_gb300 as kda
    gen = torch.Generator().manual_seed(N * 1000 + K)
    a = torch.randn(128, K, generator=gen).to(torch.bfloat16)
    b = torch.randn(K, N, generator=gen).to(torch.bfloat16)
    d = kda.selftest_tcgen05(a.cuda(), b.cuda(), N, K).cpu()
    ref = a.double() @ b.double()
    names = ["A K-major, B K-major", "A MN-major, B MN-major", "A K-major, B MN-major",
             "A MN-major, B K-major"]
    errs = {names[c]: (d[c].double() - ref).abs().max().item() for c in range(4)}
    bound = 1e-3 * max(1.0, ref.abs().max().item())
    assert all(e < bound for e in errs.values()), f"max errors {errs} (bound {bound:.3g})"
