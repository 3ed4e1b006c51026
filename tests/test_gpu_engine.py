"""The weight-streaming tcgen05 GEMM alone (dflash_linear_bf16) against an fp64 matmul of
the same bf16 operands. fp32 accumulation of exact bf16 products: error ~ 1e-6 relative."""
import numpy as np
import pytest
import torch

from synth import W_TINY

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    from gpu_util import Setup
    return Setup(W_TINY, seed=11)


@pytest.mark.parametrize("n_out,K,rows", [
    (128, 64, 1), (128, 64, 16), (256, 256, 5), (200, 128, 17), (384, 4096, 16),
    (1024, 768, 3), (640, 1024, 64), (512, 512, 256), (4096, 4096, 16), (128, 20480, 16),
    (300, 192, 300),
])
def test_linear_matches_matmul(setup, n_out, K, rows):
    g = torch.Generator().manual_seed(n_out * 7 + K + rows)
    W = (0.02 * torch.randn(n_out, K, generator=g)).to(torch.bfloat16)
    X = torch.randn(rows, K, generator=g).to(torch.bfloat16)
    ref = (X.double() @ W.double().T).numpy()
    Y = torch.full((rows, n_out), float("nan"), device="cuda")
    setup.drafter.linear(W.cuda(), X.cuda(), Y)
    torch.cuda.synchronize()
    y = Y.cpu().double().numpy()
    assert np.isfinite(y).all()
    err = np.max(np.abs(y - ref)) / np.max(np.abs(ref))
    assert err < 1e-4, err
    assert setup.drafter.device_error() == 0


def test_linear_is_deterministic_and_row_independent(setup):
    g = torch.Generator().manual_seed(5)
    W = (0.02 * torch.randn(1024, 4096, generator=g)).to(torch.bfloat16).cuda()
    X = torch.randn(16, 4096, generator=g).to(torch.bfloat16).cuda()
    Y1 = torch.empty(16, 1024, device="cuda")
    Y2 = torch.empty(16, 1024, device="cuda")
    setup.drafter.linear(W, X, Y1)
    setup.drafter.linear(W, X, Y2)
    Y3 = torch.empty(1, 1024, device="cuda")
    setup.drafter.linear(W, X[5:6].contiguous(), Y3)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)
    assert torch.equal(Y1[5], Y3[0])
