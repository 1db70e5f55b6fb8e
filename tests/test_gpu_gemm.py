"""The tensor-core projection kernel (tcgen05 + TMA) on its own, through the
C ABI entry rlt_linear, against a float64 CPU matmul of the same bf16 inputs.

Shapes cover the decoder's weight-streaming case (M = batch <= 128, K split
over CTAs), the encoder's many-row case (several 128-row tiles, ragged last
tile), ragged N and K (K not a multiple of the 64-wide k-block), and the
SwiGLU pair (gate and linear weights in one tile)."""
import numpy as np
import pytest

import rlt_inputs as ri

pytestmark = pytest.mark.gpu


def _model():
    import recurrent_looped_transformer_rlt_b300 as rlt
    wl = ri.preset("small")
    return rlt.Model(wl.cfg, ri.make_weights(wl.cfg, wl.seed))


@pytest.mark.parametrize("M,K,N,glu", [
    (64, 256, 768, False),     # decoder QKV of the small model, split K
    (64, 688, 256, False),     # ragged K (688 = 10.75 k-blocks)
    (8, 2048, 6144, False),    # few rows, long K
    (64, 256, 688, True),      # SwiGLU pair, ragged N
    (128, 1024, 2816, True),
    (300, 256, 1376, False),   # several row tiles, ragged rows and columns
    (1000, 512, 100, False),
    (1024, 128, 512, True),
    (5, 64, 32000, False),     # head-like: many column tiles
    (64, 128, 101, False),     # output rows not 16-byte aligned (scalar epilogue)
    (200, 192, 37, False),
])
def test_linear_matches_cpu_matmul(M, K, N, glu):
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    model = _model()
    g = torch.Generator().manual_seed(M * 7 + K * 3 + N)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    W3 = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16) if glu else None
    Ad, Wd = A.cuda(), W.cuda()
    W3d = W3.cuda() if glu else None
    C = torch.full((M, N), float("nan"), device="cuda")
    ws = model.workspace(1, 1)
    for _ in range(2):   # twice: the split-K counters must be reset by the kernel itself
        rlt.rlt_linear(model.handle, Ad, K, M, K, Wd, W3d, K, N, C, N, ws, ws.numel())
    torch.cuda.synchronize()
    ref = A.double() @ W.double().T
    if glu:
        lin = A.double() @ W3.double().T
        ref = torch.nn.functional.silu(ref) * lin
    got = C.cpu().double()
    assert torch.isfinite(got).all()
    err = (got - ref).abs().max().item()
    scale = ref.abs().max().item()
    assert err <= 1e-4 * scale + 1e-5, (err, scale)
    assert rlt.rlt_status(ws) == 0
    model.close()
