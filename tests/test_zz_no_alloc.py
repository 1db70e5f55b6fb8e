"""The allocation-free cross-attention entry point against the workspace one.

rlt_cross_attention_noalloc serves callers that cannot allocate device memory;
it keeps its partial results in a fixed array inside the library.  Its output
must match rlt_cross_attention (which uses a caller-provided workspace) within
the tolerances of the other GPU tests, call after call.  This file is collected
last so that a run stopping at the first failure has run every other test.
"""
import numpy as np
import pytest

import rlt_inputs as ri

pytestmark = pytest.mark.gpu

F32_ABS = 1e-4
BF16_REL = 2e-2


@pytest.mark.parametrize("name,B,T_mem,calls", [("small", 6, 300, [(129, 0), (300, 1)]),
                                                 ("tiny", 3, 64, [(64, 2), (1, 3)])])
def test_cross_attention_noalloc_matches_workspace_entry_point(name, B, T_mem, calls):
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    wl = ri.preset(name)
    c = wl.cfg
    model = rlt.Model(c, ri.make_weights(c, wl.seed))
    dt = model.dtype
    ws = model.workspace(B, T_mem)
    for t, seed in calls:       # two calls in a row, different inputs each time
        g = torch.Generator(device="cpu").manual_seed(seed)
        q = torch.randn(B, c.d, generator=g).cuda()
        km = torch.randn(B, c.n_heads, T_mem, c.head_dim, generator=g).to("cuda", dt)
        vm = torch.randn(B, c.n_heads, T_mem, c.head_dim, generator=g).to("cuda", dt)
        ref = torch.empty(B, c.d, dtype=dt, device="cuda")
        got = torch.full((B, c.d), float("nan"), dtype=dt, device="cuda")
        rlt.rlt_cross_attention(model.handle, q, km, vm, B, T_mem, t, ref, ws, ws.numel())
        rlt.rlt_cross_attention_noalloc(q, km, vm, B, c.n_heads, c.head_dim, model.ccfg.dtype, T_mem, t, got)
        torch.cuda.synchronize()
        r, o = ref.float().cpu().numpy(), got.float().cpu().numpy()
        assert np.isfinite(o).all()
        if c.dtype == "bf16":
            assert np.abs(o - r).max() <= BF16_REL * np.abs(r).max()
        else:
            assert np.abs(o - r).max() <= F32_ABS
    model.close()


def test_cross_attention_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    B, H, hd, T_mem = 64, 16, 128, 8192     # 64*16 pairs x 32 partials x 130 floats > 16 MiB
    q = torch.zeros(B, H * hd, device="cuda")
    km = torch.zeros(1, device="cuda", dtype=torch.bfloat16)
    out = torch.zeros(B, H * hd, device="cuda", dtype=torch.bfloat16)
    rc = rlt.rlt_cross_attention_noalloc(q, km, km, B, H, hd, rlt.RLT_BF16, T_mem, 1, out, check=False)
    assert rc == rlt.RLT_EUNSUPPORTED
