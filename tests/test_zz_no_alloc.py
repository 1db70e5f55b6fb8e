"""The allocation-free cross-attention entry point against the workspace one
and against the oracle.

rlt_cross_attention_noalloc serves callers that cannot allocate device memory;
it keeps its partial results in a fixed array inside the library.  Its output
must match rlt_cross_attention (which uses a caller-provided workspace) within
the tolerances of the other GPU tests, call after call, and the oracle's
attention at the shapes that reach its ring depths and the edge of its array.
This file is collected last so that a run stopping at the first failure has
run every other test.
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


def _oracle_xattn(q, km, vm, t):
    """Cross-attention of every (sequence, head) over memory positions 1..t,
    float64 (the oracle's attention step)."""
    from oracle import rlt_oracle as O
    B, H, _, hd = km.shape
    return O.swa_attend(q.reshape(B, H, hd).astype(np.float64), km[:, :, :t].astype(np.float64),
                        vm[:, :, :t].astype(np.float64), hd).reshape(B, H * hd)


@pytest.mark.parametrize("B,H,hd,T_mem,ts", [
    (5, 4, 64, 1024, [1000, 517]),     # heads up to 64 wide over >= 512 positions: the 3-stage ring
    (53, 19, 128, 2048, [2048, 33]),   # 1007 (sequence, head) pairs: the most the built-in array holds at hd 128
])
def test_cross_attention_noalloc_matches_the_oracle(B, H, hd, T_mem, ts):
    """Shapes passed directly (no model): each call against the oracle's
    attention on the same bf16 inputs, two calls in a row with different
    inputs, then the status word is clean."""
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    for i, t in enumerate(ts):
        g = torch.Generator(device="cpu").manual_seed(10 + i)
        q = torch.randn(B, H * hd, generator=g)
        km = torch.randn(B, H, T_mem, hd, generator=g).to(torch.bfloat16)
        vm = torch.randn(B, H, T_mem, hd, generator=g).to(torch.bfloat16)
        out = torch.full((B, H * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
        rlt.rlt_cross_attention_noalloc(q.cuda(), km.cuda(), vm.cuda(), B, H, hd, rlt.RLT_BF16, T_mem, t, out)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        ref = _oracle_xattn(q.numpy(), km.float().numpy(), vm.float().numpy(), t)
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() <= BF16_REL * np.abs(ref).max()
    assert rlt.rlt_cross_attention_noalloc_status() == rlt.RLT_OK


def test_cross_attention_noalloc_limit_is_exact():
    """1008 pairs at head width 128 no longer fit: rejected before any launch."""
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    B, H, hd = 63, 16, 128
    q = torch.zeros(B, H * hd, device="cuda")
    km = torch.zeros(1, device="cuda", dtype=torch.bfloat16)
    out = torch.zeros(B, H * hd, device="cuda", dtype=torch.bfloat16)
    assert rlt.rlt_cross_attention_noalloc(q, km, km, B, H, hd, rlt.RLT_BF16, 64, 1, out,
                                           check=False) == rlt.RLT_EUNSUPPORTED


def test_cross_attention_noalloc_on_a_second_device():
    """The built-in array's address and the kernel's shared-memory attribute
    are set up per device: a call on device 1 after calls on device 0."""
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    if torch.cuda.device_count() < 2:
        pytest.skip("one visible GPU")
    B, H, hd, T_mem = 2, 4, 32, 96
    for dev in (0, 1):
        with torch.cuda.device(dev):
            g = torch.Generator(device="cpu").manual_seed(dev)
            q = torch.randn(B, H * hd, generator=g)
            km = torch.randn(B, H, T_mem, hd, generator=g).to(torch.bfloat16)
            vm = torch.randn(B, H, T_mem, hd, generator=g).to(torch.bfloat16)
            out = torch.empty(B, H * hd, dtype=torch.bfloat16, device=f"cuda:{dev}")
            rlt.rlt_cross_attention_noalloc(q.to(f"cuda:{dev}"), km.to(f"cuda:{dev}"), vm.to(f"cuda:{dev}"), B, H,
                                            hd, rlt.RLT_BF16, T_mem, T_mem, out)
            assert rlt.rlt_cross_attention_noalloc_status() == rlt.RLT_OK
            ref = _oracle_xattn(q.numpy(), km.float().numpy(), vm.float().numpy(), T_mem)
            assert np.abs(out.float().cpu().numpy() - ref).max() <= BF16_REL * np.abs(ref).max()
