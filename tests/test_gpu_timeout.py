"""Bounded device waits: a wait whose arrival never comes gives up, the
kernel records RLT_ETIMEOUT in the workspace's status word, drains its other
copies, frees its tensor memory and returns; rlt_status reports it; the next
launch is unaffected.  The missing arrival is made on purpose with
rlt_debug_withhold_copy (a copy the kernel expects but never requests) and a
short wait budget, so nothing faults or hangs: each give-up takes a few
budgets of ~10 ms."""
import time

import numpy as np
import pytest
import torch

import rlt_inputs as ri

pytestmark = pytest.mark.gpu

BUDGET = 20_000_000   # clock cycles per wait (~10 ms at the B300's 2 GHz)


def _model(name="small", **over):
    import recurrent_looped_transformer_rlt_b300 as rlt
    wl = ri.preset(name, n_layers=1, mem_groups=1, vocab=64, **over)
    return rlt.Model(wl.cfg, ri.make_weights(wl.cfg, wl.seed)), wl.cfg


@pytest.mark.parametrize("M,K,N,glu", [
    (64, 4096, 256, False),     # few output tiles: split-K over a thread-block cluster
    (64, 256, 8192, False),     # many tiles, one CTA per tile
    (48, 2048, 688, True),      # SwiGLU pair tiles
])
def test_projection_wait_gives_up_and_reports_a_timeout(M, K, N, glu):
    import recurrent_looped_transformer_rlt_b300 as rlt
    model, _ = _model()
    g = torch.Generator(device="cuda").manual_seed(3)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    W3 = (torch.randn(N, K, device="cuda", generator=g) * 0.05).to(torch.bfloat16) if glu else None
    C = torch.empty(M, N, device="cuda")
    ws = model.workspace(1, 1)

    def call():
        rlt.rlt_linear(model.handle, A, K, M, K, W, W3, K, N, C, N, ws, ws.numel())

    call()
    assert rlt.rlt_status(ws) == rlt.RLT_OK
    ref = C.clone()
    y = A.double() @ W.double().T
    if glu:
        y = torch.nn.functional.silu(y) * (A.double() @ W3.double().T)
    assert (ref.double() - y).abs().max().item() <= 1e-3 * y.abs().max().item()
    rlt.rlt_debug_withhold_copy(model.handle, rlt.RLT_KERNEL_GEMM, BUDGET)
    C.fill_(0.0)
    t0 = time.perf_counter()
    call()
    assert rlt.rlt_status(ws) == rlt.RLT_ETIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert rlt.rlt_status(ws) == rlt.RLT_OK       # reading clears it
    call()                                        # one-shot: the next launch is whole again
    assert rlt.rlt_status(ws) == rlt.RLT_OK
    assert torch.equal(C, ref)
    model.close()


@pytest.mark.parametrize("name,B,T_mem,t", [
    ("small", 4, 1024, 1024),   # pairs split into segments merged through arrival counters
    ("small", 4, 1024, 5),      # one warp per pair
    ("refdep", 2, 512, 300),    # 128-wide heads
])
def test_attention_wait_gives_up_and_reports_a_timeout(name, B, T_mem, t):
    import recurrent_looped_transformer_rlt_b300 as rlt
    model, c = _model(name)
    g = torch.Generator(device="cuda").manual_seed(4)
    q = torch.randn(B, c.d, device="cuda", generator=g)
    mk = torch.randn(B, c.n_heads, T_mem, c.head_dim, device="cuda", generator=g).to(torch.bfloat16)
    mv = torch.randn(B, c.n_heads, T_mem, c.head_dim, device="cuda", generator=g).to(torch.bfloat16)
    out = torch.empty(B, c.d, device="cuda", dtype=torch.bfloat16)
    ws = model.workspace(B, T_mem)

    def call():
        rlt.rlt_cross_attention(model.handle, q, mk, mv, B, T_mem, t, out, ws, ws.numel())

    call()
    assert rlt.rlt_status(ws) == rlt.RLT_OK
    ref = out.clone()
    rlt.rlt_debug_withhold_copy(model.handle, rlt.RLT_KERNEL_XATTN, BUDGET)
    t0 = time.perf_counter()
    call()
    assert rlt.rlt_status(ws) == rlt.RLT_ETIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert rlt.rlt_status(ws) == rlt.RLT_OK
    call()
    assert rlt.rlt_status(ws) == rlt.RLT_OK
    assert torch.equal(out, ref)
    model.close()


def test_injection_arms_only_the_named_kernel():
    """Arming the projection leaves an attention launch alone (and the other
    way round); each arming is consumed by one launch of its own kernel."""
    import recurrent_looped_transformer_rlt_b300 as rlt
    model, c = _model()
    B, T_mem = 2, 64
    q = torch.randn(B, c.d, device="cuda")
    mk = torch.randn(B, c.n_heads, T_mem, c.head_dim, device="cuda").to(torch.bfloat16)
    mv = torch.randn(B, c.n_heads, T_mem, c.head_dim, device="cuda").to(torch.bfloat16)
    out = torch.empty(B, c.d, device="cuda", dtype=torch.bfloat16)
    ws = model.workspace(B, T_mem)
    rlt.rlt_debug_withhold_copy(model.handle, rlt.RLT_KERNEL_GEMM, BUDGET)
    rlt.rlt_cross_attention(model.handle, q, mk, mv, B, T_mem, T_mem, out, ws, ws.numel())
    assert rlt.rlt_status(ws) == rlt.RLT_OK
    rlt.rlt_debug_withhold_copy(model.handle, rlt.RLT_KERNEL_XATTN, BUDGET)   # replaces the GEMM arming
    A = torch.randn(64, c.d, device="cuda").to(torch.bfloat16)
    W = torch.randn(128, c.d, device="cuda").to(torch.bfloat16)
    C = torch.empty(64, 128, device="cuda")
    ws1 = model.workspace(1, 1)
    rlt.rlt_linear(model.handle, A, c.d, 64, c.d, W, None, c.d, 128, C, 128, ws1, ws1.numel())
    assert rlt.rlt_status(ws1) == rlt.RLT_OK
    rlt.rlt_cross_attention(model.handle, q, mk, mv, B, T_mem, T_mem, out, ws, ws.numel())
    assert rlt.rlt_status(ws) == rlt.RLT_ETIMEOUT
    model.close()


def test_decoder_norm_projection_wait_gives_up_and_reports_a_timeout():
    """The decoder's projections build their RMSNorm input in the kernel: the
    fp32 rows of a k-block land on their own barrier, a group of the
    epilogue warps converts them and adds its arrival to the stage.  With
    those rows never requested (layer-0 QKV projection of one step), the
    group and then the MMA give up, the launch drains and frees its tensor
    memory, the step reports RLT_ETIMEOUT, and the next call from the same
    starting state is bitwise the uninjected one."""
    import recurrent_looped_transformer_rlt_b300 as rlt
    from recurrent_looped_transformer_rlt_b300 import runner
    wl = ri.preset("small", n_layers=2, mem_groups=2)
    c = wl.cfg
    model = rlt.Model(c, ri.make_weights(c, wl.seed))
    B, T = 8, 16
    tok = ri.make_tokens(wl, B=B, T=T)
    buf = runner.alloc_buffers(model, B, T)
    runner.encode(model, torch.from_numpy(tok).cuda(), buf)
    acts = torch.from_numpy(ri.teacher_actions(tok, 0, T)).cuda()
    st0 = runner.new_state(model, B)
    runner.decode(model, st0, buf, 3, acts[:, :3].contiguous())
    assert runner.status(buf) == rlt.RLT_OK

    def step(st):
        return runner.decode(model, st, buf, 1, acts[:, 3:4].contiguous())

    st_ref = st0.clone()
    ref = step(st_ref)
    assert runner.status(buf) == rlt.RLT_OK
    rlt.rlt_debug_withhold_copy(model.handle, rlt.RLT_KERNEL_NORM_PROJ, BUDGET)
    t0 = time.perf_counter()
    step(st0.clone())
    assert runner.status(buf) == rlt.RLT_ETIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert runner.status(buf) == rlt.RLT_OK        # reading clears it
    st1 = st0.clone()
    again = step(st1)                              # one-shot: the next call is whole again
    assert runner.status(buf) == rlt.RLT_OK
    assert torch.equal(again.logp, ref.logp) and torch.equal(st1.s, st_ref.s)
    model.close()
