"""GPU parity of the decoder backward (rlt_bptt) against the float64
autograd oracle (oracle/rlt_bptt.py).  The schedule and the device kernels
are also checked on the CPU (tests/test_bptt_schedule_cpu.py,
tests/test_bptt_kernels_emulated_cpu.py).

fp32 models: every gradient (all decoder parameters, s_*, e, the memory) and
the loss within fp32 tolerance, for full BPTT and each named detach point.
bf16 models: the oracle runs in float64 on the same bf16 weights and inputs;
the GPU rounds GEMM operands to bf16, so each gradient is compared by its
relative Frobenius error (about 3e-3 expected from the CPU check with bf16
storage rounding).  Both sides take the encoder output and memory from the
seeded input generator.  Runs are deterministic, and replaying the captured
steps equals launching every kernel one by one, bitwise.
"""
import numpy as np
import pytest
import torch

import rlt_inputs as ri
from oracle import rlt_bptt as BP
from oracle import rlt_oracle as O

pytestmark = pytest.mark.gpu

GRADS = ["W_g", "b_g", "W_qkv", "W_O", "W_Qx", "W_Ox", "W_1", "W_3", "W_2", "W_o", "dec_attn_norm",
         "dec_xattn_norm", "dec_ffn_norm", "head_norm", "s_star"]
F32_REL = 2e-3     # max-abs error relative to the gradient's max |value|
BF16_FRO = 2e-2    # relative Frobenius error per gradient (bf16 operands; ~3e-3 expected)


def _setup(dtype="f32", d=16, H=2, hd=8, f=24, V=9, L=2, G=1, window=3, gate_mode=0, B=2, T=8, seed=41, scale=4.0):
    c = ri.RLTConfig(d=d, n_layers=L, n_heads=H, head_dim=hd, d_ffn=f, window=window, mem_groups=G, vocab=V,
                     dtype=dtype, gate_mode=gate_mode)
    W = ri.make_weights(c, seed, norm_jitter=0.1)
    for k in W:
        if W[k].ndim >= 2:
            W[k] = W[k] * scale
    W["s_star"] = W["s_star"] * scale
    wl = ri.Workload("t", c, B=B, T=T, tokens="uniform5", split=(2, 2), seed=seed)
    tok = ri.make_tokens(wl)
    tok = ((tok + np.arange(T)[None, :] * 2) % V).astype(np.int32)
    acts = ri.teacher_actions(tok, 0, T)
    acts[:, -1] = (tok[:, -1] + 1) % V
    return c, W, tok, acts


def _inputs(c, B, T, seed=41, e_scale=1.0, mem_scale=0.5):
    return ri.make_decoder_inputs(c, B, T, seed + 7, e_scale=e_scale, mem_scale=mem_scale)


def _gpu(c, W, e, mem, acts, **kw):
    """rlt_bptt on seeded e / mem (the same values the oracle gets)."""
    import recurrent_looped_transformer_rlt_b300 as rlt
    from recurrent_looped_transformer_rlt_b300 import runner
    B, T = e.shape[0], e.shape[1]
    model = rlt.Model(c, W)
    buf = runner.alloc_buffers(model, B, T)
    buf.e.copy_(torch.from_numpy(e))
    buf.mem.copy_(torch.from_numpy(mem))
    res = runner.bptt(model, buf, torch.from_numpy(np.ascontiguousarray(acts)).cuda(), **kw)
    torch.cuda.synchronize()
    out = dict(loss=float(res.loss.item()), logp=res.logp.cpu().numpy(),
               grads={k: v.cpu().numpy() for k, v in res.grads.items()},
               d_e=res.d_e.cpu().numpy(), d_mem=res.d_mem.cpu().numpy(), status=rlt.rlt_status(buf.ws))
    model.close()
    return out


def _oracle(c, W, e, mem, acts, tau=1.0, k=0, **kw):
    cfg = O.Cfg.of(ri.RLTConfig(**{**c.__dict__, "dtype": "f32"}))  # bf16 weights and inputs, float64 arithmetic
    return BP.gradients(cfg, W, np.asarray(e, np.float64), np.asarray(mem, np.float64), acts, temperature=tau,
                        top_k=k, **kw)


def _max_rel(x, r):
    return np.abs(x - r).max() / max(np.abs(r).max(), 1e-30)


def _fro(x, r):
    return np.linalg.norm((x - r).ravel()) / max(np.linalg.norm(r.ravel()), 1e-30)


@pytest.mark.parametrize("case", [
    dict(),
    dict(window=1),
    dict(window=5, T=10),
    dict(gate_mode=1),
    dict(G=2),
    dict(L=3, B=3, window=4),
])
def test_fp32_full_bptt_matches_the_oracle(case):
    c, W, tok, acts = _setup(**case)
    e, mem = _inputs(c, *tok.shape)
    g = _gpu(c, W, e, mem, acts)
    lref, gref = _oracle(c, W, e, mem, acts)
    assert g["status"] == 0
    assert abs(g["loss"] - lref) <= 1e-4 * max(1.0, abs(lref))
    for k in GRADS:
        assert _max_rel(g["grads"][k], gref[k]) <= F32_REL or np.abs(gref[k]).max() == 0, k
    assert _max_rel(g["d_e"], gref["e"]) <= F32_REL
    assert _max_rel(g["d_mem"], gref["mem"]) <= F32_REL


@pytest.mark.parametrize("kw", [
    dict(detach_s_every=2),
    dict(detach_cache=True),
    dict(detach_memory=True),
    dict(detach_s_every=3, detach_cache=True, detach_memory=True),
])
def test_fp32_truncated_bptt_matches_the_oracle(kw):
    c, W, tok, acts = _setup(T=9)
    e, mem = _inputs(c, *tok.shape)
    g = _gpu(c, W, e, mem, acts, **kw)
    okw = {"detach_s_every": kw.get("detach_s_every", 0), "detach_cache": kw.get("detach_cache", False),
           "detach_memory": kw.get("detach_memory", False)}
    lref, gref = _oracle(c, W, e, mem, acts, **okw)
    for k in GRADS:
        assert _max_rel(g["grads"][k], gref[k]) <= F32_REL or np.abs(gref[k]).max() == 0, k
    assert _max_rel(g["d_e"], gref["e"]) <= F32_REL
    if kw.get("detach_memory"):
        assert not np.any(g["d_mem"])
    else:
        assert _max_rel(g["d_mem"], gref["mem"]) <= F32_REL


def test_fp32_tempered_top_k():
    c, W, tok, acts = _setup(T=8)
    cfg = O.Cfg.of(c)
    e, mem = _inputs(c, *tok.shape)
    _, out = O.decode_steps(cfg, W, O.init_state(cfg, W, tok.shape[0]), e, mem, acts.shape[1], acts, 0.7, 4)
    acts = np.where(np.isfinite(out.logp), acts, -1).astype(np.int32)  # in-set actions only
    g = _gpu(c, W, e, mem, acts, temperature=0.7, top_k=4)
    lref, gref = _oracle(c, W, e, mem, acts, tau=0.7, k=4)
    assert abs(g["loss"] - lref) <= 1e-4 * max(1.0, abs(lref))
    for k in GRADS:
        assert _max_rel(g["grads"][k], gref[k]) <= F32_REL or np.abs(gref[k]).max() == 0, k


@pytest.mark.parametrize("core_memgrad", [False, True])
def test_bf16_gradients_match_the_oracle_on_the_same_weights(core_memgrad):
    """Both memory-gradient kernels: the tensor-core one (default for bf16
    models) and the CUDA-core one (RLT_BPTT_CORE_MEMGRAD)."""
    c, W, tok, acts = _setup(dtype="bf16", d=256, H=8, hd=32, f=512, V=64, L=2, G=2, window=4, B=2, T=10, scale=1.0)
    e, mem = _inputs(c, *tok.shape)
    g = _gpu(c, W, e, mem, acts, core_memgrad=core_memgrad)
    lref, gref = _oracle(c, W, e, mem, acts)
    assert abs(g["loss"] - lref) <= 2e-3 * max(1.0, abs(lref))
    for k in GRADS:
        assert _fro(g["grads"][k], gref[k]) <= BF16_FRO, k
    assert _fro(g["d_e"], gref["e"]) <= BF16_FRO and _fro(g["d_mem"], gref["mem"]) <= BF16_FRO


def test_bptt_is_deterministic_and_its_logp_is_the_decoders():
    import recurrent_looped_transformer_rlt_b300 as rlt
    from recurrent_looped_transformer_rlt_b300 import runner
    c, W, tok, acts = _setup(dtype="bf16", d=256, H=8, hd=32, f=512, V=64, L=2, G=1, window=4, B=3, T=12, scale=1.0)
    e, mem = _inputs(c, *tok.shape)
    a, b = _gpu(c, W, e, mem, acts), _gpu(c, W, e, mem, acts)
    for k in GRADS:
        assert np.array_equal(a["grads"][k], b["grads"][k]), k
    assert np.array_equal(a["d_e"], b["d_e"]) and np.array_equal(a["d_mem"], b["d_mem"])
    # the loss's log-probabilities are the decoder's within the bf16 logit tolerance
    model = rlt.Model(c, W)
    buf = runner.alloc_buffers(model, 3, 12)
    buf.e.copy_(torch.from_numpy(e))
    buf.mem.copy_(torch.from_numpy(mem))
    st = runner.new_state(model, 3)
    out = runner.decode(model, st, buf, 12, torch.from_numpy(acts).cuda())
    lp = out.logp.cpu().numpy()
    model.close()
    assert np.abs(lp - a["logp"]).max() <= 5e-2


def test_argument_errors():
    import recurrent_looped_transformer_rlt_b300 as rlt
    from recurrent_looped_transformer_rlt_b300 import runner
    c, W, tok, acts = _setup()
    model = rlt.Model(c, W)
    buf = runner.alloc_buffers(model, 2, 8)
    runner.encode(model, torch.from_numpy(tok).cuda(), buf)
    nb = rlt.rlt_bptt_workspace_size(model.handle, 2, 8)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    grads = {k: torch.empty_like(model.t[k], dtype=torch.float32) for k in GRADS}
    cg = rlt.rlt_grads(*[grads[k].data_ptr() for k in GRADS])
    loss = torch.empty(1, device="cuda")
    A = torch.from_numpy(acts).cuda()
    call = lambda **o: rlt.rlt_bptt(model.handle, buf.e, buf.mem, o.get("T_mem", 8), 2, o.get("n", 8), A,
                                    o.get("tau", 1.0), o.get("k", 0), o.get("se", 0), o.get("fl", 0), loss, None, cg,
                                    None, None, ws, o.get("wsb", nb), check=False)
    assert call(n=9) == rlt.RLT_EINVAL               # n > T_mem
    assert call(tau=0.0) == rlt.RLT_EINVAL
    assert call(fl=16) == rlt.RLT_EINVAL             # no such flag
    assert call(se=-1) == rlt.RLT_EINVAL
    assert call(wsb=nb - 1) == rlt.RLT_EWORKSPACE
    assert call() == rlt.RLT_OK
    model.close()


def test_graph_replay_equals_eager_launches():
    """Steps captured once and replayed (the default) give bitwise the
    gradients of launching every kernel one by one."""
    c, W, tok, acts = _setup(dtype="bf16", d=256, H=8, hd=32, f=512, V=64, L=2, G=2, window=4, B=3, T=21, scale=1.0)
    e, mem = _inputs(c, *tok.shape)
    a = _gpu(c, W, e, mem, acts)
    b = _gpu(c, W, e, mem, acts, graphs=False)
    for k in GRADS:
        assert np.array_equal(a["grads"][k], b["grads"][k]), k
    assert np.array_equal(a["d_e"], b["d_e"]) and np.array_equal(a["d_mem"], b["d_mem"])
    assert a["loss"] == b["loss"]


@pytest.mark.parametrize("kw", [
    dict(T=1),                      # one step: a block of one
    dict(B=1, T=5),
    dict(window=1, T=6),
])
def test_fp32_edge_shapes(kw):
    c, W, tok, acts = _setup(**kw)
    e, mem = _inputs(c, *tok.shape)
    g = _gpu(c, W, e, mem, acts)
    lref, gref = _oracle(c, W, e, mem, acts)
    assert abs(g["loss"] - lref) <= 1e-4 * max(1.0, abs(lref))
    for k in GRADS:
        assert _max_rel(g["grads"][k], gref[k]) <= F32_REL or np.abs(gref[k]).max() == 0, k


def test_bf16_batch_past_one_k_block():
    """B = 70: two 64-row k-blocks per step slot in the weight-gradient GEMMs;
    tempered head (top-k is left to the fp32 tests: with near-equal logits
    bf16 rounding flips top-k membership, which is not a kernel error)."""
    c, W, tok, acts = _setup(dtype="bf16", d=256, H=8, hd=32, f=512, V=64, L=1, G=1, window=3, B=70, T=5, scale=1.0)
    e, mem = _inputs(c, *tok.shape)
    g = _gpu(c, W, e, mem, acts, temperature=0.8)
    lref, gref = _oracle(c, W, e, mem, acts, tau=0.8)
    assert abs(g["loss"] - lref) <= 2e-3 * max(1.0, abs(lref))
    for k in GRADS:
        assert _fro(g["grads"][k], gref[k]) <= BF16_FRO, k


@pytest.mark.parametrize("hd,T", [(64, 70), (128, 40)])
def test_bf16_tensor_core_memory_gradient_head_widths(hd, T):
    """The tensor-core memory gradient at head widths 64 and 128 over more
    keys than one 64-key block, against the CUDA-core kernel on the same
    inputs (relative Frobenius error of d_mem within bf16 operand rounding)."""
    c, W, tok, acts = _setup(dtype="bf16", d=256, H=256 // hd, hd=hd, f=256, V=64, L=1, G=1, window=4, B=2, T=T,
                             scale=1.0)
    e, mem = _inputs(c, *tok.shape)
    a = _gpu(c, W, e, mem, acts)
    b = _gpu(c, W, e, mem, acts, core_memgrad=True)
    assert _fro(a["d_mem"], b["d_mem"]) <= 1e-2
    lref, gref = _oracle(c, W, e, mem, acts)
    assert _fro(a["d_mem"], gref["mem"]) <= BF16_FRO
