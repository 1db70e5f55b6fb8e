"""Pins of the BPTT oracle (oracle/rlt_bptt.py), CPU only.

Its forward is tied to rlt_oracle's recurrence, its gradients to central
finite differences of that forward, and its detach points to what the pages
say about them: detaching only s_t leaves gradient paths through the window
cache; with the cache (and the memory) also detached, nothing crosses a cut.
"""
import numpy as np
import pytest
import torch

import rlt_inputs as ri
from oracle import rlt_bptt as BP
from oracle import rlt_oracle as O


def _setup(window=3, gate_mode=0, T=6, B=2, seed=41, mem_groups=1, n_layers=2):
    c = ri.RLTConfig(d=16, n_layers=n_layers, n_heads=2, head_dim=8, d_ffn=24, window=window,
                     mem_groups=mem_groups, vocab=9, dtype="f32", gate_mode=gate_mode)
    W = ri.make_weights(c, seed, norm_jitter=0.1)
    for k in W:  # weights large enough that every path carries a visible gradient
        if W[k].ndim >= 2:
            W[k] = W[k] * 25.0
    W["s_star"] = W["s_star"] * 25.0
    wl = ri.Workload("t", c, B=B, T=T, tokens="uniform5", split=(2, 2), seed=seed)
    tok = ri.make_tokens(wl)
    tok = ((tok + np.arange(T)[None, :] * 2) % c.vocab).astype(np.int32)
    cfg = O.Cfg.of(c)
    e, mem = O.encode(cfg, W, tok)
    acts = ri.teacher_actions(tok, 0, T)
    acts[:, -1] = (tok[:, -1] + 1) % c.vocab  # score the last step too
    return cfg, W, e, mem, acts


@pytest.mark.parametrize("tau,k", [(1.0, 0), (0.7, 4)])
def test_forward_equals_the_recurrence_oracle(tau, k):
    cfg, W, e, mem, acts = _setup()
    st = O.init_state(cfg, W, e.shape[0])
    _, out = O.decode_steps(cfg, W, st, e, mem, acts.shape[1], acts, tau, k)
    ref = -np.nansum(np.where(np.isinf(out.logp), 0.0, out.logp))
    assert np.all(np.isfinite(out.logp[acts >= 0])) or k > 0
    P, et, mt = BP.leaves(W, e, mem)
    loss = float(BP.sequence_loss(cfg, P, et, mt, acts, temperature=tau, top_k=k).detach())
    if k == 0:
        np.testing.assert_allclose(loss, ref, rtol=1e-12)
    else:  # actions outside the top-k set score -inf in the oracle; here their term is dropped
        inset = np.isfinite(out.logp)
        ref_in = -np.sum(out.logp[inset])
        P2, et2, mt2 = BP.leaves(W, e, mem)
        acts2 = np.where(inset, acts, -1)
        np.testing.assert_allclose(
            float(BP.sequence_loss(cfg, P2, et2, mt2, acts2, temperature=tau, top_k=k).detach()), ref_in, rtol=1e-12)


def _fd(cfg, W, e, mem, acts, name, idx, h=1e-6, **kw):
    """Central difference of the loss in one entry of W[name], e or mem."""
    def loss_with(delta):
        W2 = {k: np.array(v, np.float64, copy=True) for k, v in W.items()}
        e2, m2 = np.array(e, np.float64, copy=True), np.array(mem, np.float64, copy=True)
        tgt = e2 if name == "e" else m2 if name == "mem" else W2[name]
        tgt[idx] += delta
        P, et, mt = BP.leaves(W2, e2, m2)
        with torch.no_grad():
            return float(BP.sequence_loss(cfg, P, et, mt, acts, **kw))
    return (loss_with(h) - loss_with(-h)) / (2 * h)


@pytest.mark.parametrize("G", [1, 2])
def test_full_bptt_gradients_match_central_differences(G):
    """Full BPTT is the derivative of the loss (a truncated gradient is by
    construction not, and is pinned by the structural tests below)."""
    kw = {}
    cfg, W, e, mem, acts = _setup(window=3, mem_groups=G)
    _, g = BP.gradients(cfg, W, e, mem, acts, **kw)
    probes = [("W_qkv", (1, 5, 3)), ("W_g", (3, 20)), ("b_g", (2,)), ("W_O", (0, 4, 9)), ("W_Qx", (1, 2, 2)),
              ("W_Ox", (0, 7, 1)), ("W_1", (1, 10, 3)), ("W_2", (0, 3, 11)), ("W_o", (4, 5)),
              ("dec_attn_norm", (1, 6)), ("head_norm", (3,)), ("s_star", (7,)), ("e", (1, 2, 5)),
              ("mem", (0, 1, 0, 1, 3, 4))]
    for name, idx in probes:
        fd = _fd(cfg, W, e, mem, acts, name, idx, **kw)
        ad = g[name][idx]
        assert abs(ad - fd) <= 1e-5 * max(1.0, abs(fd)), (name, idx, ad, fd)
    # a gradient that is not identically zero everywhere it should flow
    for name in ("W_qkv", "W_g", "s_star", "e", "mem"):
        assert np.abs(g[name]).max() > 1e-6, name


@pytest.mark.parametrize("kw", [dict(detach_s_every=2), dict(detach_s_every=1, detach_cache=True),
                                dict(detach_memory=True)])
def test_truncation_keeps_the_loss_and_cuts_paths(kw):
    cfg, W, e, mem, acts = _setup(window=3)
    l_full, g_full = BP.gradients(cfg, W, e, mem, acts)
    l_tr, g_tr = BP.gradients(cfg, W, e, mem, acts, **kw)
    assert l_full == l_tr
    cut = "mem" if kw.get("detach_memory") else "s_star"
    assert np.abs(g_full[cut] - g_tr[cut]).max() > 1e-6 * np.abs(g_full[cut]).max()


def _first_step_only(cfg, W, e, mem, acts):
    a1 = acts.copy()
    a1[:, 1:] = -1
    return BP.gradients(cfg, W, e, mem, a1, wrt=("s_star",))[1]["s_star"]


def test_detaching_s_alone_leaves_paths_through_the_cache():
    """With s_t detached after every step, s_* reaches later losses only
    through the window's keys and values: a nonzero gradient for W > 1, none
    once the cache is detached too, and none for W = 1 (no history)."""
    cfg, W, e, mem, acts = _setup(window=3)
    g_s = BP.gradients(cfg, W, e, mem, acts, wrt=("s_star",), detach_s_every=1)[1]["s_star"]
    g_1 = _first_step_only(cfg, W, e, mem, acts)
    assert np.abs(g_s - g_1).max() > 1e-4 * np.abs(g_1).max()
    g_sc = BP.gradients(cfg, W, e, mem, acts, wrt=("s_star",), detach_s_every=1, detach_cache=True)[1]["s_star"]
    np.testing.assert_allclose(g_sc, g_1, rtol=1e-12, atol=1e-14)
    cfg1, W1, e1, m1, a1 = _setup(window=1)
    g_w1 = BP.gradients(cfg1, W1, e1, m1, a1, wrt=("s_star",), detach_s_every=1)[1]["s_star"]
    np.testing.assert_allclose(g_w1, _first_step_only(cfg1, W1, e1, m1, a1), rtol=1e-12, atol=1e-14)


def test_gate_discard_cuts_every_path_from_the_start_state():
    """z = 0: s_t does not depend on s_{t-1}, so s_* has no gradient at all
    (any window: the cache entries are built from h, which no longer sees s)."""
    for w in (1, 3):
        cfg, W, e, mem, acts = _setup(window=w, gate_mode=1)
        g = BP.gradients(cfg, W, e, mem, acts, wrt=("s_star", "W_g"))[1]
        assert np.abs(g["s_star"]).max() == 0.0 and np.abs(g["W_g"]).max() == 0.0


def test_memory_gradient_is_causal_and_detachable():
    """The loss at step t reads memory positions 1..t only: a loss that ends at
    step t has no gradient on later memory positions; detach_memory removes it."""
    cfg, W, e, mem, acts = _setup(window=3, T=6)
    a = acts.copy()
    a[:, 3:] = -1  # only steps 1..3 scored
    g = BP.gradients(cfg, W, e, mem, a, wrt=("mem", "e"))[1]
    assert np.abs(g["mem"][..., :3, :]).max() > 0 and np.abs(g["mem"][..., 3:, :]).max() == 0.0
    assert np.abs(g["e"][:, 3:]).max() == 0.0 and np.abs(g["e"][:, :3]).max() > 0
    gd = BP.gradients(cfg, W, e, mem, a, wrt=("mem",), detach_memory=True)[1]
    assert np.abs(gd["mem"]).max() == 0.0


# ---------------------------------------------------------------------------
# the whole model: encoder and decoder, tied weights

@pytest.mark.parametrize("G,src", [(1, 0), (2, 1)])
def test_encoder_forward_equals_the_oracle_encoder(G, src):
    c = ri.RLTConfig(d=16, n_layers=2, n_heads=2, head_dim=8, d_ffn=24, window=3, mem_groups=G, vocab=9,
                     dtype="f32", mem_source=src)
    W = ri.make_weights(c, 5, norm_jitter=0.1)
    tok = (np.arange(14).reshape(2, 7) * 5 % 9).astype(np.int32)
    cfg = O.Cfg.of(c)
    e, mem = O.encode(cfg, W, tok)
    P = {k: torch.tensor(np.asarray(W[k], np.float64)) for k in BP.DECODER_PARAMS + BP.ENCODER_PARAMS}
    et, mt = BP.encode(cfg, P, tok)
    np.testing.assert_allclose(et.numpy(), e, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(mt.numpy(), mem, rtol=1e-12, atol=1e-12)


def _model_fd(cfg, W, tok, acts, name, idx, h=1e-6):
    def loss_with(delta):
        W2 = {k: np.array(v, np.float64, copy=True) for k, v in W.items()}
        W2[name][idx] += delta
        P = {k: torch.tensor(W2[k]) for k in BP.DECODER_PARAMS + BP.ENCODER_PARAMS}
        with torch.no_grad():
            e, mem = BP.encode(cfg, P, tok)
            return float(BP.sequence_loss(cfg, P, e, mem, acts))
    return (loss_with(h) - loss_with(-h)) / (2 * h)


def test_whole_model_gradients_match_central_differences():
    c = ri.RLTConfig(d=16, n_layers=2, n_heads=2, head_dim=8, d_ffn=24, window=3, mem_groups=2, vocab=9,
                     dtype="f32")
    W = ri.make_weights(c, 17, norm_jitter=0.1)
    for k in W:
        if W[k].ndim >= 2:
            W[k] = W[k] * 25.0
    tok = (np.arange(12).reshape(2, 6) * 4 % 9).astype(np.int32)
    acts = ri.teacher_actions(tok, 0, 6)
    cfg = O.Cfg.of(c)
    _, g = BP.model_gradients(cfg, W, tok, acts)
    for name, idx in [("tok_emb", (4, 3)), ("enc_attn_norm", (1, 2)), ("enc_ffn_norm", (0, 9)), ("enc_norm", (5,)),
                      ("W_K", (1, 3, 4)), ("W_V", (0, 6, 2)), ("W_qkv", (0, 17, 5)), ("W_2", (1, 2, 13)),
                      ("W_g", (1, 30)), ("W_o", (2, 7))]:
        fd = _model_fd(cfg, W, tok, acts, name, idx)
        assert abs(g[name][idx] - fd) <= 1e-5 * max(1.0, abs(fd)), (name, idx, g[name][idx], fd)


def test_tied_weights_collect_both_uses():
    """A tied matrix's gradient is the sum of its encoder use and its decoder
    use (each measured with the other's copy held constant)."""
    c = ri.RLTConfig(d=16, n_layers=2, n_heads=2, head_dim=8, d_ffn=24, window=3, mem_groups=1, vocab=9,
                     dtype="f32")
    W = ri.make_weights(c, 23, norm_jitter=0.1)
    tok = (np.arange(10).reshape(2, 5) * 2 % 9).astype(np.int32)
    acts = ri.teacher_actions(tok, 0, 5)
    cfg = O.Cfg.of(c)
    _, g = BP.model_gradients(cfg, W, tok, acts, wrt=("W_qkv", "W_2"))

    def split_use(which):
        P = {k: torch.tensor(np.asarray(W[k], np.float64), requires_grad=True)
             for k in BP.DECODER_PARAMS + BP.ENCODER_PARAMS}
        Pe = dict(P)
        Pd = dict(P)
        for k in ("W_qkv", "W_O", "W_1", "W_3", "W_2"):
            (Pd if which == "enc" else Pe)[k] = P[k].detach()
        e, mem = BP.encode(cfg, Pe, tok)
        loss = BP.sequence_loss(cfg, Pd, e, mem, acts)
        return [t.detach().numpy() for t in torch.autograd.grad(loss, [P["W_qkv"], P["W_2"]], allow_unused=True)]
    ge, gd = split_use("enc"), split_use("dec")
    for j, name in enumerate(("W_qkv", "W_2")):
        np.testing.assert_allclose(g[name], ge[j] + gd[j], rtol=1e-10, atol=1e-12)
        assert np.abs(ge[j]).max() > 0 and np.abs(gd[j]).max() > 0
