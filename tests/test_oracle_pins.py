"""Pins of the CPU oracle to things other than itself (CPU only).

Each test ties one part of the oracle to a library routine, a closed form, an
invariant the pages state, or a brute-force construction; the planted-mistake
tests at the end check that plausible slips in the oracle fail at least one pin.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import rlt_inputs as ri
from oracle import rlt_oracle as O
from tests import _torch_ref as TR


def tiny_cfg(**kw):
    base = dict(d=32, n_layers=2, n_heads=4, head_dim=8, d_ffn=48, window=3, mem_groups=1,
                vocab=11, dtype="f32", rms_eps=1e-6, rope_theta=1e4, gate_mode=0, mem_source=0)
    base.update(kw)
    c = ri.RLTConfig(**{k: v for k, v in base.items()})
    return c


def setup(seed=100, B=3, Tn=7, jitter=0.1, gate_bias=0.0, **kw):
    c = tiny_cfg(**kw)
    W = ri.make_weights(c, seed, norm_jitter=jitter, gate_bias=gate_bias)
    # larger weights than N(0, 0.02) so every term matters at these tiny sizes
    for k in W:
        if W[k].ndim >= 2:
            W[k] = W[k] * 20.0
    W["s_star"] = W["s_star"] * 20.0
    wl = ri.Workload("t", c, B=B, T=Tn, tokens="uniform5", split=(2, 2), seed=seed)
    tok = ri.make_tokens(wl)
    tok = (tok + np.arange(Tn)[None, :] * 3) % c.vocab
    return O.Cfg.of(c), W, tok.astype(np.int32)


# ---------------------------------------------------------------------------
# elementary operations

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(100000).astype(np.float32).astype(np.float64) * 10.0 ** rng.integers(-6, 6, 100000)
    x = x.astype(np.float32).astype(np.float64)
    ref = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16(x), ref)
    # exact ties round to even
    one = 1.0
    assert O.bf16(one + 2.0 ** -8) == 1.0
    assert O.bf16(one + 3 * 2.0 ** -8) == one + 2.0 ** -6
    assert O.bf16(-(one + 2.0 ** -8)) == -1.0


def test_rmsnorm_matches_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 37))
    g = rng.standard_normal(37)
    ref = F.rms_norm(torch.tensor(x), (37,), weight=torch.tensor(g), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rmsnorm(x, g, 1e-6), ref, rtol=1e-13, atol=1e-13)
    # constant row c -> sign(c) * g (up to eps)
    np.testing.assert_allclose(O.rmsnorm(np.full((1, 8), -3.0), np.ones(8), 0.0), -np.ones((1, 8)))


def test_rope_complex_form_and_invariants():
    rng = np.random.default_rng(2)
    hd, P = 16, 9
    x = rng.standard_normal((2, 3, P, hd))
    pos = np.arange(P) * 37 + 5
    ref = TR.rope_complex(torch.tensor(x), pos, 1e4).numpy()
    y = O.rope(x, pos, 1e4)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    # p = 0 is the identity; rotations keep the norm
    np.testing.assert_array_equal(O.rope(x[..., :1, :], [0], 1e4), x[..., :1, :])
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    # <R(q,p1), R(k,p2)> depends only on p1 - p2
    q, k = rng.standard_normal(hd), rng.standard_normal(hd)
    d1 = O.rope(q[None], [40], 1e4)[0] @ O.rope(k[None], [33], 1e4)[0]
    d2 = O.rope(q[None], [7], 1e4)[0] @ O.rope(k[None], [0], 1e4)[0]
    assert abs(d1 - d2) < 1e-10


def test_causal_attention_matches_sdpa():
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((13, 8)) for _ in range(3))
    nx = O.Numerics(False)
    ref = F.scaled_dot_product_attention(torch.tensor(q)[None], torch.tensor(k)[None],
                                         torch.tensor(v)[None], is_causal=True)[0].numpy()
    np.testing.assert_allclose(O.causal_attention(q, k, v, nx, False), ref, rtol=1e-12, atol=1e-12)


def test_softmax_and_lse():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((4, 50)) * 30
    np.testing.assert_allclose(O.softmax_last(x).sum(-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(O.logsumexp_last(x), scipy.special.logsumexp(x, axis=-1), rtol=1e-14)


# ---------------------------------------------------------------------------
# encoder and memory

@pytest.mark.parametrize("G,src", [(1, 0), (2, 0), (2, 1)])
def test_encoder_matches_library_composition(G, src):
    cfg, W, tok = setup(mem_groups=G, mem_source=src)
    e, mem = O.encode(cfg, W, tok)
    e_ref, mem_ref = TR.encoder(cfg, W, tok)
    np.testing.assert_allclose(e, e_ref, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(mem, mem_ref, rtol=1e-11, atol=1e-11)
    assert mem.shape == (G, 2, tok.shape[0], cfg.n_heads, tok.shape[1], cfg.head_dim)


def test_encoder_cache_matches_library_composition():
    """The encoder keys (after RoPE) and values that incremental encoding of
    later tokens attends to: every layer's, equal to the torch composition's
    (complex-form RoPE, scaled_dot_product_attention), and causal - those of
    a prefix equal the prefix of those of the whole sequence."""
    cfg, W, tok = setup(mem_groups=2, mem_source=1)
    e, mem, kv = O.encode(cfg, W, tok, return_kv=True)
    e_ref, mem_ref, kv_ref = TR.encoder(cfg, W, tok, return_kv=True)
    assert kv.shape == (cfg.n_layers, 2, tok.shape[0], cfg.n_heads, tok.shape[1], cfg.head_dim)
    np.testing.assert_allclose(kv, kv_ref, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(e, e_ref, rtol=1e-11, atol=1e-11)
    _, _, kv4 = O.encode(cfg, W, tok[:, :4], return_kv=True)
    np.testing.assert_array_equal(kv4, kv[:, :, :, :, :4])


def test_per_layer_memory_reading():
    """Group l from encoder layer l (the other reading of per-layer memory):
    the last group is the final-e group, a single-layer encoder gives the same
    memory under both readings, and group l does not depend on encoder layers
    after l."""
    cfg0, W, tok = setup(mem_groups=2, mem_source=0)
    cfg1, _, _ = setup(mem_groups=2, mem_source=1)
    e0, m0 = O.encode(cfg0, W, tok)
    e1, m1 = O.encode(cfg1, W, tok)
    np.testing.assert_array_equal(e0, e1)
    np.testing.assert_array_equal(m0[1], m1[1])
    assert np.abs(m0[0] - m1[0]).max() > 1e-3 * np.abs(m0[0]).max()
    c1a, W1, tok1 = setup(n_layers=1, mem_groups=1, mem_source=0)
    c1b, _, _ = setup(n_layers=1, mem_groups=1, mem_source=1)
    np.testing.assert_array_equal(O.encode(c1a, W1, tok1)[1], O.encode(c1b, W1, tok1)[1])
    W2 = {k: v.copy() for k, v in W.items()}
    for name in ("W_qkv", "W_O", "W_1", "W_3", "W_2", "enc_attn_norm", "enc_ffn_norm"):
        W2[name][1] = W2[name][1] * 1.5 + 0.01
    _, m2 = O.encode(cfg1, W2, tok)
    np.testing.assert_array_equal(m1[0], m2[0])
    assert np.abs(m1[1] - m2[1]).max() > 1e-3 * np.abs(m1[1]).max()


def test_memory_depends_only_on_tokens():
    cfg, W, tok = setup()
    e, mem = O.encode(cfg, W, tok)
    W2 = dict(W)
    for name in ("s_star", "W_g", "b_g", "W_Qx", "W_Ox", "dec_attn_norm", "dec_xattn_norm",
                 "dec_ffn_norm", "head_norm", "W_o"):
        W2[name] = W[name] + 0.5
    e2, mem2 = O.encode(cfg, W2, tok)
    assert np.array_equal(e, e2) and np.array_equal(mem, mem2)
    # causal: positions <= t are unchanged when tokens after t change
    t = 3
    tok2 = tok.copy()
    tok2[:, t + 1:] = (tok2[:, t + 1:] + 1) % cfg.vocab
    e3, mem3 = O.encode(cfg, W, tok2)
    assert np.array_equal(e3[:, : t + 1], e[:, : t + 1])
    assert np.array_equal(mem3[..., : t + 1, :], mem[..., : t + 1, :])
    assert not np.allclose(e3[:, t + 1:], e[:, t + 1:])


# ---------------------------------------------------------------------------
# decoder recurrence

def _merge_torch(W, e_t, s_prev):
    x = torch.cat([TR.T(e_t), TR.T(s_prev)], dim=-1)
    z = torch.sigmoid(F.linear(x, TR.T(W["W_g"]), TR.T(W["b_g"])))
    return (z * TR.T(s_prev) + (1 - z) * TR.T(e_t)).numpy()


def brute_force_states(cfg, W, e, mem, n):
    """s_1..s_n by brute force: at step t rebuild every decoder activation from scratch
    with a token-parallel pass over u_1..u_t, where u_i = Merge(e_i, s_{i-1})."""
    B = e.shape[0]
    s = np.broadcast_to(W["s_star"], (B, cfg.d)).astype(np.float64)
    us, out = [], []
    for t in range(1, n + 1):
        if cfg.gate_mode == 1:
            u_t = np.asarray(e[:, t - 1], np.float64)
        else:
            u_t = _merge_torch(W, e[:, t - 1], s)
        us.append(u_t)
        H = TR.parallel_decoder(cfg, W, e[:, :t], mem, cfg.window, u=np.stack(us, axis=1))
        s = H[:, t - 1]
        out.append(s)
    return np.stack(out, axis=1)


@pytest.mark.parametrize("window", [1, 2, 3, 4, 5, 16])
@pytest.mark.parametrize("G", [1, 2])
def test_recurrence_equals_brute_force(window, G):
    cfg, W, tok = setup(window=window, mem_groups=G, Tn=8)
    e, mem = O.encode(cfg, W, tok)
    st = O.init_state(cfg, W, tok.shape[0])
    st, out = O.decode_steps(cfg, W, st, e, mem, tok.shape[1], keep_s=True)
    S = np.stack(out.s_hist, axis=1)
    ref = brute_force_states(cfg, W, e, mem, tok.shape[1])
    np.testing.assert_allclose(S, ref, rtol=1e-10, atol=1e-10)


def test_hand_unrolled_three_steps():
    """T=3, W=2: written out step by step (the window drops x_1 at step 3)."""
    cfg, W, tok = setup(window=2, Tn=3)
    e, mem = O.encode(cfg, W, tok)
    s0 = np.broadcast_to(W["s_star"], (tok.shape[0], cfg.d)).astype(np.float64)
    u1 = _merge_torch(W, e[:, 0], s0)
    s1 = TR.parallel_decoder(cfg, W, e[:, :1], mem, 2, u=u1[:, None])[:, 0]
    u2 = _merge_torch(W, e[:, 1], s1)
    s2 = TR.parallel_decoder(cfg, W, e[:, :2], mem, 2, u=np.stack([u1, u2], 1))[:, 1]
    u3 = _merge_torch(W, e[:, 2], s2)
    s3 = TR.parallel_decoder(cfg, W, e[:, :3], mem, 2, u=np.stack([u1, u2, u3], 1))[:, 2]
    st = O.init_state(cfg, W, tok.shape[0])
    st1 = O.decode_step(cfg, W, st, e[:, 0], mem)
    st2 = O.decode_step(cfg, W, st1, e[:, 1], mem)
    st3 = O.decode_step(cfg, W, st2, e[:, 2], mem)
    for a, b in ((st1.s, s1), (st2.s, s2), (st3.s, s3)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-10)
    assert [len(c) for c in st3.cache] == [1] * cfg.n_layers


@pytest.mark.parametrize("window", [1, 2, 4, 64])
def test_gate_discard_equals_parallel_pass(window):
    """z = 0 makes u_t = e_t: the recurrence equals one token-parallel decoder pass
    (the W >= t case is full causal attention over decoder history)."""
    cfg, W, tok = setup(window=window, gate_mode=1, Tn=9)
    e, mem = O.encode(cfg, W, tok)
    st = O.init_state(cfg, W, tok.shape[0])
    st, out = O.decode_steps(cfg, W, st, e, mem, tok.shape[1], keep_s=True)
    S = np.stack(out.s_hist, axis=1)
    H = TR.parallel_decoder(cfg, W, e, mem, window)
    np.testing.assert_allclose(S, H, rtol=1e-10, atol=1e-10)
    lg = O.head_logits(cfg, W, S)
    np.testing.assert_allclose(lg, TR.head_logits(cfg, W, H), rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("window", [1, 4])
def test_learned_gate_not_a_parallel_pass(window):
    """With the learned gate the feedback path is live: a parallel SWA pass differs."""
    cfg, W, tok = setup(window=window, gate_mode=0, Tn=9)
    e, mem = O.encode(cfg, W, tok)
    st = O.init_state(cfg, W, tok.shape[0])
    st, out = O.decode_steps(cfg, W, st, e, mem, tok.shape[1], keep_s=True)
    S = np.stack(out.s_hist, axis=1)
    H = TR.parallel_decoder(cfg, W, e, mem, window)
    assert np.max(np.abs(S - H)) > 1e-2 * np.max(np.abs(S))


def test_merge_closed_forms():
    cfg, W, tok = setup(Tn=2)
    e, mem = O.encode(cfg, W, tok)
    st = O.init_state(cfg, W, tok.shape[0])
    # W_g = 0, b_g = c: z = sigmoid(c) exactly, u = z s + (1 - z) e
    W0 = dict(W)
    W0["W_g"] = np.zeros_like(W["W_g"])
    W0["b_g"] = np.full_like(W["b_g"], 0.7)
    tr = {}
    O.decode_step(cfg, W0, st, e[:, 0], mem, trace=tr)
    z = 1 / (1 + math.exp(-float(W0["b_g"][0])))
    np.testing.assert_allclose(tr["z"], z, rtol=1e-15)
    np.testing.assert_allclose(tr["u"], z * st.s + (1 - z) * e[:, 0], rtol=1e-13)
    # the gate reads [e; s] with e first: zero the s half, z depends on e only
    W1 = dict(W)
    W1["W_g"] = W["W_g"].copy()
    W1["W_g"][:, cfg.d:] = 0
    tr = {}
    O.decode_step(cfg, W1, st, e[:, 0], mem, trace=tr)
    ref = scipy.special.expit(e[:, 0] @ W["W_g"][:, : cfg.d].T.astype(np.float64))
    np.testing.assert_allclose(tr["z"], ref, rtol=1e-13)


def test_window_one_ignores_queries_and_keys():
    """W = 1: attention is over the current entry only, so q and k rows of W_qkv are dead."""
    cfg, W, tok = setup(window=1)
    e, mem = O.encode(cfg, W, tok)
    W2 = dict(W)
    W2["W_qkv"] = W["W_qkv"].copy()
    W2["W_qkv"][:, : 2 * cfg.d] = np.random.default_rng(5).standard_normal(W2["W_qkv"][:, : 2 * cfg.d].shape)
    a = O.decode_steps(cfg, W, O.init_state(cfg, W, 3), e, mem, 7)[0]
    b = O.decode_steps(cfg, W2, O.init_state(cfg, W2, 3), e, mem, 7)[0]
    assert np.array_equal(a.s, b.s)
    assert all(len(c) == 0 for c in a.cache)


def test_cross_attention_at_first_step_is_first_value():
    cfg, W, tok = setup(mem_groups=2)
    e, mem = O.encode(cfg, W, tok)
    tr = {}
    O.decode_step(cfg, W, O.init_state(cfg, W, 3), e[:, 0], mem, trace=tr)
    for l in range(cfg.n_layers):
        ref = mem[l, 1, :, :, 0, :].reshape(3, cfg.d)
        np.testing.assert_allclose(tr["x_out"][l], ref, rtol=1e-14, atol=1e-15)


def test_cross_attention_reads_through_current_position():
    cfg, W, tok = setup()
    e, mem = O.encode(cfg, W, tok)
    st = O.init_state(cfg, W, 3)
    st = O.decode_steps(cfg, W, st, e, mem, 3)[0]       # next step is t = 4
    base = O.decode_step(cfg, W, st, e[:, 3], mem).s
    after = mem.copy()
    after[..., 4:, :] += 1.0                            # positions 5.. are invisible
    assert np.array_equal(O.decode_step(cfg, W, st, e[:, 3], after).s, base)
    cur = mem.copy()
    cur[..., 3, :] += 1.0                               # position 4 = t is visible
    assert not np.allclose(O.decode_step(cfg, W, st, e[:, 3], cur).s, base)


def test_window_retains_w_minus_one():
    cfg, W, tok = setup(window=3, Tn=7)
    e, mem = O.encode(cfg, W, tok)
    st = O.init_state(cfg, W, 3)
    for t in range(1, 8):
        st = O.decode_step(cfg, W, st, e[:, t - 1], mem)
        assert all(len(c) == min(t, 2) for c in st.cache)


@pytest.mark.parametrize("cut", [0, 1, 3, 6, 7])
def test_split_invariance(cut):
    """Proposition 3.1: splitting the token stream anywhere leaves states and
    distributions unchanged (no reset at the boundary)."""
    cfg, W, tok = setup(window=3, Tn=7)
    e, mem = O.encode(cfg, W, tok)
    acts = ri.teacher_actions(tok, 0, 7)
    st0 = O.init_state(cfg, W, 3)
    full, out = O.decode_steps(cfg, W, st0, e, mem, 7, acts)
    a, oa = O.decode_steps(cfg, W, st0, e, mem, cut, acts[:, :cut])
    b, ob = O.decode_steps(cfg, W, a, e, mem, 7 - cut, acts[:, cut:])
    assert np.array_equal(full.s, b.s)
    assert all(np.array_equal(np.stack([x[0] for x in c1]), np.stack([x[0] for x in c2]))
               for c1, c2 in zip(full.cache, b.cache))
    lp = np.concatenate([oa.logp, ob.logp], axis=1)
    assert np.array_equal(lp, out.logp, equal_nan=True)


# ---------------------------------------------------------------------------
# head and scoring

def test_head_matches_library():
    cfg, W, tok = setup()
    s = np.random.default_rng(6).standard_normal((4, cfg.d))
    np.testing.assert_allclose(O.head_logits(cfg, W, s), TR.head_logits(cfg, W, s), rtol=1e-12)


@pytest.mark.parametrize("tau,k", [(1.0, 0), (0.7, 0), (0.7, 5), (1.3, 1), (1.0, 11), (0.5, 50)])
def test_score_matches_library(tau, k):
    rng = np.random.default_rng(7)
    V = 11
    lg = rng.standard_normal((64, V)) * 3
    act = rng.integers(0, V, 64)
    lp, lpf = O.score(lg, act, tau, k)
    ls = scipy.special.log_softmax(lg / tau, axis=-1)
    np.testing.assert_allclose(lpf, ls[np.arange(64), act], rtol=1e-13)
    if k == 0 or k >= V:
        np.testing.assert_allclose(lp, lpf, rtol=1e-13)
    else:
        vals, idx = torch.topk(torch.tensor(lg / tau), k, dim=-1)
        lse_k = torch.logsumexp(vals, dim=-1).numpy()
        in_k = (idx.numpy() == act[:, None]).any(-1)
        ref = np.where(in_k, lg[np.arange(64), act] / tau - lse_k, -np.inf)
        np.testing.assert_allclose(lp, ref, rtol=1e-13)
        # the renormalised top-k distribution sums to one
        for b in range(4):
            tot = sum(math.exp(O.score(lg[b:b + 1], [int(a)], tau, k)[0][0]) for a in idx[b].numpy())
            assert abs(tot - 1) < 1e-12


def test_topk_ties_prefer_lower_id():
    lg = np.array([[1.0, 3.0, 3.0, 3.0, 0.0]])
    m = O.topk_mask(lg, 2)
    assert m.tolist() == [[False, True, True, False, False]]
    lp, _ = O.score(lg, [3], 1.0, 2)
    assert lp[0] == -np.inf
    lp, _ = O.score(lg, [2], 1.0, 2)
    assert abs(lp[0] - math.log(0.5)) < 1e-14


def test_negative_action_is_unscored():
    lp, lpf = O.score(np.zeros((2, 3)), [-1, 1])
    assert np.isnan(lp[0]) and np.isnan(lpf[0]) and abs(lpf[1] + math.log(3)) < 1e-14


# ---------------------------------------------------------------------------
# bf16 emulation mode

def test_bf16_mode_rounds_at_contract_points():
    c = ri.RLTConfig(d=32, n_layers=2, n_heads=4, head_dim=8, d_ffn=48, window=3, mem_groups=1,
                     vocab=11, dtype="bf16")
    W = ri.make_weights(c, 101)
    wl = ri.Workload("t", c, B=2, T=5, tokens="uniform5", split=(2, 2), seed=101)
    tok = ri.make_tokens(wl)
    cfg = O.Cfg.of(c)
    e, mem = O.encode(cfg, W, tok)
    assert np.array_equal(O.bf16(e), e) and np.array_equal(O.bf16(mem), mem)
    st = O.decode_steps(cfg, W, O.init_state(cfg, W, 2), e, mem, 5)[0]
    for c_l in st.cache:
        for k, v in c_l:
            assert np.array_equal(O.bf16(k), k) and np.array_equal(O.bf16(v), v)
    cfg64 = O.Cfg.of(c)
    cfg64.bf16 = False
    st64 = O.decode_steps(cfg64, W, O.init_state(cfg64, W, 2), *O.encode(cfg64, W, tok), 5)[0]
    rel = np.max(np.abs(st.s - st64.s)) / np.max(np.abs(st64.s))
    assert 1e-5 < rel < 3e-2


# ---------------------------------------------------------------------------
# generation: the draw of the next token

def test_uniform24_is_uniform_and_independent():
    from scipy import stats
    u = np.array([O.uniform24(7, b, p) for b in range(40) for p in range(1000)])
    assert u.min() >= 0.0 and u.max() < 1.0
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))           # 24-bit grid
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    # neighbouring sequences, positions and seeds are uncorrelated
    a = u.reshape(40, 1000)
    assert abs(np.corrcoef(a[0], a[1])[0, 1]) < 0.1
    assert abs(np.corrcoef(a[:, :-1].ravel(), a[:, 1:].ravel())[0, 1]) < 0.05
    v = np.array([O.uniform24(8, b, p) for b in range(40) for p in range(1000)])
    assert abs(np.corrcoef(u, v)[0, 1]) < 0.05 and not np.array_equal(u, v)
    assert O.uniform24(7, 3, 5) == O.uniform24(7, 3, 5)


def test_uniform24_follows_the_published_splitmix64_outputs():
    """Draw (seed, b, pos=0) is output b+1 of SplitMix64 started at state seed,
    top 24 bits; the expected outputs are the generator's published reference
    values (tests/golden/splitmix64.txt, cited there)."""
    import pathlib
    rows = [ln.split() for ln in (pathlib.Path(__file__).parent / "golden" / "splitmix64.txt").read_text().splitlines()
            if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 2
    for row in rows:
        seed, outs = int(row[0]), [int(x) for x in row[1:]]
        assert len(outs) == 5
        for b, z in enumerate(outs):
            assert O.uniform24(seed, b, 0) == (z >> 40) / float(1 << 24)


def test_sample_token_inverts_the_cdf():
    # two tokens with probabilities 1/4 and 3/4
    lg = np.log(np.array([1.0, 3.0]))
    assert O.sample_token(lg, 0.0) == 0 and O.sample_token(lg, 0.2499) == 0
    assert O.sample_token(lg, 0.2501) == 1 and O.sample_token(lg, 0.9999) == 1
    # top-1 is the argmax with the lowest id on ties; top-k >= V is the full distribution
    rng = np.random.default_rng(3)
    x = rng.standard_normal(50)
    x[[7, 31]] = x.max() + 1.0
    assert all(O.sample_token(x, u, 0.7, 1) == 7 for u in (0.0, 0.5, 0.999))
    np.testing.assert_allclose(O.sampling_distribution(x, 0.7, 50), O.sampling_distribution(x, 0.7, 0))
    # top-k support: exactly k tokens, the k largest
    p = O.sampling_distribution(x, 0.7, 5)
    assert (p > 0).sum() == 5 and set(np.nonzero(p)[0]) == set(np.argsort(-x, kind="stable")[:5])
    # frequencies match the tempered softmax (chi-square)
    from scipy import stats
    x2 = rng.standard_normal(8)
    p2 = O.sampling_distribution(x2, 1.3, 0)
    q = scipy.special.softmax(x2 / 1.3)
    np.testing.assert_allclose(p2, q, rtol=1e-12)
    draws = np.array([O.sample_token(x2, O.uniform24(11, 0, i), 1.3) for i in range(20000)])
    counts = np.bincount(draws, minlength=8)
    assert stats.chisquare(counts, 20000 * q).pvalue > 1e-4


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin above fail

def _fails(fn, *a, **kw):
    try:
        fn(*a, **kw)
    except AssertionError:
        return True
    return False


def test_planted_mistakes_are_caught(monkeypatch):
    orig_rope, orig_keep, orig_range, orig_merge = O.rope, O.history_keep, O.memory_range, O.merge
    orig_attn = O.causal_attention
    orig_proj = O.memory_projection

    def rope_sign(x, pos, theta):
        hd = x.shape[-1]
        ang = O.rope_angles(pos, hd, theta)
        c, s = np.cos(ang), np.sin(ang)
        x1, x2 = x[..., : hd // 2], x[..., hd // 2:]
        return np.concatenate([x1 * c + x2 * s, x2 * c - x1 * s], axis=-1)

    cases = [
        ("rope", rope_sign, lambda: test_encoder_matches_library_composition(1, 0)),
        ("history_keep", lambda w: w, lambda: test_gate_discard_equals_parallel_pass(4)),
        ("memory_range", lambda t: max(t - 1, 1), lambda: test_gate_discard_equals_parallel_pass(4)),
        ("merge", lambda cfg, W, e, s, nx, trace=None: orig_merge(cfg, W, s, e, nx, trace),
         lambda: test_recurrence_equals_brute_force(3, 1)),
        ("causal_attention",
         lambda q, k, v, nx, round_p: (O.softmax_last((q @ np.swapaxes(k, -1, -2)) / math.sqrt(q.shape[-1])) @ v),
         lambda: test_encoder_matches_library_composition(1, 0)),
        # per-layer memory taken from the wrong layers
        ("memory_projection", lambda cfg, W, sources: orig_proj(cfg, W, sources[::-1]),
         lambda: test_encoder_matches_library_composition(2, 1)),
    ]
    for name, bad, pin in cases:
        with monkeypatch.context() as m:
            m.setattr(O, name, bad)
            assert _fails(pin), f"planted mistake in {name} not caught"
    # and the unpatched oracle passes the same pins
    assert O.rope is orig_rope and O.history_keep is orig_keep and O.memory_range is orig_range
    assert O.causal_attention is orig_attn
