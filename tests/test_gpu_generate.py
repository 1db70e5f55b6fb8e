"""Autoregressive generation on the GPU against the oracle.

The pages' order: the state gives the next token's distribution, a token is
drawn from it, encoded incrementally and consumed by the decoder once.  The
GPU draws with a counter-based uniform per (seed, sequence, position); the
oracle then runs teacher-forced over the prompt and the generated tokens, and
the states, encoder rows, memory rows and behaviour log-probabilities must
agree within the bf16 tolerances.  Each draw must be the inverse-CDF draw of
the GPU's own distribution at its uniform number, and the oracle's draw at the
same number wherever that number is farther from every CDF boundary than the
row's measured logit difference can move it (at least 99% of all draws).
"""
import numpy as np
import pytest
import torch

import rlt_inputs as ri
from oracle import rlt_oracle as O
from tests.gpu_common import BF16_REL_LOGIT

pytestmark = pytest.mark.gpu


class Gen:
    def __init__(self, B=4, T0=24, T_max=64, name="small", path=None):
        import recurrent_looped_transformer_rlt_b300 as rlt
        from recurrent_looped_transformer_rlt_b300 import runner
        self.rlt, self.runner = rlt, runner
        self.wl = ri.preset(name)
        c = self.c = self.wl.cfg
        self.W = ri.make_weights(c, self.wl.seed, norm_jitter=0.1)
        self.B, self.T0, self.T_max = B, T0, T_max
        self.tok = ri.make_tokens(self.wl, B=B, T=T0)
        self.model = rlt.Model(c, self.W)
        if path:
            self.model.set_decode_path(path)
        dt = self.model.dtype
        self.e = torch.empty(B, T_max, c.d, dtype=dt, device="cuda")
        self.mem = torch.empty(c.mem_groups, 2, B, c.n_heads, T_max, c.head_dim, dtype=dt, device="cuda")
        self.kv = torch.empty(c.n_layers, 2, B, c.n_heads, T_max, c.head_dim, dtype=dt, device="cuda")
        self.ws = self.model.workspace(B, T_max)

    def prefill(self):
        rlt = self.rlt
        B, T0 = self.B, self.T0
        rlt.rlt_encode_kv(self.model.handle, torch.from_numpy(self.tok).cuda(), B, T0, self.T_max, self.e, self.mem,
                          self.kv, self.ws, self.ws.numel())
        st = self.runner.new_state(self.model, B)
        acts = torch.from_numpy(ri.teacher_actions(self.tok, 0, T0)).cuda()
        lp = torch.empty(B, T0, device="cuda")
        rlt.rlt_decode_steps(self.model.handle, st.c, self.e, self.mem, self.T_max, T0, acts, 1.0, 0, lp, None, None,
                             (), None, self.ws, self.ws.numel(), None)
        return st

    def generate(self, st, n, seed, tau, k, check=True):
        toks = torch.full((self.B, max(n, 1)), -7, dtype=torch.int32, device="cuda")
        lp = torch.full((self.B, max(n, 1)), float("nan"), device="cuda")
        rc = self.rlt.rlt_generate(self.model.handle, st.c, self.e, self.mem, self.kv, self.T_max, n, seed, tau, k,
                                   toks, lp, self.ws, self.ws.numel(), check=check)
        return rc, toks.cpu().numpy()[:, :n], lp.cpu().numpy()[:, :n]


def test_generation_matches_the_oracle_on_the_generated_sequence(path=None):
    g = Gen(path=path)
    B, T0, n, seed, tau, k = g.B, g.T0, 40, 123, 0.8, 5
    st = g.prefill()
    rc, gtok, glp = g.generate(st, n, seed, tau, k)
    assert rc == 0 and st.c.pos == T0 + n and g.rlt.rlt_status(g.ws) == 0
    V = g.c.vocab
    assert gtok.min() >= 0 and gtok.max() < V
    T = T0 + n
    tok_all = np.concatenate([g.tok, gtok], axis=1).astype(np.int32)
    c = O.Cfg.of(g.c)
    acts = ri.teacher_actions(tok_all, 0, T)
    e_o, mem_o, st_o, out = O.run_sequence(c, g.W, tok_all, acts, tau, k, emit=list(range(T)))
    # encoder rows (prompt token-parallel, generated positions incremental) and memory
    ge = g.e[:, :T].float().cpu().numpy()
    gm = g.mem[:, :, :, :, :T].float().cpu().numpy()
    assert np.abs(ge - e_o).max() <= BF16_REL_LOGIT * np.abs(e_o).max()
    assert np.abs(gm - mem_o).max() <= BF16_REL_LOGIT * np.abs(mem_o).max()
    # the state after the last generated token
    s = st.s.cpu().numpy()
    assert np.abs(s - st_o.s).max() <= BF16_REL_LOGIT * np.abs(st_o.s).max()
    # behaviour log-probabilities: generated token i is the action of step T0 - 1 + i
    olp = out.logp[:, T0 - 1:T0 - 1 + n]
    lmax = max(np.abs(out.logits[t]).max() for t in range(T0 - 1, T0 - 1 + n))
    assert np.all(np.isfinite(glp)) and np.all(np.isfinite(olp))
    assert np.abs(glp - olp).max() <= 2 * BF16_REL_LOGIT * lmax / tau + 1e-3
    # each draw against the distribution it came from.  The GPU's own logits of
    # those distributions: a teacher-forced decode from H_0 over the generated
    # sequence, reading the encoder and memory rows the generation wrote (the
    # same decoder steps, so the same logits)
    T1 = T - 1
    emit = list(range(T0 - 1, T1))
    st_g = g.runner.new_state(g.model, B)
    gl = torch.empty(len(emit), B, V, device="cuda")
    g.rlt.rlt_decode_steps(g.model.handle, st_g.c, g.e, g.mem, g.T_max, T1, None, 1.0, 0, None, None, None, emit, gl,
                           g.ws, g.ws.numel(), None)
    gl = gl.cpu().numpy().astype(np.float64)
    exact, robust, agree_robust, agree = 0, 0, 0, 0
    for b in range(B):
        for i in range(n):
            u = O.uniform24(seed, b, T0 + i)
            j = int(gtok[b, i])
            # (1) the GPU's draw is the inverse-CDF draw of its own distribution
            #     at u (up to the fp32 rounding of its running sums)
            pg = O.sampling_distribution(gl[i, b], tau, k)
            cg = np.cumsum(pg)
            assert pg[j] > 0 and cg[j] - pg[j] - 1e-5 <= u <= cg[j] + 1e-5, (b, i, j, u)
            exact += int(O.sample_token(gl[i, b], u, tau, k) == j)
            # (2) against the oracle's distribution: the tempered logits differ by
            #     at most delta on this row, so every probability by a factor
            #     within exp(+-2 delta) and every CDF value by at most
            #     exp(2 delta) - 1; a draw whose u is farther than that from
            #     every CDF boundary (and whose top-k set is not decided by a
            #     near-tie) must be the oracle's draw
            lo = out.logits[T0 - 1 + i][b]
            assert np.abs(gl[i, b] - lo).max() <= BF16_REL_LOGIT * np.abs(lo).max()
            delta = np.abs(gl[i, b] - lo).max() / tau
            slack = np.expm1(2 * delta)
            po = O.sampling_distribution(lo, tau, k)
            co = np.cumsum(po)
            srt = np.sort(lo / tau)[::-1]
            topk_tie = 0 < k < V and srt[k - 1] - srt[k] <= 2 * delta
            jo = O.sample_token(lo, u, tau, k)
            agree += int(jo == j)
            if not topk_tie and np.min(np.abs(co - u)) > slack:
                robust += 1
                agree_robust += int(jo == j)
    total = B * n
    print(f"generation: {exact}/{total} draws equal the GPU's own inverse-CDF draw, {agree}/{total} the oracle's; "
          f"{agree_robust}/{robust} of the draws away from a CDF boundary")
    assert exact >= total - 1                    # at most one fp32 tie at a boundary
    assert agree_robust == robust and robust >= 0.5 * total
    assert agree >= 0.99 * total
    g.model.close()


def test_generation_does_not_depend_on_the_call_split(path=None):
    ga, gb = Gen(B=3, T0=16, T_max=48, path=path), Gen(B=3, T0=16, T_max=48, path=path)
    sa, sb = ga.prefill(), gb.prefill()
    _, ta, la = ga.generate(sa, 24, 5, 1.0, 0)
    _, t1, l1 = gb.generate(sb, 9, 5, 1.0, 0)
    _, t2, l2 = gb.generate(sb, 15, 5, 1.0, 0)
    assert np.array_equal(ta, np.concatenate([t1, t2], 1))
    assert np.array_equal(la, np.concatenate([l1, l2], 1), equal_nan=True)
    assert torch.equal(sa.s, sb.s)
    T = 16 + 24
    assert torch.equal(ga.e[:, :T], gb.e[:, :T]) and torch.equal(ga.mem[:, :, :, :, :T], gb.mem[:, :, :, :, :T])
    assert torch.equal(ga.kv[:, :, :, :, :T], gb.kv[:, :, :, :, :T])
    ga.model.close()
    gb.model.close()


def test_generation_seeds_range_and_prefill_encoder():
    import recurrent_looped_transformer_rlt_b300 as rlt
    g = Gen(B=2, T0=8, T_max=24)
    # the prompt's e and memory from rlt_encode_kv equal rlt_encode's, bitwise
    st = g.prefill()
    buf = g.runner.alloc_buffers(g.model, 2, 8)
    g.runner.encode(g.model, torch.from_numpy(g.tok).cuda(), buf)
    assert torch.equal(g.e[:, :8], buf.e) and torch.equal(g.mem[:, :, :, :, :8], buf.mem)
    snap_e = g.e.clone()
    # same seed from the same state: same tokens; another seed: other tokens
    st2 = st.clone()
    _, t_a, _ = g.generate(st, 10, 1, 1.0, 0)
    g.e.copy_(snap_e)
    _, t_b, _ = g.generate(st2, 10, 1, 1.0, 0)
    assert np.array_equal(t_a, t_b)
    st3 = g.prefill()
    _, t_c, _ = g.generate(st3, 10, 2, 1.0, 0)
    assert not np.array_equal(t_a, t_c)
    # n = 0 is a no-op; past T_max is a range error
    pos = st3.c.pos
    assert g.generate(st3, 0, 2, 1.0, 0, check=False)[0] == 0 and st3.c.pos == pos
    assert g.generate(st3, 24 - pos + 1, 2, 1.0, 0, check=False)[0] == rlt.RLT_ERANGE
    g.model.close()
    # fp32 models: not supported by the generation entries
    f = Gen(B=2, T0=4, T_max=8, name="tiny")
    st = f.runner.new_state(f.model, 2)
    assert f.generate(st, 2, 1, 1.0, 0, check=False)[0] == rlt.RLT_EUNSUPPORTED
    f.model.close()
