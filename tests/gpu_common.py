"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the CPU oracle on the same seeded inputs, and compare."""
import numpy as np

import rlt_inputs as ri
from oracle import rlt_oracle as O

# tolerances (fp32 models: absolute; bf16 models: relative to the row's max |logit|)
F32_ABS = 1e-4
BF16_REL_LOGIT = 2e-2
BF16_ARGMAX_AGREE = 0.999


def gpu_run(wl, W, tok, acts, n_split=None, emit=(), temperature=1.0, top_k=0, gate_mode=None, window=None,
            return_model=False):
    """Encode tok and decode all positions on the GPU; returns numpy outputs."""
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    from recurrent_looped_transformer_rlt_b300 import runner
    cfg = wl.cfg
    if gate_mode is not None or window is not None:
        cfg = ri.RLTConfig(**{**cfg.__dict__, **({"gate_mode": gate_mode} if gate_mode is not None else {}),
                              **({"window": window} if window is not None else {})})
    B, T = tok.shape
    model = rlt.Model(cfg, W)
    buf = runner.alloc_buffers(model, B, T)
    runner.encode(model, torch.from_numpy(tok).cuda(), buf)
    st = runner.new_state(model, B)
    cuts = [0] + list(n_split or []) + [T]
    logp, logp_full, amax, logits = [], [], [], {}
    acts_t = torch.from_numpy(acts).cuda()
    for a, b in zip(cuts[:-1], cuts[1:]):
        n = b - a
        if n == 0:
            continue
        em = [i - a for i in emit if a <= i < b]
        out = runner.decode(model, st, buf, n, acts_t[:, a:b].contiguous(), temperature, top_k, emit_steps=em)
        logp.append(out.logp.cpu().numpy())
        logp_full.append(out.logp_full.cpu().numpy())
        amax.append(out.argmax.cpu().numpy())
        for j, i in enumerate(em):
            logits[a + i] = out.logits[j].cpu().numpy()
    torch.cuda.synchronize()
    status = runner.status(buf)
    res = dict(e=buf.e.float().cpu().numpy(), mem=buf.mem.float().cpu().numpy(), s=st.s.cpu().numpy(),
               ring_k=st.ring_k.float().cpu().numpy(), ring_v=st.ring_v.float().cpu().numpy(),
               logp=np.concatenate(logp, 1), logp_full=np.concatenate(logp_full, 1),
               argmax=np.concatenate(amax, 1), logits=logits, status=status, pos=st.pos)
    if return_model:
        return res, (model, buf, st)
    model.close()
    return res


def oracle_run(wl, W, tok, acts, emit=(), temperature=1.0, top_k=0, gate_mode=None, window=None):
    c = O.Cfg.of(wl.cfg)
    if gate_mode is not None:
        c.gate_mode = gate_mode
    if window is not None:
        c.window = window
    e, mem, st, out = O.run_sequence(c, W, tok, acts, temperature, top_k, emit=emit)
    return dict(e=e, mem=mem, s=st.s, logp=out.logp, logp_full=out.logp_full, argmax=out.argmax,
                logits=out.logits, cache=st.cache)


def check_argmax(g_argmax, g_logits, o_logits, tol_rel=BF16_REL_LOGIT, agree=BF16_ARGMAX_AGREE):
    """Argmax is an integer decided by floating point, so each side decides in its own
    precision: (1) the GPU's argmax equals the argmax of its own fp32 logits (lowest id
    on ties); (2) on rows whose oracle top-2 gap exceeds twice the row's measured logit
    difference, the two argmaxes agree on >= `agree` of the rows; (3) on the remaining
    near-tie rows the GPU's pick is a maximiser of the oracle logits within the logit
    tolerance.  Arrays: g_argmax [R], g_logits/o_logits [R, V].  Returns raw agreement."""
    own = np.argmax(g_logits, axis=-1)
    assert np.array_equal(g_argmax, own), "argmax differs from the GPU's own logits"
    o_arg = np.argmax(o_logits, axis=-1)
    err = np.max(np.abs(g_logits - o_logits), axis=-1)
    top2 = np.sort(o_logits, axis=-1)[:, -2:]
    gap = top2[:, 1] - top2[:, 0]
    decided = gap > 2 * err
    if decided.any():
        a = np.mean(g_argmax[decided] == o_arg[decided])
        assert a >= agree, (a, int(decided.sum()))
    deficit = o_logits.max(-1) - o_logits[np.arange(len(g_argmax)), g_argmax]
    tol = tol_rel * np.max(np.abs(o_logits), axis=-1)
    assert np.all(deficit <= tol), deficit.max()
    return float(np.mean(g_argmax == o_arg))


def rel_logit_err(g, o):
    """Per row ||dl||_inf / ||l_ref||_inf."""
    return np.max(np.abs(g - o), axis=-1) / np.max(np.abs(o), axis=-1)


def oracle_ring(cfg, cache, pos):
    """Oracle cache -> ring layout [L][B][H][W][hd] (slots of retained positions)."""
    L, W = cfg.n_layers, cfg.window
    out = {}
    for l in range(L):
        ent = cache[l]
        n = len(ent)
        for j, (k, v) in enumerate(ent):
            p = pos - n + j
            out[(l, p % W)] = (k, v)
    return out
