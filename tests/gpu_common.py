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
            return_model=False, decode_path=None, cluster_size=0):
    """Encode tok and decode all positions on the GPU; returns numpy outputs.
    decode_path: None (the library's default), 'graph' or 'fused'."""
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    from recurrent_looped_transformer_rlt_b300 import runner
    cfg = wl.cfg
    if gate_mode is not None or window is not None:
        cfg = ri.RLTConfig(**{**cfg.__dict__, **({"gate_mode": gate_mode} if gate_mode is not None else {}),
                              **({"window": window} if window is not None else {})})
    B, T = tok.shape
    model = rlt.Model(cfg, W)
    if decode_path:
        model.set_decode_path(decode_path, cluster_size)
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


def gpu_transition_snapshots(wl, W, tok, acts, t0s, rows, temperature=1.0, top_k=0):
    """Run the CUDA path over all of tok; before each step t0 + 1 (t0 in t0s) keep
    the state of the sequences `rows` (s, the window's ring entries, position) and
    the outputs of that step.  Returns (e, mem) of those rows and a list of dicts."""
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    from recurrent_looped_transformer_rlt_b300 import runner
    B, T = tok.shape
    model = rlt.Model(wl.cfg, W)
    buf = runner.alloc_buffers(model, B, T)
    runner.encode(model, torch.from_numpy(tok).cuda(), buf)
    st = runner.new_state(model, B)
    acts_t = torch.from_numpy(acts).cuda()
    snaps = []
    for t0 in sorted(t0s):
        if t0 > st.pos:
            runner.decode(model, st, buf, t0 - st.pos, acts_t[:, st.pos:t0].contiguous(), temperature, top_k)
        torch.cuda.synchronize()
        snap = dict(pos=st.pos, s=st.s[rows].cpu().numpy().astype(np.float64),
                    ring_k=st.ring_k[:, rows].float().cpu().numpy(), ring_v=st.ring_v[:, rows].float().cpu().numpy())
        out = runner.decode(model, st, buf, 1, acts_t[:, t0:t0 + 1].contiguous(), temperature, top_k, emit_steps=[0])
        torch.cuda.synchronize()
        snap.update(logits=out.logits[0][rows].cpu().numpy(), logp=out.logp[rows, 0].cpu().numpy(),
                    logp_full=out.logp_full[rows, 0].cpu().numpy(), argmax=out.argmax[rows, 0].cpu().numpy(),
                    s_next=st.s[rows].cpu().numpy())
        snaps.append(snap)
    assert runner.status(buf) == 0
    e = buf.e[rows].float().cpu().numpy().astype(np.float64)
    mem = buf.mem[:, :, rows].float().cpu().numpy().astype(np.float64)
    model.close()
    return e, mem, snaps


def oracle_transition(wl, W, e, mem, snap, acts_col, temperature=1.0, top_k=0):
    """One oracle step from the CUDA path's state: s, the ring entries of positions
    pos - W + 1 .. pos - 1 (oldest first), e and memory of the same run."""
    c = O.Cfg.of(wl.cfg)
    pos, Wn = snap["pos"], c.window
    cache = []
    for l in range(c.n_layers):
        ent = []
        for p in range(max(0, pos - (Wn - 1)), pos):
            ent.append((snap["ring_k"][l, :, :, p % Wn].astype(np.float64),
                        snap["ring_v"][l, :, :, p % Wn].astype(np.float64)))
        cache.append(ent)
    st = O.State(snap["s"].copy(), cache, pos)
    st2, out = O.decode_steps(c, W, st, e, mem, 1, acts_col, temperature, top_k, emit=[0])
    return dict(logits=out.logits[0], logp=out.logp[:, 0], logp_full=out.logp_full[:, 0], argmax=out.argmax[:, 0],
                s_next=st2.s)
