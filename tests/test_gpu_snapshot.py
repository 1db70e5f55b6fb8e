"""Exact prefix snapshots on the GPU: save a state at position p with the
encoder output and memory of its prefix, restore it, decode on.

The pages ask that a fixed-weight snapshot be reusable across requests (the
state does not depend on how the computation is split) and that a weight
update invalidate it; the checks are bitwise against never having stopped.
"""
import numpy as np
import pytest
import torch

import rlt_inputs as ri

pytestmark = pytest.mark.gpu


def _setup(name, B, T, seed=None):
    import recurrent_looped_transformer_rlt_b300 as rlt
    from recurrent_looped_transformer_rlt_b300 import runner
    wl = ri.preset(name)
    W = ri.make_weights(wl.cfg, wl.seed if seed is None else seed, norm_jitter=0.1)
    tok = ri.make_tokens(wl, B=B, T=T)
    model = rlt.Model(wl.cfg, W)
    return rlt, runner, wl, model, tok


def _decode(runner, model, st, buf, acts, a, b):
    out = runner.decode(model, st, buf, b - a, torch.from_numpy(acts[:, a:b]).cuda().contiguous())
    return out.logp.cpu().numpy(), out.argmax.cpu().numpy()


@pytest.mark.parametrize("name,B,T,p", [("tiny", 4, 40, 17), ("small", 3, 60, 33), ("small", 2, 20, 0)])
def test_snapshot_restore_continues_bit_identically(name, B, T, p):
    rlt, runner, wl, model, tok = _setup(name, B, T)
    acts = ri.teacher_actions(tok, 0, T)
    buf = runner.alloc_buffers(model, B, T)
    runner.encode(model, torch.from_numpy(tok).cuda(), buf)
    # uninterrupted run, snapshot taken at p on the way
    st = runner.new_state(model, B)
    if p:
        _decode(runner, model, st, buf, acts, 0, p)
    n = rlt.rlt_snapshot_size(model.handle, B, p)
    snap = torch.empty(n, dtype=torch.uint8, device="cuda")
    rlt.rlt_snapshot_save(model.handle, st.c, buf.e, buf.mem, T, snap, n)
    lp_a, am_a = _decode(runner, model, st, buf, acts, p, T)
    s_a = st.s.cpu().numpy()
    ring_a = st.ring_k.float().cpu().numpy()
    # restore into a fresh state and into encoder buffers whose prefix rows are
    # garbage (the snapshot brings them back), then decode the rest
    buf2 = runner.alloc_buffers(model, B, T)
    buf2.e.copy_(buf.e)
    buf2.mem.copy_(buf.mem)
    if p:
        buf2.e[:, :p] = float("nan")
        buf2.mem[:, :, :, :, :p] = float("nan")
    st2 = rlt.State(model, B)
    st2.s.fill_(float("nan"))
    rlt.rlt_snapshot_restore(model.handle, snap, n, st2.c, buf2.e, buf2.mem, T)
    assert st2.c.pos == p and st2.c.version == model.version
    assert torch.equal(buf2.e, buf.e) and torch.equal(buf2.mem, buf.mem)
    lp_b, am_b = _decode(runner, model, st2, buf2, acts, p, T)
    assert np.array_equal(lp_a, lp_b, equal_nan=True)
    assert np.array_equal(am_a, am_b)
    assert np.array_equal(s_a, st2.s.cpu().numpy())
    assert np.array_equal(ring_a, st2.ring_k.float().cpu().numpy(), equal_nan=True)
    assert runner.status(buf2) == 0
    model.close()


def test_snapshot_reused_by_another_request_with_the_same_prefix():
    """Request A stops after its prompt; request B shares that prompt and goes
    on with other tokens.  B restored from A's snapshot equals B from scratch."""
    rlt, runner, wl, model, tokA = _setup("small", 3, 48)
    B, T, p = 3, 48, 20
    tokB = tokA.copy()
    rng = np.random.default_rng(9)
    tokB[:, p:] = rng.integers(0, 5, size=(B, T - p))
    assert not np.array_equal(tokA[:, p:], tokB[:, p:])
    actsA, actsB = ri.teacher_actions(tokA, 0, T), ri.teacher_actions(tokB, 0, T)
    # A: prompt only, snapshot
    bufA = runner.alloc_buffers(model, B, T)
    runner.encode(model, torch.from_numpy(tokA).cuda(), bufA)
    stA = runner.new_state(model, B)
    _decode(runner, model, stA, bufA, actsA, 0, p)
    n = rlt.rlt_snapshot_size(model.handle, B, p)
    snap = torch.empty(n, dtype=torch.uint8, device="cuda")
    rlt.rlt_snapshot_save(model.handle, stA.c, bufA.e, bufA.mem, T, snap, n)
    # B from scratch
    bufB = runner.alloc_buffers(model, B, T)
    runner.encode(model, torch.from_numpy(tokB).cuda(), bufB)
    stB = runner.new_state(model, B)
    lp_ref, _ = _decode(runner, model, stB, bufB, actsB, 0, T)
    # B from A's snapshot: encode B, restore the prefix, decode only the suffix
    bufC = runner.alloc_buffers(model, B, T)
    runner.encode(model, torch.from_numpy(tokB).cuda(), bufC)
    stC = rlt.State(model, B)
    rlt.rlt_snapshot_restore(model.handle, snap, n, stC.c, bufC.e, bufC.mem, T)
    lp_c, _ = _decode(runner, model, stC, bufC, actsB, p, T)
    assert np.array_equal(lp_ref[:, p:], lp_c, equal_nan=True)
    assert np.array_equal(stB.s.cpu().numpy(), stC.s.cpu().numpy())
    model.close()


def test_snapshot_rejected_after_weight_update_and_on_mismatch():
    rlt, runner, wl, model, tok = _setup("tiny", 2, 12)
    buf = runner.alloc_buffers(model, 2, 12)
    runner.encode(model, torch.from_numpy(tok).cuda(), buf)
    st = runner.new_state(model, 2)
    _decode(runner, model, st, buf, ri.teacher_actions(tok, 0, 12), 0, 5)
    n = rlt.rlt_snapshot_size(model.handle, 2, 5)
    snap = torch.empty(n, dtype=torch.uint8, device="cuda")
    rlt.rlt_snapshot_save(model.handle, st.c, buf.e, buf.mem, 12, snap, n)
    # another batch size, a buffer too small, a position beyond the encoded length
    st3 = rlt.State(model, 3)
    assert rlt.rlt_snapshot_restore(model.handle, snap, n, st3.c, buf.e, buf.mem, 12, check=False) == rlt.RLT_EINVAL
    st2 = rlt.State(model, 2)
    assert rlt.rlt_snapshot_restore(model.handle, snap, n - 16, st2.c, buf.e, buf.mem, 12,
                                    check=False) == rlt.RLT_EINVAL
    assert rlt.rlt_snapshot_restore(model.handle, snap, n, st2.c, buf.e, buf.mem, 4, check=False) == rlt.RLT_EINVAL
    # not a snapshot
    junk = torch.zeros(n, dtype=torch.uint8, device="cuda")
    assert rlt.rlt_snapshot_restore(model.handle, junk, n, st2.c, buf.e, buf.mem, 12, check=False) == rlt.RLT_EINVAL
    # a weight update invalidates the snapshot and the state it came from
    model.set_version(model.version + 1)
    assert rlt.rlt_snapshot_restore(model.handle, snap, n, st2.c, buf.e, buf.mem, 12, check=False) == rlt.RLT_ESTALE
    assert rlt.rlt_snapshot_save(model.handle, st.c, buf.e, buf.mem, 12, snap, n, check=False) == rlt.RLT_ESTALE
    model.close()


@pytest.mark.parametrize("p", [0, 9, 23])
def test_snapshot_continuation_matches_the_oracle(p):
    """A continuation restored from a snapshot, into fresh buffers, against
    the oracle's uninterrupted run (fp32 model: absolute 1e-4 on every
    scored log-probability, the logits of every step and the final state)."""
    from oracle import rlt_oracle as O
    rlt, runner, wl, model, tok = _setup("tiny", 3, 30)
    B, T = 3, 30
    acts = ri.teacher_actions(tok, 0, T)
    buf = runner.alloc_buffers(model, B, T)
    runner.encode(model, torch.from_numpy(tok).cuda(), buf)
    st = runner.new_state(model, B)
    if p:
        _decode(runner, model, st, buf, acts, 0, p)
    n = rlt.rlt_snapshot_size(model.handle, B, p)
    snap = torch.empty(n, dtype=torch.uint8, device="cuda")
    rlt.rlt_snapshot_save(model.handle, st.c, buf.e, buf.mem, T, snap, n)
    buf2 = runner.alloc_buffers(model, B, T)   # fresh: the prefix comes from the snapshot,
    runner.encode(model, torch.from_numpy(tok).cuda(), buf2)   # the suffix from this request's encode
    if p:
        buf2.e[:, :p] = float("nan")
        buf2.mem[:, :, :, :, :p] = float("nan")
    st2 = rlt.State(model, B)
    rlt.rlt_snapshot_restore(model.handle, snap, n, st2.c, buf2.e, buf2.mem, T)
    out = runner.decode(model, st2, buf2, T - p, torch.from_numpy(acts[:, p:]).cuda().contiguous(),
                        emit_steps=list(range(T - p)))
    _, _, ost, oout = O.run_sequence(O.Cfg.of(wl.cfg), ri.make_weights(wl.cfg, wl.seed, norm_jitter=0.1), tok, acts,
                                     emit=list(range(T)))
    assert np.abs(st2.s.cpu().numpy() - ost.s).max() <= 1e-4
    for i in range(T - p):
        assert np.abs(out.logits[i].cpu().numpy() - oout.logits[p + i]).max() <= 1e-4
    lp, olp = out.logp.cpu().numpy(), oout.logp[:, p:]
    m = ~np.isnan(olp)
    assert np.array_equal(np.isnan(lp), ~m) and np.abs(lp[m] - olp[m]).max() <= 1e-4
    model.close()


def test_snapshot_with_the_encoder_cache_resumes_generation_bitwise():
    """A snapshot that carries the encoder's key/value cache: generation
    restored from it (into buffers whose prefix rows are garbage) draws the
    same tokens with the same log-probabilities, and leaves the same state,
    encoder rows, memory rows and cache rows, as generation that never
    stopped."""
    import recurrent_looped_transformer_rlt_b300 as rlt
    from tests.test_gpu_generate import Gen
    g = Gen(B=3, T0=16, T_max=64)
    st = g.prefill()
    g.generate(st, 10, 77, 0.9, 7)
    p = st.c.pos
    n = rlt.rlt_snapshot_size(g.model.handle, g.B, p, with_enc_kv=True)
    assert n > rlt.rlt_snapshot_size(g.model.handle, g.B, p)
    snap = torch.empty(n, dtype=torch.uint8, device="cuda")
    rlt.rlt_snapshot_save(g.model.handle, st.c, g.e, g.mem, g.T_max, snap, n, enc_kv=g.kv)
    _, ta, la = g.generate(st, 20, 77, 0.9, 7)
    ref = dict(s=st.s.clone(), e=g.e.clone(), mem=g.mem.clone(), kv=g.kv.clone())
    # restore: garbage everywhere the snapshot must bring back, a fresh state
    g.e.fill_(float("nan"))
    g.mem.fill_(float("nan"))
    g.kv.fill_(float("nan"))
    st2 = rlt.State(g.model, g.B)
    st2.s.fill_(float("nan"))
    # the cache section is restored exactly when asked for
    assert rlt.rlt_snapshot_restore(g.model.handle, snap, n, st2.c, g.e, g.mem, g.T_max, check=False) == rlt.RLT_EINVAL
    rlt.rlt_snapshot_restore(g.model.handle, snap, n, st2.c, g.e, g.mem, g.T_max, enc_kv=g.kv)
    assert st2.c.pos == p
    _, tb, lb = g.generate(st2, 20, 77, 0.9, 7)
    assert np.array_equal(ta, tb) and np.array_equal(la, lb, equal_nan=True)
    T = p + 20
    assert torch.equal(st2.s, ref["s"])
    assert torch.equal(g.e[:, :T], ref["e"][:, :T]) and torch.equal(g.mem[..., :T, :], ref["mem"][..., :T, :])
    assert torch.equal(g.kv[..., :T, :], ref["kv"][..., :T, :])
    # a snapshot without the section cannot restore a cache
    n0 = rlt.rlt_snapshot_size(g.model.handle, g.B, p)
    snap0 = torch.empty(n0, dtype=torch.uint8, device="cuda")
    st3 = g.runner.new_state(g.model, g.B)
    g.runner.decode(g.model, st3, g.runner.Buffers(g.e, g.mem, g.ws, g.B, g.T_max), p)
    rlt.rlt_snapshot_save(g.model.handle, st3.c, g.e, g.mem, g.T_max, snap0, n0)
    assert rlt.rlt_snapshot_restore(g.model.handle, snap0, n0, st2.c, g.e, g.mem, g.T_max, check=False,
                                    enc_kv=g.kv) == rlt.RLT_EINVAL
    g.model.close()
