"""Pins of the oracle's bf16 emulation mode (CPU only).

The bf16 configurations store in bfloat16 exactly at the points of the
numerics contract (every matrix-product input, e, the memory, the window
keys/values after RoPE, the encoder's q/k/v after RoPE and its unnormalised
attention weights before the product with the values); everything else stays
in float64 in the oracle.  These tests tie the oracle's rounding points to a
composition of torch library routines that rounds with torch's own bfloat16
conversion at the same points (tests/_torch_ref.py: encoder_bf16,
decoder_bf16), for the encoder, the recurrent decoder steps and the head; and
they drop each rounding the oracle performs, one at a time, and check that
the pin then fails, so that no rounding point is left unpinned.
"""
import math
import sys

import numpy as np
import pytest
import torch

import rlt_inputs as ri
from oracle import rlt_oracle as O
from tests import _torch_ref as TR

TOL = 1e-12   # relative to the largest magnitude of the compared tensor


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def test_single_rounding_helper_matches_the_definition():
    """TR.bf16_rne rounds float64 to the nearest bfloat16 (ties to even) in
    one step: checked against exact ties, values just off a tie that the
    float32 step would carry onto it, and random values against the oracle's
    bit-level rounding."""
    one = 1.0
    cases = {one + 2.0 ** -8: 1.0,                        # tie, even below
             one + 3 * 2.0 ** -8: one + 2.0 ** -6,        # tie, even above
             one + 2.0 ** -8 + 2.0 ** -30: one + 2.0 ** -7,   # just above a tie: rounds up
             one + 2.0 ** -8 - 2.0 ** -30: 1.0,           # just below a tie: rounds down
             -(one + 2.0 ** -8 + 2.0 ** -30): -(one + 2.0 ** -7)}
    for x, want in cases.items():
        assert TR.bf16_rne(torch.tensor([x], dtype=torch.float64)).item() == want, x
    rng = np.random.default_rng(5)
    x = rng.standard_normal(200000) * 10.0 ** rng.integers(-5, 5, 200000)
    # plus values a float32 rounding puts on a bfloat16 tie
    base = rng.standard_normal(2000).astype(np.float32)
    ties = (base.view(np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    t64 = ties.view(np.float32).astype(np.float64)
    x = np.concatenate([x, t64 * (1 + 2.0 ** -40), t64 * (1 - 2.0 ** -40), t64])
    assert np.array_equal(TR.bf16_rne(torch.from_numpy(x)).numpy(), O.bf16(x))


def _setup(G=1, src=0, gate_mode=0, window=3, seed=210, B=3, Tn=6):
    c = ri.RLTConfig(d=32, n_layers=2, n_heads=4, head_dim=8, d_ffn=48, window=window, mem_groups=G,
                     vocab=13, dtype="bf16", gate_mode=gate_mode, mem_source=src)
    W = ri.make_weights(c, seed, norm_jitter=0.1, gate_bias=0.1)
    # power-of-two scale keeps the matrices bfloat16 values and makes every term matter
    for k in W:
        if W[k].ndim >= 2:
            W[k] = W[k] * np.float32(16.0)
    W["s_star"] = W["s_star"] * np.float32(16.0)
    wl = ri.Workload("t", c, B=B, T=Tn, tokens="uniform5", split=(2, 2), seed=seed)
    tok = ((ri.make_tokens(wl) + np.arange(Tn)[None, :] * 3) % c.vocab).astype(np.int32)
    return O.Cfg.of(c), W, tok


def _pin(G=1, src=0, gate_mode=0, window=3):
    """The oracle's bf16 mode against the torch composition: e, memory, the
    state after every step, every step's logits and the window caches."""
    cfg, W, tok = _setup(G, src, gate_mode, window)
    Tn = tok.shape[1]
    e, mem = O.encode(cfg, W, tok)
    te, tm = TR.encoder_bf16(cfg, W, tok)
    assert _rel(e, te) <= TOL
    assert _rel(mem, tm) <= TOL
    st, out = O.decode_steps(cfg, W, O.init_state(cfg, W, tok.shape[0]), e, mem, Tn, emit=range(Tn))
    ts, tlog, tcache = TR.decoder_bf16(cfg, W, e, mem, Tn)
    assert _rel(st.s, ts) <= TOL
    for i in range(Tn):
        assert _rel(out.logits[i], tlog[i]) <= TOL
    for l in range(cfg.n_layers):
        assert len(st.cache[l]) == len(tcache[l])
        for (k, v), (tk, tv) in zip(st.cache[l], tcache[l]):
            assert _rel(k, tk) <= TOL and _rel(v, tv) <= TOL


@pytest.mark.parametrize("G,src,gate_mode,window", [(1, 0, 0, 3), (2, 1, 0, 2), (1, 0, 1, 1), (2, 0, 0, 8)])
def test_bf16_mode_equals_the_library_composition(G, src, gate_mode, window):
    _pin(G, src, gate_mode, window)


class _DropOne(O.Numerics):
    """The oracle's rounding policy with the rounding at one call site (the
    calling function and line) left out; records every site it sees."""
    drop = None
    seen = set()

    def r(self, x):
        f = sys._getframe(1)
        site = (f.f_code.co_name, f.f_lineno)
        _DropOne.seen.add(site)
        if self.bf16 and site == _DropOne.drop:
            return np.asarray(x, dtype=np.float64)
        return super().r(x)


def _fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_every_rounding_point_is_pinned(monkeypatch):
    """Dropping any single rounding of the oracle's bf16 mode (the SwiGLU
    product, an attention output before its projection, [e; s] into the gate,
    the encoder's attention weights, a memory projection, ...) makes the pin
    above fail."""
    cases = [(1, 0, 0, 3), (2, 1, 0, 2)]
    monkeypatch.setattr(O, "Numerics", _DropOne)
    _DropOne.seen, _DropOne.drop = set(), None
    for case in cases:
        _pin(*case)
    sites = sorted(_DropOne.seen)
    funcs = {fn for fn, _ in sites}
    # encoder (normed inputs, q, k, v, weights, outputs, SwiGLU product, e, per-layer
    # memory sources), memory projection, merge, decoder step, head
    assert {"encode", "causal_attention", "memory_projection", "merge", "decode_step", "head_logits"} <= funcs
    assert len(sites) >= 20, sites
    missed = []
    for site in sites:
        _DropOne.drop = site
        if not any(_fails(lambda c=case: _pin(*c)) for case in cases):
            missed.append(site)
    _DropOne.drop = None
    assert not missed, f"roundings whose removal no pin detects: {missed}"


def test_the_swiglu_product_rounding_is_pinned(monkeypatch):
    """The planted mistake named on its own: the decoder's SwiGLU product
    left in float64."""
    import inspect
    src, first = inspect.getsourcelines(O.decode_step)
    line = first + next(i for i, s in enumerate(src) if "silu(" in s and "nx.r(" in s)
    monkeypatch.setattr(O, "Numerics", _DropOne)
    _DropOne.drop = ("decode_step", line)
    try:
        assert _fails(lambda: _pin(1, 0, 0, 3))
    finally:
        _DropOne.drop = None
