"""The schedule of the decoder's backward (bptt_plan.h, host logic) against
the float64 autograd oracle, on the CPU.

The library's own bptt_plan.h - forward recording pass, reverse pass with
per-step recomputation, window-gradient ring, detach points, transposed
operands, workspace layout - is compiled with g++ over host-loop stand-ins
for its device primitives (tests/bptt_host_ops.cpp) and run on seeded
inputs; every gradient (decoder parameters, s_*, e, memory) and the loss must
equal the oracle's within fp32 storage rounding, for any size of the step
blocks over which weight and memory gradients are added.  The device kernels
themselves are checked against the oracle by the GPU tests.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import rlt_inputs as ri
from oracle import rlt_bptt as BP
from oracle import rlt_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))
PARAMS = ["W_g", "W_qkv", "W_O", "W_Qx", "W_Ox", "W_1", "W_3", "W_2", "W_o", "b_g", "s_star", "dec_attn_norm",
          "dec_xattn_norm", "dec_ffn_norm", "head_norm"]
GRADS = ["W_g", "b_g", "W_qkv", "W_O", "W_Qx", "W_Ox", "W_1", "W_3", "W_2", "W_o", "dec_attn_norm",
         "dec_xattn_norm", "dec_ffn_norm", "head_norm", "s_star"]
REL = 1e-4   # max-abs error relative to the gradient's largest entry (fp32 storage)


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not available")
    out = str(tmp_path_factory.mktemp("bptt") / "libbptt_host.so")
    subprocess.run([cxx, "-O2", "-std=c++17", "-shared", "-fPIC", "-o", out, os.path.join(HERE, "bptt_host_ops.cpp")],
                   check=True, capture_output=True)
    h = ctypes.CDLL(out)
    h.bptt_host.restype = ctypes.c_int
    h.bptt_host.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_float),
                            ctypes.POINTER(ctypes.c_void_p)]
    return h


def _setup(window=3, gate_mode=0, T=7, B=2, seed=41, G=1, L=2, scale=4.0):
    c = ri.RLTConfig(d=16, n_layers=L, n_heads=2, head_dim=8, d_ffn=24, window=window, mem_groups=G, vocab=9,
                     dtype="f32", gate_mode=gate_mode)
    W = ri.make_weights(c, seed, norm_jitter=0.1)
    for k in W:  # large enough weights that every path carries gradient
        if W[k].ndim >= 2:
            W[k] = W[k] * scale
    W["s_star"] = W["s_star"] * scale
    e, mem = ri.make_decoder_inputs(c, B, T, seed + 7, mem_scale=0.5)
    wl = ri.Workload("t", c, B=B, T=T, tokens="uniform5", split=(2, 2), seed=seed)
    tok = ((ri.make_tokens(wl) + np.arange(T)[None, :] * 2) % c.vocab).astype(np.int32)
    acts = ri.teacher_actions(tok, 0, T)
    acts[:, -1] = (tok[:, -1] + 1) % c.vocab
    return c, W, e, mem, acts


def _host(lib, c, W, e, mem, acts, tau=1.0, k=0, s_every=0, cache=False, memory=False, block=4, bf16=False):
    B, n = acts.shape
    sh = [B, n, e.shape[1], c.d, c.n_heads, c.head_dim, c.d_ffn, c.n_layers, c.window, c.vocab, c.mem_groups,
          1 if c.gate_mode == 0 else 0, k, s_every, int(cache), int(memory), block, int(bf16)]
    keep = []

    def buf(x, dt=np.float32):
        a = np.ascontiguousarray(np.asarray(x, dt))
        keep.append(a)
        return a.ctypes.data

    ptrs = [buf(W[p]) for p in PARAMS] + [buf(e), buf(mem), buf(acts, np.int32)]
    loss, logp = np.zeros(1, np.float32), np.zeros((B, n), np.float32)
    grads = {g: np.zeros(np.shape(W[g]), np.float32) for g in GRADS}
    d_e, d_mem = np.zeros(e.shape, np.float32), np.zeros(mem.shape, np.float32)
    ptrs += [loss.ctypes.data, logp.ctypes.data] + [grads[g].ctypes.data for g in GRADS]
    ptrs += [d_e.ctypes.data, d_mem.ctypes.data]
    rc = lib.bptt_host((ctypes.c_int * len(sh))(*sh), (ctypes.c_float * 3)(c.rms_eps, c.rope_theta, tau),
                       (ctypes.c_void_p * len(ptrs))(*ptrs))
    assert rc == 0
    return float(loss[0]), logp, grads, d_e, d_mem


def _compare(lib, setup_kw=None, tau=1.0, k=0, s_every=0, cache=False, memory=False, block=4):
    c, W, e, mem, acts = _setup(**(setup_kw or {}))
    cfg = O.Cfg.of(c)
    if k:  # actions inside the top-k set (outside it the loss is infinite)
        _, out = O.decode_steps(cfg, W, O.init_state(cfg, W, e.shape[0]), e, mem, acts.shape[1], acts, tau, k)
        acts = np.where(np.isfinite(out.logp), acts, -1).astype(np.int32)
    loss, logp, g, d_e, d_mem = _host(lib, c, W, e, mem, acts, tau, k, s_every, cache, memory, block)
    lref, gref = BP.gradients(cfg, W, e, mem, acts, temperature=tau, top_k=k, detach_s_every=s_every,
                              detach_cache=cache, detach_memory=memory)
    assert abs(loss - lref) <= 1e-5 * max(1.0, abs(lref))
    for name, x in list(g.items()) + [("e", d_e), ("mem", d_mem)]:
        r = gref[name]
        scale = np.abs(r).max()
        assert np.abs(x - r).max() <= REL * scale + 1e-7, name
    return g, d_e, d_mem, gref


@pytest.mark.parametrize("setup_kw", [
    {},                                   # window 3 over 7 steps: the ring wraps twice
    {"window": 1},                        # no history: keys/values get only their own step's gradient
    {"window": 5, "T": 9},
    {"gate_mode": 1},                     # z = 0: no gradient reaches s_{t-1}, W_g, b_g or s_*
    {"G": 2},                             # one memory group per layer
    {"L": 3, "B": 3, "window": 4, "T": 8},
])
def test_full_bptt_schedule_matches_the_oracle(lib, setup_kw):
    g, _, _, _ = _compare(lib, setup_kw)
    if setup_kw.get("gate_mode") == 1:
        assert not np.any(g["W_g"]) and not np.any(g["b_g"]) and not np.any(g["s_star"])


@pytest.mark.parametrize("kw", [
    {"s_every": 2},
    {"cache": True},
    {"memory": True},
    {"s_every": 3, "cache": True, "memory": True},
])
def test_truncated_bptt_schedule_matches_the_oracle(lib, kw):
    _, _, d_mem, _ = _compare(lib, {"T": 9}, **kw)
    if kw.get("memory"):
        assert not np.any(d_mem)


@pytest.mark.parametrize("block", [1, 3, 7, 16])
def test_step_blocks(lib, block):
    """Weight and memory gradients added once per block of steps: any block
    size (a partial last block, a single block longer than the sequence) gives
    the oracle's gradients."""
    _compare(lib, {"T": 7, "G": 2}, block=block)


def test_tempered_top_k_head(lib):
    _compare(lib, {"T": 8}, tau=0.7, k=4)


def test_detaching_only_s_leaves_cache_paths(lib):
    """With s detached every step, gradient still crosses steps through the
    window keys and values (the pages' point about the cross terms): the
    encoder output of an earlier position in the window receives gradient
    from a later step's loss unless the cache is detached too."""
    c, W, e, mem, acts = _setup(window=3, T=5)
    step4 = np.full_like(acts, -1)
    step4[:, 3] = acts[:, 3]   # score only step 4's action (position 3)
    _, _, _, de_s, _ = _host(lib, c, W, e, mem, step4, s_every=1)
    _, _, _, de_sc, _ = _host(lib, c, W, e, mem, step4, s_every=1, cache=True)
    assert np.abs(de_s[:, 2]).max() > 0        # position 2 is in step 4's window
    assert np.abs(de_sc[:, 2]).max() == 0      # ... and reaches it only through the cache
    assert np.abs(de_sc[:, 3]).max() > 0       # the step's own input always has gradient


def test_bf16_storage_stays_within_bf16_error(lib):
    """With every storage-type write rounded to bf16 (what the bf16 models'
    kernels store: normalised activations, attention outputs, keys and
    values, and every gradient that enters a GEMM), the gradients stay within
    a few bf16 roundings of the float64 oracle on the same bf16 weights and
    inputs: relative Frobenius error ~3e-3 per gradient at this size."""
    c = ri.RLTConfig(d=256, n_layers=2, n_heads=8, head_dim=32, d_ffn=512, window=4, mem_groups=2, vocab=64,
                     dtype="bf16")
    W = ri.make_weights(c, 41, norm_jitter=0.1)
    B, T = 2, 10
    e, mem = ri.make_decoder_inputs(c, B, T, 48, mem_scale=0.5)
    wl = ri.Workload("t", c, B=B, T=T, tokens="uniform5", split=(2, 2), seed=41)
    tok = ((ri.make_tokens(wl) + np.arange(T)[None, :] * 2) % c.vocab).astype(np.int32)
    acts = ri.teacher_actions(tok, 0, T)
    loss, _, g, d_e, d_mem = _host(lib, c, W, e, mem, acts, block=16, bf16=True)
    cfg = O.Cfg.of(ri.RLTConfig(**{**c.__dict__, "dtype": "f32"}))  # float64 arithmetic on the same values
    lref, gref = BP.gradients(cfg, W, e, mem, acts)
    assert abs(loss - lref) <= 1e-3 * abs(lref)
    for name, x in list(g.items()) + [("e", d_e), ("mem", d_mem)]:
        r = gref[name]
        rel = np.linalg.norm((x - r).ravel()) / np.linalg.norm(r.ravel())
        assert 1e-5 < rel < 1e-2, (name, rel)   # rounding is visible, and small
