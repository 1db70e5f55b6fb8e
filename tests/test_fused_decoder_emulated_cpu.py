"""The persistent cluster decoder (dec_fused_kernel: every step of a decode
call in one launch, one thread-block cluster per group of sequences) run
under the host emulation of the CUDA execution model (tests/simt_emu),
against the oracle's decode_steps on bf16 models.

The kernel is compiled with g++ against stand-in CUDA headers: one host
thread per CUDA thread, the blocks of a cluster concurrently with their own
shared memory (filled with NaN bytes before the launch), cluster barriers,
distributed shared memory as addresses into the other blocks' buffers, and
the warp-level bf16 MMA computed from its documented fragment layout.  The
launch uses the library's plan (fused_plan.h): cluster size, sequences per
cluster, row split of every projection, shared-memory layout.  This checks
the kernel's work split, exchanges and index arithmetic without a GPU; the
GPU tests check the same kernel on the device.
"""
import ctypes
import os
import re
import shutil
import subprocess
import sys

import numpy as np
import pytest

import rlt_inputs as ri
from oracle import rlt_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "recurrent_looped_transformer_rlt_b300", "csrc")
EMU = os.path.join(ROOT, "tests", "simt_emu")
MATS = ["W_g", "W_qkv", "W_O", "W_Qx", "W_Ox", "W_1", "W_3", "W_2", "W_o"]
VECS = ["b_g", "dec_attn_norm", "dec_xattn_norm", "dec_ffn_norm", "head_norm"]


@pytest.fixture(scope="module")
def fz(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not available")
    d = str(tmp_path_factory.mktemp("fused_emu"))
    src = open(os.path.join(CSRC, "dec_fused.cuh")).read()
    src, n = re.subn(r"extern __shared__ __align__\(128\) unsigned char (\w+)\[\];",
                     r"unsigned char* \1 = emu_dyn_smem<unsigned char>();", src)
    assert n == 1
    open(os.path.join(d, "dec_fused_emu.cuh"), "w").write(src)
    lib = os.path.join(d, "libfused.so")
    # the emulator's directory first: its fused_ptx.cuh stands in for the library's
    r = subprocess.run([cxx, "-std=c++20", "-O1", "-shared", "-fPIC", "-pthread", "-I", d, "-I", EMU, "-I", CSRC,
                        "-o", lib, os.path.join(EMU, "fused_harness.cpp")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    h = ctypes.CDLL(lib)
    h.fused_emu.restype = ctypes.c_int
    return h


def _call(h, c, W, e, mem, s, rk, rv, acts, p0, n, CS, Bc, tau=1.0, k=0, emit=()):
    B, T = e.shape[:2]
    sh = [B, T, c.d, c.n_heads, c.head_dim, c.d_ffn, c.n_layers, c.window, c.vocab, c.mem_groups,
          1 if c.gate_mode == 0 else 0, p0, n, k, CS, Bc, 0, 0, 0]
    keep = []

    def f32(x):
        a = np.ascontiguousarray(np.asarray(x, np.float32))
        keep.append(a)
        return a.ctypes.data

    s, rk, rv = np.array(s, np.float32), rk.copy(), rv.copy()
    a = np.ascontiguousarray(acts[:, p0:p0 + n], np.int32)
    emap = np.full(n, -1, np.int32)
    for j, i in enumerate(emit):
        emap[i] = j
    lg = np.zeros((max(len(emit), 1), B, c.vocab), np.float32)
    lp, lf = np.zeros((B, n), np.float32), np.zeros((B, n), np.float32)
    am, status = np.zeros((B, n), np.int32), np.zeros(1, np.int32)
    ptr = [f32(W[p]) for p in MATS] + [f32(W[p]) for p in VECS] + [f32(e), f32(mem)]
    ptr += [s.ctypes.data, rk.ctypes.data, rv.ctypes.data, a.ctypes.data, emap.ctypes.data, lg.ctypes.data,
            lp.ctypes.data, lf.ctypes.data, am.ctypes.data, status.ctypes.data]
    rc = h.fused_emu((ctypes.c_int * len(sh))(*sh), (ctypes.c_float * 3)(c.rms_eps, c.rope_theta, tau),
                     (ctypes.c_void_p * len(ptr))(*ptr))
    assert rc == 0, "plan rejected the shape"
    assert status[0] == 0
    return dict(s=s, rk=rk, rv=rv, logp=lp, logp_full=lf, argmax=am, logits=lg[:len(emit)])


def _case(h, CS, Bc, B=5, T=8, d=64, H=2, hd=32, f=96, L=2, window=3, G=2, V=40, gate_mode=0, tau=1.0, k=0,
          split=(), emit=(), seed=5):
    c = ri.RLTConfig(d=d, n_layers=L, n_heads=H, head_dim=hd, d_ffn=f, window=window, mem_groups=G, vocab=V,
                     dtype="bf16", gate_mode=gate_mode)
    W = ri.make_weights(c, seed, norm_jitter=0.1)
    e, mem = ri.make_decoder_inputs(c, B, T, seed + 4, mem_scale=0.5)
    acts = (np.arange(B * T).reshape(B, T) * 7 % V).astype(np.int32)
    acts[0, 1] = -1                                   # an unscored step
    cfg = O.Cfg.of(c)
    st0 = O.init_state(cfg, W, B)
    rk = np.full((L, B, H, window, hd), np.nan, np.float32)
    s, rv = st0.s, rk.copy()
    cuts = [0] + list(split) + [T]
    outs = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o = _call(h, c, W, e, mem, s, rk, rv, acts, a, b - a, CS, Bc, tau, k, [i - a for i in emit if a <= i < b])
        s, rk, rv = o["s"], o["rk"], o["rv"]
        outs.append(o)
    got = dict(s=s, rk=rk, rv=rv, **{key: np.concatenate([o[key] for o in outs], 1)
                                       for key in ("logp", "logp_full", "argmax")})
    got["logits"] = np.concatenate([o["logits"] for o in outs], 0) if emit else None
    ref_st, ref = O.decode_steps(cfg, W, st0, e, mem, T, acts, tau, k, emit=emit)
    return c, got, ref_st, ref


def _check(c, got, ref_st, ref, T):
    # bf16 model: the same values rounded at the same points; a rounding that
    # lands on the other side of a bf16 boundary moves a stored value by one
    # bf16 step (2^-8 relative), which is all the difference there is
    assert np.abs(got["s"] - ref_st.s).max() <= 2e-3 * np.abs(ref_st.s).max()
    fin = np.isfinite(ref.logp)
    assert np.array_equal(np.isfinite(got["logp"]), fin)
    assert np.isnan(got["logp"][0, 1]) and np.isnan(got["logp_full"][0, 1])
    assert np.nanmax(np.abs(got["logp"][fin] - ref.logp[fin])) <= 2e-3 * max(1.0, np.abs(ref.logp[fin]).max())
    assert np.nanmax(np.abs(got["logp_full"] - ref.logp_full)) <= 2e-3 * max(1.0, np.nanmax(np.abs(ref.logp_full)))
    assert (got["argmax"] == ref.argmax).mean() >= 0.99
    for l in range(c.n_layers):  # the ring holds the window's keys (after RoPE) and values
        ents = ref_st.cache[l]
        for j, (kk, vv) in enumerate(ents):
            p = T - len(ents) + j
            assert np.abs(got["rk"][l, :, :, p % c.window] - kk).max() <= 1e-2 * max(1.0, np.abs(kk).max())
            assert np.abs(got["rv"][l, :, :, p % c.window] - vv).max() <= 1e-2 * max(1.0, np.abs(vv).max())


@pytest.mark.parametrize("kw", [
    dict(CS=2, Bc=3),                                 # two CTAs per head, ragged last cluster
    dict(CS=4, Bc=8, B=11),                           # four CTAs per head: d rows split 1:1
    dict(CS=2, Bc=16, B=17),                          # two 8-column MMA tiles
    dict(CS=1, Bc=5),                                 # one CTA: no exchange
    dict(CS=2, Bc=4, H=4, hd=16),                     # two heads per CTA
    dict(CS=4, Bc=4, H=4, hd=16, gate_mode=1),        # the gate discards s: h = e
    dict(CS=2, Bc=5, k=7, tau=0.7),                   # tempered top-k scoring
    dict(CS=2, Bc=3, window=1),                       # the window holds the current token only
    dict(CS=2, Bc=3, G=1, window=5, T=11),            # one memory group; the ring wraps
    dict(CS=4, Bc=2, d=128, hd=64, f=200, V=70),      # 64-wide heads, ragged f and V tiles
    dict(CS=2, Bc=5, split=(3, 4), emit=(0, 5)),      # three calls, logits of two steps
    dict(CS=2, Bc=2, B=2, L=1, G=1, window=70, T=75),     # window over several row passes; the ring wraps
])
def test_fused_decoder_matches_the_oracle(fz, kw):
    c, got, ref_st, ref = _case(fz, **kw)
    _check(c, got, ref_st, ref, kw.get("T", 8))
    for j, i in enumerate(kw.get("emit", ())):
        assert np.abs(got["logits"][j] - ref.logits[i]).max() <= 2e-3 * max(1.0, np.abs(ref.logits[i]).max())


def test_fused_decoder_call_split_is_bitwise(fz):
    """Proposition 3.1 for this path: splitting the n steps across calls gives
    bit-identical states, caches and scores."""
    _, a, _, _ = _case(fz, CS=2, Bc=5)
    _, b, _, _ = _case(fz, CS=2, Bc=5, split=(3, 4))
    for key in ("s", "rk", "rv", "logp", "logp_full", "argmax"):
        assert np.array_equal(a[key], b[key], equal_nan=True), key


def test_plan_rejects_unsupported_shapes(fz):
    c = ri.RLTConfig(d=64, n_layers=1, n_heads=2, head_dim=32, d_ffn=96, window=3, mem_groups=1, vocab=40,
                     dtype="bf16")
    W = ri.make_weights(c, 5)
    e, mem = ri.make_decoder_inputs(c, 2, 4, 9)
    st = O.init_state(O.Cfg.of(c), W, 2)
    rk = np.zeros((1, 2, 2, 3, 32), np.float32)
    acts = np.zeros((2, 4), np.int32)
    for CS, Bc in ((3, 2), (2, 17), (32, 2)):  # cluster not a multiple or divisor of H; > 16 columns; > 16 CTAs
        with pytest.raises(AssertionError, match="plan rejected"):
            _call(fz, c, W, e, mem, st.s, rk, rk, acts, 0, 4, CS, Bc)


def test_fused_decoder_small_workload_plan(fz):
    """The plan the library picks for the small bf16 model on a B300 (16 CTAs
    per cluster, 8 sequences per cluster, two CTAs per head, 43 W_1/W_3 tiles
    over 16 CTAs, a 16-slot window), three steps of one cluster."""
    c = ri.preset("small").cfg
    W = ri.make_weights(c, 3, norm_jitter=0.1)
    B, n = 8, 3
    e, mem = ri.make_decoder_inputs(c, B, n, 7, mem_scale=0.5)
    acts = (np.arange(B * n).reshape(B, n) * 5 % c.vocab).astype(np.int32)
    cfg = O.Cfg.of(c)
    st0 = O.init_state(cfg, W, B)
    rk = np.full((c.n_layers, B, c.n_heads, c.window, c.head_dim), np.nan, np.float32)
    got = _call(fz, c, W, e, mem, st0.s, rk, rk.copy(), acts, 0, n, 16, 8)
    ref_st, ref = O.decode_steps(cfg, W, st0, e, mem, n, acts)
    assert np.abs(got["s"] - ref_st.s).max() <= 2e-3 * np.abs(ref_st.s).max()
    assert np.nanmax(np.abs(got["logp"] - ref.logp)) <= 2e-3 * max(1.0, np.nanmax(np.abs(ref.logp)))
    assert (got["argmax"] == ref.argmax).mean() >= 0.99


def test_fused_decoder_has_no_unordered_shared_accesses(fz, tmp_path):
    """With EMU_JITTER=1 every emulated thread sleeps a random time after each
    block and cluster barrier, so a shared-memory access not ordered by a
    barrier gives results that differ between runs (a barrier removed from
    the kernel does).  Three jittered runs of a 4-CTA cluster case and of a
    two-column-tile case must be bitwise identical, and two of generation
    (token exchange, encoder cache, per-layer memory rows)."""
    lib = os.path.join(os.path.dirname(fz._name), "libfused.so")
    script = tmp_path / "jitter.py"
    script.write_text(
        "import ctypes, sys\n"
        "import numpy as np\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "from tests import test_fused_decoder_emulated_cpu as T\n"
        f"h = ctypes.CDLL({lib!r})\n"
        "h.fused_emu.restype = ctypes.c_int\n"
        "for kw in (dict(CS=4, Bc=8, B=11), dict(CS=2, Bc=16, B=17)):\n"
        "    runs = [T._case(h, **kw)[1] for _ in range(3)]\n"
        "    for k in ('s', 'rk', 'rv', 'logp', 'logp_full', 'argmax'):\n"
        "        assert all(np.array_equal(runs[0][k], r[k], equal_nan=True) for r in runs[1:]), (kw, k)\n"
        "c, W = T._gen_cfg(mem_source=1)\n"
        "prompt = (np.arange(20).reshape(4, 5) * 7 % c.vocab).astype(np.int32)\n"
        "st0 = T._prefill_state(c, W, prompt, 3)\n"
        "g = [T._gen(h, c, W, st0, 3, 4, 4, T.SEED, 0.8, 5) for _ in range(2)]\n"
        "assert np.array_equal(g[0][0], g[1][0]) and np.array_equal(g[0][1], g[1][1])\n"
        "for k in ('s', 'rk', 'rv', 'e', 'mem', 'kv'):\n"
        "    assert np.array_equal(g[0][2][k], g[1][2][k], equal_nan=True), k\n")
    env = dict(os.environ, EMU_JITTER="1")
    r = subprocess.run([sys.executable, str(script)], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]


# ---------------------------------------------------------------------------
# generation through the persistent kernel: each step draws x_p from s_p,
# encodes it against the encoder cache and consumes it

def _prefill_state(c, W, prompt, n):
    """The oracle's prefill of the prompt (e, memory and encoder cache of its
    positions, the decoder state after it) in buffers with room for n more
    positions."""
    cfg = O.Cfg.of(c)
    B, T0 = prompt.shape
    L, H, hd, G, d, Wn = c.n_layers, c.n_heads, c.head_dim, c.mem_groups, c.d, c.window
    Tm = T0 + n
    e0, mem0, kv0 = O.encode(cfg, W, prompt, return_kv=True)
    st, _ = O.decode_steps(cfg, W, O.init_state(cfg, W, B), e0, mem0, T0)
    e = np.full((B, Tm, d), np.nan, np.float32)
    e[:, :T0] = e0
    mem = np.full((G, 2, B, H, Tm, hd), np.nan, np.float32)
    mem[..., :T0, :] = mem0
    kv = np.full((L, 2, B, H, Tm, hd), np.nan, np.float32)
    kv[..., :T0, :] = kv0
    rk = np.full((L, B, H, Wn, hd), np.nan, np.float32)
    rv = rk.copy()
    for l in range(L):
        for j, (kk, vv) in enumerate(st.cache[l]):
            pos = T0 - len(st.cache[l]) + j
            rk[l, :, :, pos % Wn], rv[l, :, :, pos % Wn] = kk, vv
    return dict(s=np.asarray(st.s, np.float32), rk=rk, rv=rv, e=e, mem=mem, kv=kv, pos=T0, T_max=Tm)


def _gen(h, c, W, state, n, CS, Bc, seed, tau=1.0, k=0):
    """n emulated generation steps from state (see _prefill_state); returns
    the tokens, their log-probabilities and the state after them."""
    B = state["s"].shape[0]
    keep = []

    def f32(x):
        a = np.ascontiguousarray(np.asarray(x, np.float32))
        keep.append(a)
        return a.ctypes.data

    s, rk, rv, kv = (np.array(state[key], np.float32) for key in ("s", "rk", "rv", "kv"))
    e_out, m_out = np.array(state["e"], np.float32), np.array(state["mem"], np.float32)
    lp, status, toks = np.zeros((B, n), np.float32), np.zeros(1, np.int32), np.full((B, n), -7, np.int32)
    P = [f32(W[p]) for p in MATS] + [f32(W[p]) for p in VECS] + [f32(state["e"]), f32(state["mem"])]
    P += [s.ctypes.data, rk.ctypes.data, rv.ctypes.data, None, None, None, lp.ctypes.data, None, None,
          status.ctypes.data]
    Q = [f32(W["tok_emb"]), f32(W["enc_attn_norm"]), f32(W["enc_ffn_norm"]), f32(W["enc_norm"]), f32(W["W_K"]),
         f32(W["W_V"]), kv.ctypes.data, toks.ctypes.data, e_out.ctypes.data, m_out.ctypes.data]
    p0 = state["pos"]
    sh = [B, state["T_max"], c.d, c.n_heads, c.head_dim, c.d_ffn, c.n_layers, c.window, c.vocab, c.mem_groups,
          1 if c.gate_mode == 0 else 0, p0, n, k, CS, Bc, c.mem_source, seed >> 32, seed & 0xffffffff]
    rc = h.fused_gen_emu((ctypes.c_int * len(sh))(*sh), (ctypes.c_float * 3)(c.rms_eps, c.rope_theta, tau),
                         (ctypes.c_void_p * len(P))(*P), (ctypes.c_void_p * len(Q))(*Q))
    assert rc == 0 and status[0] == 0
    return toks, lp, dict(s=s, rk=rk, rv=rv, e=e_out, mem=m_out, kv=kv, pos=p0 + n, T_max=state["T_max"])


def _gen_cfg(G=2, mem_source=0, gate_mode=0, hd=32, window=3):
    c = ri.RLTConfig(d=2 * hd, n_layers=2, n_heads=2, head_dim=hd, d_ffn=96, window=window, mem_groups=G, vocab=40,
                     dtype="bf16", gate_mode=gate_mode, mem_source=mem_source)
    return c, ri.make_weights(c, 5, norm_jitter=0.1)


SEED = 0x12345678ABCD


@pytest.mark.parametrize("kw,ckw", [
    (dict(CS=2, Bc=3), {}),
    (dict(CS=4, Bc=8, B=9), {}),                              # one full and one ragged cluster
    (dict(CS=2, Bc=4), dict(mem_source=1)),                   # memory group l from encoder layer l
    (dict(CS=2, Bc=3, k=5, tau=0.8), {}),                     # tempered top-k draws
    (dict(CS=2, Bc=3), dict(gate_mode=1, G=1)),               # the gate discards s; one memory group
    (dict(CS=4, Bc=3), dict(hd=64, window=1)),                # 64-wide heads; the window holds the current token
])
def test_fused_generation_matches_the_oracle(fz, kw, ckw):
    """The generated tokens, fed to the oracle teacher-forced (encoder over
    prompt + generated tokens, decoder from H_0): every draw is the oracle's
    draw at the same uniform number (unless that number lies within 1e-3 of a
    CDF boundary), and the draw's log-probability, the final state and the
    encoder rows, memory rows and encoder cache the kernel wrote agree within
    bf16 rounding (the incremental encoder keeps the attention weights in
    fp32 where the token-parallel oracle rounds them to bf16)."""
    kw = dict(kw)
    B = kw.pop("B", 5)
    k, tau = kw.pop("k", 0), kw.pop("tau", 1.0)
    c, W = _gen_cfg(**ckw)
    T0, n = 5, 4
    prompt = (np.arange(B * T0).reshape(B, T0) * 7 % c.vocab).astype(np.int32)
    toks, lp, st = _gen(fz, c, W, _prefill_state(c, W, prompt, n), n, kw["CS"], kw["Bc"], SEED, tau, k)
    cfg = O.Cfg.of(c)
    full = np.concatenate([prompt, toks], 1)
    e, mem, kv = O.encode(cfg, W, full, return_kv=True)
    acts = np.concatenate([full[:, 1:], np.full((B, 1), -1)], 1).astype(np.int32)
    ref, out = O.decode_steps(cfg, W, O.init_state(cfg, W, B), e, mem, T0 + n, acts, tau, k,
                              emit=range(T0 - 1, T0 + n - 1))
    assert np.abs(lp - out.logp[:, T0 - 1:T0 + n - 1]).max() <= 5e-3
    assert np.abs(st["s"] - ref.s).max() <= 1e-2 * np.abs(ref.s).max()
    for got, want in ((st["e"][:, T0:], e[:, T0:]), (st["mem"][..., T0:, :], mem[..., T0:, :]),
                      (st["kv"][..., T0:, :], kv[..., T0:, :])):
        assert np.abs(got - want).max() <= 2e-2 * np.abs(want).max()
    for b in range(B):
        for j in range(n):
            row, u = out.logits[T0 - 1 + j][b], O.uniform24(SEED, b, T0 + j)
            want = O.sample_token(row, u, tau, k)
            if toks[b, j] != want:
                assert np.abs(np.cumsum(O.sampling_distribution(row, tau, k)) - u).min() < 1e-3, (b, j)


def test_fused_generation_call_split_is_bitwise(fz):
    """Draws use the uniform number of the absolute position, so generating
    4 tokens in one call or in calls of 1 and 3 gives the same tokens,
    log-probabilities, state and written rows, bit for bit."""
    c, W = _gen_cfg()
    B, T0 = 5, 5
    prompt = (np.arange(B * T0).reshape(B, T0) * 7 % c.vocab).astype(np.int32)
    st0 = _prefill_state(c, W, prompt, 4)
    t4, lp4, s4 = _gen(fz, c, W, st0, 4, 2, 3, SEED)
    ta, la, sa = _gen(fz, c, W, st0, 1, 2, 3, SEED)
    tb, lb, sb = _gen(fz, c, W, sa, 3, 2, 3, SEED)
    assert np.array_equal(np.concatenate([ta, tb], 1), t4)
    assert np.array_equal(np.concatenate([la, lb], 1), lp4)
    for key in ("s", "rk", "rv", "e", "mem", "kv"):
        assert np.array_equal(sb[key], s4[key], equal_nan=True), key


def test_fused_generation_small_workload_plan(fz):
    """Generation with the plan the library picks for the small bf16 model
    (16 CTAs per cluster, 8 sequences, four memory groups), two tokens."""
    c = ri.preset("small").cfg
    W = ri.make_weights(c, 3, norm_jitter=0.1)
    B, T0, n = 8, 4, 2
    prompt = (np.arange(B * T0).reshape(B, T0) * 3 % c.vocab).astype(np.int32)
    toks, lp, st = _gen(fz, c, W, _prefill_state(c, W, prompt, n), n, 16, 8, SEED, 0.7, 20)
    cfg = O.Cfg.of(c)
    full = np.concatenate([prompt, toks], 1)
    e, mem = O.encode(cfg, W, full)
    acts = np.concatenate([full[:, 1:], np.full((B, 1), -1)], 1).astype(np.int32)
    ref, out = O.decode_steps(cfg, W, O.init_state(cfg, W, B), e, mem, T0 + n, acts, 0.7, 20,
                              emit=range(T0 - 1, T0 + n - 1))
    assert np.abs(lp - out.logp[:, T0 - 1:T0 + n - 1]).max() <= 5e-3
    assert np.abs(st["s"] - ref.s).max() <= 1e-2 * np.abs(ref.s).max()
    agree = sum(int(toks[b, j] == O.sample_token(out.logits[T0 - 1 + j][b], O.uniform24(SEED, b, T0 + j), 0.7, 20))
                for b in range(B) for j in range(n))
    assert agree >= B * n - 1


@pytest.mark.parametrize("CS,Bc", [(16, 10), (8, 8)])
def test_fused_decoder_phases_in_parts(fz, CS, Bc):
    """Plans whose largest weight phases exceed a stage half (10 sequences
    on 16-CTA clusters; 8-CTA clusters) run those projections in tile-range
    parts, each its own pipeline step: the small model, two steps."""
    c = ri.preset("small").cfg
    W = ri.make_weights(c, 3, norm_jitter=0.1)
    B, n = Bc, 2
    e, mem = ri.make_decoder_inputs(c, B, n, 7, mem_scale=0.5)
    acts = (np.arange(B * n).reshape(B, n) * 5 % c.vocab).astype(np.int32)
    cfg = O.Cfg.of(c)
    st0 = O.init_state(cfg, W, B)
    rk = np.full((c.n_layers, B, c.n_heads, c.window, c.head_dim), np.nan, np.float32)
    got = _call(fz, c, W, e, mem, st0.s, rk, rk.copy(), acts, 0, n, CS, Bc)
    ref_st, ref = O.decode_steps(cfg, W, st0, e, mem, n, acts)
    assert np.abs(got["s"] - ref_st.s).max() <= 2e-3 * np.abs(ref_st.s).max()
    assert np.nanmax(np.abs(got["logp"] - ref.logp)) <= 2e-3 * max(1.0, np.nanmax(np.abs(ref.logp)))
    assert (got["argmax"] == ref.argmax).mean() >= 0.95
