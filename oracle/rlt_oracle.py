"""Plain CPU oracle of the Recurrent Looped Transformer (RLT) hot path.

TEST INFRASTRUCTURE.  This module exists to check the CUDA path.  Only the test
suite, the smoke check and the benchmark's CPU-baseline leg may import it; the
product library never calls it and has no CPU fallback.  It shares no code with
the CUDA path (it has its own rounding, RoPE, softmax and top-k).

What it computes (sources, by page title and section):

* "Understanding and Applying the Recurrent Looped Transformer Architecture",
  section "How the Architecture Works": the state H_t = (s_t, C_t^D), H_0 =
  (s_*, empty), the transition (s_t, C_t^D) = D_phi(Merge(e_t, s_{t-1}), M_<=t,
  C_{t-1}^D, t) and the head p(x_{t+1}|x_{1:t}) = softmax(W_o RMSNorm_o(s_t));
  sub-section "Three forms of context": cross-attention reads memory only
  through the current position, the window W includes the current token and
  leaves at most W-1 historical entries.
* "Princeton Researcher Proposes Recurrent Looped Transformer to Carry Decoder
  State Across Tokens", architecture paragraph: causal token-parallel encoder
  producing e_t, memory M_<=t projected from it in G groups (G=1 shared, G=L_D
  per layer); gated merge of e_t with s_{t-1}; each decoder block runs causal
  SWA over decoder activations, cross-attention to encoder memory and an FFN;
  attention and FFN weights of corresponding encoder/decoder layers are tied.
  Prior-work paragraph: the decoder's global KV is projected from the final
  encoder states.
* Same page, RL paragraph, and "Understanding and Applying...", section
  "Current-Policy Reinforcement Learning Replay": an action is scored before it
  is consumed; the behaviour log-probability includes temperature and top-k
  truncation.

Readings taken where the pages are silent (each is the plainest one):
pre-norm RMSNorm x/sqrt(mean(x^2)+eps)*g before every sub-layer with residual
adds; a final RMSNorm on the encoder output; every memory group projected from
that final e; decoder-only cross-attention projections W_Qx, W_Ox; untied norm
gains; vector gate z = sigmoid(W_g [e_t; s_{t-1}] + b_g), u = z*s_{t-1} +
(1-z)*e_t; rotate-half RoPE (theta 1e4) on encoder and decoder self-attention
at absolute position p = t-1, none on cross-attention; SWA keys cached after
RoPE; cross-attention over memory positions 1..t inclusive; s_t is the residual
stream after the last decoder block (no norm); SwiGLU FFN W_2(silu(W_1 a) *
W_3 a); tempered top-k log-prob renormalised over the k largest logits (ties to
the lower token id), -inf outside.

Precision: float64 throughout.  With ``bf16=True`` the values are rounded to
bfloat16 (nearest even) at exactly the points the bf16 configurations store in
bf16: every matrix-multiply input (normed activations, attention outputs before
the output projections, the SwiGLU product, [e; s] into the gate, the head's
normed state), e, the memory K/V, the ring K/V after RoPE, the encoder's
q/k/v after RoPE, and P before the P.V product in the encoder attention.  The
residual stream, s, softmax statistics and logits are not rounded.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

F64 = np.float64


# ----------------------------------------------------------------------------
# elementary operations

def bf16(x):
    """Round float64 values to the nearest bfloat16 value (ties to even)."""
    x = np.ascontiguousarray(x, dtype=F64)
    b = x.view(np.uint64)
    # bfloat16 keeps 7 explicit mantissa bits; float64 has 52: drop 45 bits.
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    b = (b + lsb + np.uint64((1 << 44) - 1)) & ~np.uint64((1 << 45) - 1)
    return b.view(F64)


class Numerics:
    """Rounding policy: identity in fp32/fp64 configs, bfloat16 in bf16 configs."""

    def __init__(self, bf16_mode: bool):
        self.bf16 = bool(bf16_mode)

    def r(self, x):
        return bf16(x) if self.bf16 else np.asarray(x, dtype=F64)


def rmsnorm(x, g, eps):
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    x = np.asarray(x, F64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(g, F64)


def silu(x):
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def sigmoid(x):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-x))


def rope_angles(pos, head_dim, theta):
    """angle[p, i] = p * theta^(-2i/head_dim), i < head_dim/2."""
    i = np.arange(head_dim // 2, dtype=F64)
    inv = theta ** (-2.0 * i / head_dim)
    return np.asarray(pos, F64)[..., None] * inv


def rope(x, pos, theta):
    """Rotate-half RoPE: pairs (x_i, x_{i+hd/2}) rotated by angle(p, i).

    x: [..., P, hd] with positions pos[P] on the second-to-last axis.
    """
    hd = x.shape[-1]
    ang = rope_angles(pos, hd, theta)             # [P, hd/2]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., : hd // 2], x[..., hd // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softmax_last(x):
    m = np.max(x, axis=-1, keepdims=True)
    p = np.exp(x - m)
    return p / np.sum(p, axis=-1, keepdims=True)


def logsumexp_last(x):
    m = np.max(x, axis=-1, keepdims=True)
    return (m + np.log(np.sum(np.exp(x - m), axis=-1, keepdims=True)))[..., 0]


# ----------------------------------------------------------------------------
# configuration

@dataclass
class Cfg:
    d: int
    n_layers: int
    n_heads: int
    head_dim: int
    d_ffn: int
    window: int
    mem_groups: int
    vocab: int
    bf16: bool
    rms_eps: float = 1e-6
    rope_theta: float = 1e4
    gate_mode: int = 0          # 1: gate forced to discard s_{t-1} (z = 0)
    mem_source: int = 0         # 0: every group from the final e; 1: group l from layer l's state

    @staticmethod
    def of(c) -> "Cfg":
        """Build from any object or dict with the same field names (dtype 'bf16'/'f32')."""
        if isinstance(c, dict):
            get = lambda k, dflt=None: c.get(k, dflt)  # noqa: E731
        else:
            get = lambda k, dflt=None: getattr(c, k, dflt)  # noqa: E731
        return Cfg(d=get("d"), n_layers=get("n_layers"), n_heads=get("n_heads"),
                   head_dim=get("head_dim"), d_ffn=get("d_ffn"), window=get("window"),
                   mem_groups=get("mem_groups"), vocab=get("vocab"),
                   bf16=(get("dtype") == "bf16"), rms_eps=get("rms_eps"),
                   rope_theta=get("rope_theta"), gate_mode=get("gate_mode"),
                   mem_source=get("mem_source", 0))

    def group_of(self, layer: int) -> int:
        """Memory group read by decoder layer l: 0 when G=1, l when G=L_D."""
        return 0 if self.mem_groups == 1 else layer


def _w(W, name, l=None):
    a = W[name] if l is None else W[name][l]
    return np.asarray(a, F64)


# ----------------------------------------------------------------------------
# encoder (producer): e and memory M, token-parallel with a causal mask

def causal_attention(q, k, v, nx: Numerics, round_p: bool):
    """softmax(q k^T / sqrt(hd)) v over positions j <= i; q,k,v [..., P, hd].

    With round_p the unnormalised weights exp(s - rowmax) are rounded before
    the product with v and the row sum is taken from the unrounded weights.
    """
    P, hd = q.shape[-2:]
    s = (q @ np.swapaxes(k, -1, -2)) / math.sqrt(hd)
    s = np.where(np.tril(np.ones((P, P), bool)), s, -np.inf)
    m = np.max(s, axis=-1, keepdims=True)
    p = np.exp(s - m)
    lsum = np.sum(p, axis=-1, keepdims=True)
    pv = nx.r(p) if round_p else p
    return (pv @ v) / lsum


def encode(cfg: Cfg, W: Dict[str, np.ndarray], tokens: np.ndarray, return_hidden=False, return_kv=False):
    """Causal encoder and memory projection.

    tokens int [B, T] (position p = column index).  Returns e [B, T, d] and
    mem [G, 2, B, H, T, hd] (index 0 = keys, 1 = values); with return_kv
    also every layer's self-attention keys (after RoPE) and values
    [L, 2, B, H, T, hd] as the attention used them (the encoder cache that
    incremental encoding of later tokens attends to).

    Memory source.  The reading taken projects every group from the final e
    (P5 architecture paragraph: decoder global keys and values come from the
    final encoder states).  The other reading of per-layer memory (G = L_D, the
    configs with per-layer memory projections) takes group l from encoder
    layer l's state: mem_source = 1 projects group l from
    RMSNorm_e(h^l), the residual stream after layer l under the final norm's
    gain, so that the last group coincides with the first reading's.
    """
    nx = Numerics(cfg.bf16)
    B, T = tokens.shape
    d, H, hd = cfg.d, cfg.n_heads, cfg.head_dim
    pos = np.arange(T)
    if cfg.mem_source == 1 and cfg.mem_groups != cfg.n_layers:
        raise ValueError("per-layer memory needs one group per layer")
    layer_states = []
    kv = np.empty((cfg.n_layers, 2, B, H, T, hd), F64) if return_kv else None
    h = _w(W, "tok_emb")[tokens]                                  # [B, T, d]
    for l in range(cfg.n_layers):
        a = nx.r(rmsnorm(h, _w(W, "enc_attn_norm", l), cfg.rms_eps))
        qkv = a @ _w(W, "W_qkv", l).T                             # [B, T, 3d]
        q = qkv[..., :d].reshape(B, T, H, hd).transpose(0, 2, 1, 3)
        k = qkv[..., d:2 * d].reshape(B, T, H, hd).transpose(0, 2, 1, 3)
        v = qkv[..., 2 * d:].reshape(B, T, H, hd).transpose(0, 2, 1, 3)
        q = nx.r(rope(q, pos, cfg.rope_theta))
        k = nx.r(rope(k, pos, cfg.rope_theta))
        v = nx.r(v)
        if return_kv:
            kv[l, 0], kv[l, 1] = k, v
        o = np.empty((B, H, T, hd), F64)
        for b in range(B):
            o[b] = causal_attention(q[b], k[b], v[b], nx, round_p=cfg.bf16)
        o = o.transpose(0, 2, 1, 3).reshape(B, T, d)
        h = h + nx.r(o) @ _w(W, "W_O", l).T
        bb = nx.r(rmsnorm(h, _w(W, "enc_ffn_norm", l), cfg.rms_eps))
        m = nx.r(silu(bb @ _w(W, "W_1", l).T) * (bb @ _w(W, "W_3", l).T))
        h = h + m @ _w(W, "W_2", l).T
        if cfg.mem_source == 1:
            layer_states.append(nx.r(rmsnorm(h, _w(W, "enc_norm"), cfg.rms_eps)))
    e = nx.r(rmsnorm(h, _w(W, "enc_norm"), cfg.rms_eps))
    if cfg.mem_source == 1:
        mem = memory_projection(cfg, W, layer_states)
    else:
        mem = memory_projection(cfg, W, [e] * cfg.mem_groups)
    out = (e, mem)
    if return_hidden:
        out += (h,)
    if return_kv:
        out += (kv,)
    return out


def memory_projection(cfg: Cfg, W, sources):
    """M^g = (x_g W_K^g^T, x_g W_V^g^T) for each group g from its source x_g
    [B, T, d], stored [G, 2, B, H, T, hd]."""
    nx = Numerics(cfg.bf16)
    B, T, d = sources[0].shape
    H, hd = cfg.n_heads, cfg.head_dim
    mem = np.empty((cfg.mem_groups, 2, B, H, T, hd), F64)
    for g in range(cfg.mem_groups):
        kk = nx.r(sources[g] @ _w(W, "W_K", g).T)
        vv = nx.r(sources[g] @ _w(W, "W_V", g).T)
        mem[g, 0] = kk.reshape(B, T, H, hd).transpose(0, 2, 1, 3)
        mem[g, 1] = vv.reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    return mem


# ----------------------------------------------------------------------------
# recurrent decoder

@dataclass
class State:
    """H_t = (s_t, C_t^D) for B sequences, plus the number of consumed tokens.

    cache[l] is a list (oldest first) of (k, v) pairs [B, H, hd] holding at most
    window-1 historical entries after a step.
    """
    s: np.ndarray
    cache: List[list]
    pos: int = 0

    def copy(self):
        return State(self.s.copy(), [list(c) for c in self.cache], self.pos)


def init_state(cfg: Cfg, W, B: int) -> State:
    """H_0 = (s_*, empty cache), taken once before the first token."""
    s = np.broadcast_to(_w(W, "s_star"), (B, cfg.d)).copy()
    return State(s, [[] for _ in range(cfg.n_layers)], 0)


def history_keep(window: int) -> int:
    """Historical entries retained after a step: the window holds the current token
    plus at most W-1 previous ones."""
    return window - 1


def merge(cfg: Cfg, W, e_t, s_prev, nx: Numerics, trace=None):
    """u = z * s_{t-1} + (1 - z) * e_t with z = sigmoid(W_g [e_t; s_{t-1}] + b_g)."""
    if cfg.gate_mode == 1:
        z = np.zeros_like(s_prev)
    else:
        x = nx.r(np.concatenate([e_t, s_prev], axis=-1))
        z = sigmoid(x @ _w(W, "W_g").T + _w(W, "b_g"))
    if trace is not None:
        trace["z"] = z
    return z * s_prev + (1.0 - z) * e_t


def swa_attend(q, ks, vs, hd):
    """Attention of q [B,H,hd] over entries ks, vs [B,H,n,hd] (all inside the window)."""
    s = np.einsum("bhd,bhnd->bhn", q, ks) / math.sqrt(hd)
    p = softmax_last(s)
    return np.einsum("bhn,bhnd->bhd", p, vs)


def memory_range(t: int) -> int:
    """Cross-attention reads memory positions 1..t (inclusive) at step t."""
    return t


def decode_step(cfg: Cfg, W, st: State, e_t, mem, trace=None) -> State:
    """One transition: consume the token at position p = st.pos (step t = p + 1).

    e_t [B, d] is the encoder output at position p, mem [G, 2, B, H, T_mem, hd].
    Returns the new state; st is not modified.
    """
    nx = Numerics(cfg.bf16)
    B = e_t.shape[0]
    d, H, hd = cfg.d, cfg.n_heads, cfg.head_dim
    t = st.pos + 1
    p = st.pos
    h = merge(cfg, W, np.asarray(e_t, F64), st.s, nx, trace)
    if trace is not None:
        trace["u"] = h.copy()
        trace["swa_out"], trace["x_out"] = [], []
    new_cache = []
    for l in range(cfg.n_layers):
        # sliding-window self-attention over this layer's decoder activations
        a = nx.r(rmsnorm(h, _w(W, "dec_attn_norm", l), cfg.rms_eps))
        qkv = a @ _w(W, "W_qkv", l).T
        q = qkv[:, :d].reshape(B, H, 1, hd)
        k = qkv[:, d:2 * d].reshape(B, H, 1, hd)
        v = qkv[:, 2 * d:].reshape(B, H, hd)
        q = rope(q, [p], cfg.rope_theta)[:, :, 0]
        k = nx.r(rope(k, [p], cfg.rope_theta)[:, :, 0])
        v = nx.r(v)
        entries = st.cache[l] + [(k, v)]
        ks = np.stack([e[0] for e in entries], axis=2)           # [B, H, n, hd]
        vs = np.stack([e[1] for e in entries], axis=2)
        o = swa_attend(q, ks, vs, hd).reshape(B, d)
        if trace is not None:
            trace["swa_out"].append(o.copy())
        h = h + nx.r(o) @ _w(W, "W_O", l).T
        keep = history_keep(cfg.window)
        new_cache.append(entries[max(0, len(entries) - keep):] if keep > 0 else [])
        # cross-attention to encoder memory positions 1..t
        c = nx.r(rmsnorm(h, _w(W, "dec_xattn_norm", l), cfg.rms_eps))
        qx = (c @ _w(W, "W_Qx", l).T).reshape(B, H, hd)
        g = cfg.group_of(l)
        n_mem = memory_range(t)
        km = np.asarray(mem[g, 0, :, :, :n_mem], F64)
        vm = np.asarray(mem[g, 1, :, :, :n_mem], F64)
        ox = swa_attend(qx, km, vm, hd).reshape(B, d)
        if trace is not None:
            trace["x_out"].append(ox.copy())
        h = h + nx.r(ox) @ _w(W, "W_Ox", l).T
        # SwiGLU feed-forward
        bb = nx.r(rmsnorm(h, _w(W, "dec_ffn_norm", l), cfg.rms_eps))
        m = nx.r(silu(bb @ _w(W, "W_1", l).T) * (bb @ _w(W, "W_3", l).T))
        h = h + m @ _w(W, "W_2", l).T
    return State(h, new_cache, t)


# ----------------------------------------------------------------------------
# output head and replay scoring

def head_logits(cfg: Cfg, W, s):
    """logits = W_o RMSNorm_o(s) (unnormalised log-probabilities of x_{t+1})."""
    nx = Numerics(cfg.bf16)
    a = nx.r(rmsnorm(s, _w(W, "head_norm"), cfg.rms_eps))
    return a @ _w(W, "W_o").T


def topk_mask(logits, k):
    """Boolean mask of the k largest entries per row, ties broken by lower id."""
    Bn, V = logits.shape
    mask = np.zeros((Bn, V), bool)
    if k <= 0 or k >= V:
        mask[:] = True
        return mask
    ids = np.arange(V)
    for b in range(Bn):
        order = np.lexsort((ids, -logits[b]))     # by value desc, then id asc
        mask[b, order[:k]] = True
    return mask


def score(logits, actions, temperature=1.0, top_k=0):
    """Behaviour log-probabilities of actions under tempered (top-k) sampling.

    Returns (lp, lp_full): lp_full = l_a/tau - LSE(l/tau) over the vocabulary;
    lp is the same renormalised over the top-k set, -inf for actions outside it
    (lp = lp_full when top_k is 0 or >= V).  Rows with action < 0 give NaN.
    """
    x = np.asarray(logits, F64) / temperature
    Bn, V = x.shape
    lse = logsumexp_last(x)
    mask = topk_mask(x, top_k)
    xm = np.where(mask, x, -np.inf)
    lse_k = logsumexp_last(xm)
    lp_full = np.full(Bn, np.nan)
    lp = np.full(Bn, np.nan)
    for b in range(Bn):
        a = int(actions[b])
        if a < 0:
            continue
        lp_full[b] = x[b, a] - lse[b]
        lp[b] = (x[b, a] - lse_k[b]) if mask[b, a] else -np.inf
    return lp, lp_full


# ----------------------------------------------------------------------------
# generation: drawing the next token ("Understanding and Applying the Recurrent
# Looped Transformer Architecture", "Autoregressive generation": the
# distribution of the next token comes from the preceding state, a token is
# sampled from it, encoded incrementally and consumed once)

_M64 = (1 << 64) - 1


def uniform24(seed: int, b: int, pos: int) -> float:
    """The uniform number in [0, 1) of draw (seed, sequence b, position pos):
    the SplitMix64 output function (Steele, Lea and Flood, "Fast splittable
    pseudorandom number generators", OOPSLA 2014) on the counter
    seed + (pos * 2^32 + b + 1) * 0x9E3779B97F4A7C15 (mod 2^64), keeping the
    top 24 bits.  Written from the published mixing function; the library has
    its own copy (the two share no code, only the definition)."""
    z = (seed + ((pos << 32) + b + 1) * 0x9E3779B97F4A7C15) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    z ^= z >> 31
    return (z >> 40) / float(1 << 24)


def sampling_distribution(logits_row, temperature=1.0, top_k=0):
    """Probabilities of the tempered (top-k) distribution over the vocabulary
    (zero outside the top-k set, ties to the lower id), float64."""
    x = np.asarray(logits_row, F64)[None, :] / temperature
    mask = topk_mask(x, top_k)[0]
    xm = np.where(mask, x[0], -np.inf)
    p = np.exp(xm - np.max(xm))
    return p / p.sum()


def sample_token(logits_row, u, temperature=1.0, top_k=0):
    """The token drawn with uniform number u: the first id, in id order, at
    which the cumulative probability of the tempered (top-k) distribution
    exceeds u (the last member when rounding leaves none)."""
    p = sampling_distribution(logits_row, temperature, top_k)
    c = np.cumsum(p)
    hit = np.nonzero(c > u)[0]
    if len(hit):
        return int(hit[0])
    return int(np.nonzero(p > 0)[0][-1])


@dataclass
class StepsOut:
    logp: np.ndarray            # [B, n]
    logp_full: np.ndarray       # [B, n]
    argmax: np.ndarray          # [B, n]
    logits: Dict[int, np.ndarray] = field(default_factory=dict)   # step index -> [B, V]
    s_hist: List[np.ndarray] = field(default_factory=list)


def decode_steps(cfg: Cfg, W, st: State, e, mem, n: int, actions=None, temperature=1.0,
                 top_k=0, emit=(), keep_s=False):
    """Advance every sequence n tokens from st.pos; score actions[b, i] after step i.

    e [B, T_mem, d], mem [G, 2, B, H, T_mem, hd].  Returns (new_state, StepsOut).
    """
    B = st.s.shape[0]
    out = StepsOut(np.full((B, n), np.nan), np.full((B, n), np.nan), np.zeros((B, n), np.int64))
    emit = set(int(i) for i in emit)
    for i in range(n):
        st = decode_step(cfg, W, st, e[:, st.pos], mem)
        lg = head_logits(cfg, W, st.s)
        out.argmax[:, i] = np.argmax(lg, axis=-1)
        if actions is not None:
            lp, lpf = score(lg, actions[:, i], temperature, top_k)
            out.logp[:, i], out.logp_full[:, i] = lp, lpf
        if i in emit:
            out.logits[i] = lg
        if keep_s:
            out.s_hist.append(st.s.copy())
    return st, out


def run_sequence(cfg: Cfg, W, tokens, actions=None, temperature=1.0, top_k=0, emit=(), keep_s=False):
    """encode + H_0 + decode every position of tokens [B, T]."""
    e, mem = encode(cfg, W, tokens)
    st = init_state(cfg, W, tokens.shape[0])
    st, out = decode_steps(cfg, W, st, e, mem, tokens.shape[1], actions, temperature, top_k,
                           emit, keep_s)
    return e, mem, st, out
