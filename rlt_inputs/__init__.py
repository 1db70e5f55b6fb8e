"""Seeded synthetic inputs for the RLT decoder transition: shapes, weights, tokens.

This module is shared by the test-side oracle and the CUDA path.  It holds no
arithmetic of the method itself: it only draws seeded random numbers, converts
them to the storage format of a configuration (float32 or bfloat16, rounding
to nearest even), and describes the five workload shapes.

Sources for the shapes (page "Understanding and Applying the Recurrent Looped
Transformer Architecture", sections "Concrete model configuration" and
"Preliminary Synthetic Results"; page "Princeton Researcher Proposes Recurrent
Looped Transformer...", architecture paragraph: 48 tied encoder and decoder
layers, window W, G memory groups).  The exact sizes (d, heads, FFN width,
window, vocabulary, batch, length, token distribution) are those of the five
synthetic workloads this project measures; the pages themselves give only the
48+48 layer count.

Weight draw order and streams
-----------------------------
Every tensor is drawn from its own PCG64 stream, keyed by (seed, tensor index)
through ``numpy.random.SeedSequence``, as float32 ``standard_normal`` times its
scale.  bf16 configurations round those float32 draws to bfloat16
(round-to-nearest-even) and both sides use the rounded values exactly.
Norm gains are 1 and the gate bias is 0 unless a test asks for jitter.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, asdict, replace
from typing import Dict, Optional, Tuple

import numpy as np

__all__ = [
    "RLTConfig", "Workload", "PRESETS", "preset", "weight_specs", "make_weights",
    "make_tokens", "make_splits", "teacher_actions", "bf16_round_f32",
    "weights_nbytes", "make_decoder_inputs",
]


@dataclass(frozen=True)
class RLTConfig:
    """Model shape.  d = n_heads * head_dim; L_E = L_D = n_layers (tied)."""
    d: int
    n_layers: int
    n_heads: int
    head_dim: int
    d_ffn: int
    window: int
    mem_groups: int          # 1 (shared memory) or n_layers (one group per layer)
    vocab: int
    dtype: str               # "f32" or "bf16" (bf16 storage, fp32 accumulation)
    sigma: float = 0.02      # std of every weight matrix
    s_star_sigma: float = 0.02
    rms_eps: float = 1e-6
    rope_theta: float = 1e4
    gate_mode: int = 0       # 0 learned gate, 1 gate forced to discard s_{t-1}
    mem_source: int = 0      # 0 every memory group from the final e, 1 group l from encoder layer l

    def __post_init__(self):
        assert self.d == self.n_heads * self.head_dim
        assert self.mem_groups in (1, self.n_layers)
        assert self.mem_source in (0, 1)
        assert self.mem_source == 0 or self.mem_groups == self.n_layers
        assert self.dtype in ("f32", "bf16")
        assert self.head_dim % 2 == 0


@dataclass(frozen=True)
class Workload:
    """A batch of synthetic sequences for one configuration."""
    name: str
    cfg: RLTConfig
    B: int
    T: int
    tokens: str                      # "bits", "uniform5", "zipf"
    split: Tuple[int, int]           # prompt/response split range [lo, hi] (inclusive)
    seed: int
    zipf_s: float = 1.1
    temperature: float = 1.0
    top_k: int = 0
    score_prompt: bool = True        # False: only response positions are scored


def _cfg(**kw) -> RLTConfig:
    return RLTConfig(**kw)


PRESETS: Dict[str, Workload] = {
    # Tiny fp32 model of the size of the pages' ~79k-parameter experiments.
    "tiny": Workload(
        "tiny", _cfg(d=64, n_layers=2, n_heads=4, head_dim=16, d_ffn=172, window=4,
                     mem_groups=1, vocab=2, dtype="f32"),
        B=8, T=64, tokens="bits", split=(32, 32), seed=0),
    "small": Workload(
        "small", _cfg(d=256, n_layers=4, n_heads=8, head_dim=32, d_ffn=688, window=16,
                      mem_groups=4, vocab=64, dtype="bf16"),
        B=64, T=512, tokens="uniform5", split=(64, 448), seed=1),
    "medium": Workload(
        "medium", _cfg(d=1024, n_layers=12, n_heads=16, head_dim=64, d_ffn=2816, window=128,
                       mem_groups=1, vocab=32000, dtype="bf16"),
        B=128, T=2048, tokens="zipf", split=(1536, 1536), seed=2),
    "refdep": Workload(
        "refdep", _cfg(d=2048, n_layers=48, n_heads=16, head_dim=128, d_ffn=5632, window=256,
                       mem_groups=1, vocab=32000, dtype="bf16", sigma=0.02 / math.sqrt(96.0)),
        B=64, T=4096, tokens="zipf", split=(3072, 3072), seed=3),
    "rlreplay": Workload(
        "rlreplay", _cfg(d=1024, n_layers=24, n_heads=16, head_dim=64, d_ffn=2816, window=64,
                         mem_groups=24, vocab=32000, dtype="bf16"),
        B=1024, T=256, tokens="zipf", split=(32, 192), seed=4,
        temperature=0.7, top_k=50, score_prompt=False),
}


def preset(name: str, **overrides) -> Workload:
    """Return a preset workload; keyword overrides apply to the workload or its config."""
    w = PRESETS[name]
    cfg_keys = set(RLTConfig.__dataclass_fields__)
    cfg_over = {k: v for k, v in overrides.items() if k in cfg_keys}
    wl_over = {k: v for k, v in overrides.items() if k not in cfg_keys}
    cfg = replace(w.cfg, **cfg_over) if cfg_over else w.cfg
    return replace(w, cfg=cfg, **wl_over)


def weight_specs(cfg: RLTConfig):
    """(name, shape, kind) in draw order.  kind: 'mat' N(0, sigma), 'sstar', 'ones', 'zeros'.

    Matrices follow the y = x W^T convention: W[out, in].  Per-layer tensors are
    stacked on a leading layer axis.  W_qkv rows are [q; k; v], each head-major
    (row h*head_dim + i).  W_g acts on [e_t; s_{t-1}] (e first).
    """
    d, L, f, V, G = cfg.d, cfg.n_layers, cfg.d_ffn, cfg.vocab, cfg.mem_groups
    return [
        ("tok_emb", (V, d), "mat"),
        ("s_star", (d,), "sstar"),
        ("W_g", (d, 2 * d), "mat"),
        ("b_g", (d,), "zeros"),
        ("W_qkv", (L, 3 * d, d), "mat"),
        ("W_O", (L, d, d), "mat"),
        ("W_1", (L, f, d), "mat"),
        ("W_3", (L, f, d), "mat"),
        ("W_2", (L, d, f), "mat"),
        ("W_Qx", (L, d, d), "mat"),
        ("W_Ox", (L, d, d), "mat"),
        ("W_K", (G, d, d), "mat"),
        ("W_V", (G, d, d), "mat"),
        ("W_o", (V, d), "mat"),
        ("enc_attn_norm", (L, d), "ones"),
        ("enc_ffn_norm", (L, d), "ones"),
        ("enc_norm", (d,), "ones"),
        ("dec_attn_norm", (L, d), "ones"),
        ("dec_xattn_norm", (L, d), "ones"),
        ("dec_ffn_norm", (L, d), "ones"),
        ("head_norm", (d,), "ones"),
    ]


def weights_nbytes(cfg: RLTConfig) -> int:
    n = 0
    for _, shape, kind in weight_specs(cfg):
        el = 2 if (kind == "mat" and cfg.dtype == "bf16") else 4
        n += int(np.prod(shape)) * el
    return n


def bf16_round_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32.

    This is a storage-format conversion of generated inputs, not method arithmetic.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = (b + (((b >> 16) & 1) + 0x7FFF)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


def _stream(seed: int, idx: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, idx])))


def make_weights(cfg: RLTConfig, seed: int, norm_jitter: float = 0.0,
                 gate_bias: float = 0.0, only: Optional[set] = None) -> Dict[str, np.ndarray]:
    """Seeded weights as float32 arrays (bf16-representable values for bf16 configs).

    norm_jitter > 0 draws norm gains 1 + N(0, norm_jitter) (tests use it so that
    a gain applied to the wrong sub-layer is visible); gate_bias fills b_g.
    """
    out = {}
    for idx, (name, shape, kind) in enumerate(weight_specs(cfg)):
        if only is not None and name not in only:
            continue
        rng = _stream(seed, idx)
        if kind == "mat":
            a = rng.standard_normal(shape, dtype=np.float32) * np.float32(cfg.sigma)
            if cfg.dtype == "bf16":
                a = bf16_round_f32(a)
        elif kind == "sstar":
            a = rng.standard_normal(shape, dtype=np.float32) * np.float32(cfg.s_star_sigma)
        elif kind == "ones":
            a = np.ones(shape, np.float32)
            if norm_jitter:
                a = a + rng.standard_normal(shape, dtype=np.float32) * np.float32(norm_jitter)
        else:
            a = np.full(shape, gate_bias, np.float32)
        out[name] = np.ascontiguousarray(a, dtype=np.float32)
    return out


def make_decoder_inputs(cfg: RLTConfig, B: int, T: int, seed: int, e_scale: float = 1.0,
                        mem_scale: float = 0.3) -> Tuple[np.ndarray, np.ndarray]:
    """Seeded stand-ins for the encoder output and memory, for calls that take
    them as inputs (the decoder's backward pass): e [B, T, d] ~ N(0, e_scale^2)
    (unit-RMS rows, like an RMSNorm output at unit gain) and mem
    [G, 2, B, H, T, hd] ~ N(0, mem_scale^2) (a projection of such rows by
    N(0, sigma^2) weights has std sigma sqrt(d)), float32, bf16-representable
    for bf16 configurations."""
    e = _stream(seed, 2000).standard_normal((B, T, cfg.d), dtype=np.float32) * np.float32(e_scale)
    mem = _stream(seed, 2001).standard_normal((cfg.mem_groups, 2, B, cfg.n_heads, T, cfg.head_dim),
                                              dtype=np.float32) * np.float32(mem_scale)
    if cfg.dtype == "bf16":
        e, mem = bf16_round_f32(e), bf16_round_f32(mem)
    return np.ascontiguousarray(e), np.ascontiguousarray(mem)


def make_tokens(wl: Workload, B: Optional[int] = None, T: Optional[int] = None,
                seed: Optional[int] = None) -> np.ndarray:
    """int32 [B, T] token ids drawn per the workload's distribution.

    'bits': uniform {0,1}; 'uniform5': uniform {0..4}; 'zipf': Zipf(s) over the
    vocabulary, rank k (1-based) has probability proportional to k^-s and id k-1,
    drawn by a finite inverse CDF.
    """
    B = wl.B if B is None else B
    T = wl.T if T is None else T
    rng = _stream(wl.seed if seed is None else seed, 1000)
    V = wl.cfg.vocab
    if wl.tokens == "bits":
        x = rng.integers(0, 2, size=(B, T))
    elif wl.tokens == "uniform5":
        x = rng.integers(0, min(5, V), size=(B, T))
    elif wl.tokens == "zipf":
        k = np.arange(1, V + 1, dtype=np.float64)
        p = k ** (-wl.zipf_s)
        cdf = np.cumsum(p)
        cdf /= cdf[-1]
        u = rng.random(size=(B, T))
        x = np.minimum(np.searchsorted(cdf, u, side="right"), V - 1)
    else:
        raise ValueError(wl.tokens)
    return np.ascontiguousarray(x, dtype=np.int32)


def make_splits(wl: Workload, B: Optional[int] = None, seed: Optional[int] = None) -> np.ndarray:
    """int32 [B] prompt lengths, uniform in the workload's inclusive split range."""
    B = wl.B if B is None else B
    rng = _stream(wl.seed if seed is None else seed, 2000)
    lo, hi = wl.split
    return rng.integers(lo, hi + 1, size=B).astype(np.int32)


def teacher_actions(tokens: np.ndarray, p0: int, n: int, prompt_len: Optional[np.ndarray] = None) -> np.ndarray:
    """int32 [B, n]: the action scored after consuming token index p0+i is token p0+i+1.

    Steps with no next token, and (when prompt_len is given) steps whose next
    token lies inside the prompt, get -1 (not scored).
    """
    B, T = tokens.shape
    a = np.full((B, n), -1, np.int32)
    for i in range(n):
        j = p0 + i + 1
        if j < T:
            a[:, i] = tokens[:, j]
            if prompt_len is not None:
                a[prompt_len > j, i] = -1
    return a
