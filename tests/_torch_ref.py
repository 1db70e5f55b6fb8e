"""Token-parallel compositions of PyTorch library routines, used to pin the oracle.

These are not a second copy of the oracle's loops: attention comes from
``scaled_dot_product_attention`` with explicit masks, normalisation from
``rms_norm``, RoPE from complex multiplication (``torch.polar``), and the head
from ``log_softmax`` / ``topk``.  Everything runs in float64 on the CPU and
applies to float32-storage configurations (no bf16 rounding points).
"""
import math

import numpy as np
import torch
import torch.nn.functional as F

D = torch.float64


def T(x):
    return torch.as_tensor(np.asarray(x), dtype=D)


def rope_complex(x, pos, theta):
    """x [..., P, hd]: pair i with i + hd/2 as one complex number, multiplied by e^{i p w_i}."""
    hd = x.shape[-1]
    w = theta ** (-torch.arange(hd // 2, dtype=D) * 2.0 / hd)
    ang = torch.as_tensor(pos, dtype=D)[:, None] * w[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)
    z = torch.complex(x[..., : hd // 2], x[..., hd // 2:]) * rot
    return torch.cat([z.real, z.imag], dim=-1)


def _heads(x, H):
    B, P, d = x.shape
    return x.reshape(B, P, H, d // H).transpose(1, 2)


def _merge_heads(x):
    B, H, P, hd = x.shape
    return x.transpose(1, 2).reshape(B, P, H * hd)


def encoder(cfg, W, tokens, return_kv=False):
    """Return e [B,T,d] and memory [G,2,B,H,T,hd] for an f32-storage config
    (and with return_kv every layer's keys after RoPE and values
    [L,2,B,H,T,hd])."""
    d, H = cfg.d, cfg.n_heads
    tok = torch.as_tensor(tokens, dtype=torch.long)
    B, P = tok.shape
    pos = torch.arange(P)
    h = F.embedding(tok, T(W["tok_emb"]))
    hidden, kv = [], []
    for l in range(cfg.n_layers):
        a = F.rms_norm(h, (d,), weight=T(W["enc_attn_norm"][l]), eps=cfg.rms_eps)
        q, k, v = F.linear(a, T(W["W_qkv"][l])).split(d, dim=-1)
        q, k, v = _heads(q, H), _heads(k, H), _heads(v, H)
        q, k = rope_complex(q, pos, cfg.rope_theta), rope_complex(k, pos, cfg.rope_theta)
        kv.append(torch.stack([k, v]))
        o = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        h = h + F.linear(_merge_heads(o), T(W["W_O"][l]))
        b = F.rms_norm(h, (d,), weight=T(W["enc_ffn_norm"][l]), eps=cfg.rms_eps)
        h = h + F.linear(F.silu(F.linear(b, T(W["W_1"][l]))) * F.linear(b, T(W["W_3"][l])),
                         T(W["W_2"][l]))
        hidden.append(h)
    e = F.rms_norm(h, (d,), weight=T(W["enc_norm"]), eps=cfg.rms_eps)
    mem = []
    for g in range(cfg.mem_groups):
        # per-layer source: the residual stream after layer g under the final norm
        src = F.rms_norm(hidden[g], (d,), weight=T(W["enc_norm"]), eps=cfg.rms_eps) \
            if getattr(cfg, "mem_source", 0) == 1 else e
        mem.append(torch.stack([_heads(F.linear(src, T(W["W_K"][g])), H),
                                _heads(F.linear(src, T(W["W_V"][g])), H)]))
    if return_kv:
        return e.numpy(), torch.stack(mem).numpy(), torch.stack(kv).numpy()
    return e.numpy(), torch.stack(mem).numpy()


def parallel_decoder(cfg, W, e, mem, window, u=None):
    """Token-parallel decoder pass: every position's first-layer input is u (default e),
    self-attention over the band of the last `window` positions, cross-attention to
    memory positions <= the query position.  Returns the final residual stream
    [B, T, d] (s_t for every t when the recurrence ignores s_{t-1})."""
    d, H = cfg.d, cfg.n_heads
    h = T(e if u is None else u).clone()
    B, P, _ = h.shape
    pos = torch.arange(P)
    i = pos[:, None]
    j = pos[None, :]
    band = (j <= i) & (j > i - window)
    for l in range(cfg.n_layers):
        a = F.rms_norm(h, (d,), weight=T(W["dec_attn_norm"][l]), eps=cfg.rms_eps)
        q, k, v = F.linear(a, T(W["W_qkv"][l])).split(d, dim=-1)
        q, k, v = _heads(q, H), _heads(k, H), _heads(v, H)
        q, k = rope_complex(q, pos, cfg.rope_theta), rope_complex(k, pos, cfg.rope_theta)
        o = F.scaled_dot_product_attention(q, k, v, attn_mask=band)
        h = h + F.linear(_merge_heads(o), T(W["W_O"][l]))
        c = F.rms_norm(h, (d,), weight=T(W["dec_xattn_norm"][l]), eps=cfg.rms_eps)
        qx = _heads(F.linear(c, T(W["W_Qx"][l])), H)
        g = 0 if cfg.mem_groups == 1 else l
        km, vm = T(mem[g, 0, :, :, :P]), T(mem[g, 1, :, :, :P])
        ox = F.scaled_dot_product_attention(qx, km, vm, is_causal=True)
        h = h + F.linear(_merge_heads(ox), T(W["W_Ox"][l]))
        b = F.rms_norm(h, (d,), weight=T(W["dec_ffn_norm"][l]), eps=cfg.rms_eps)
        h = h + F.linear(F.silu(F.linear(b, T(W["W_1"][l]))) * F.linear(b, T(W["W_3"][l])),
                         T(W["W_2"][l]))
    return h.numpy()


def head_logits(cfg, W, s):
    a = F.rms_norm(T(s), (cfg.d,), weight=T(W["head_norm"]), eps=cfg.rms_eps)
    return F.linear(a, T(W["W_o"])).numpy()
