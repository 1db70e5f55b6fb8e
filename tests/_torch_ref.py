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


# ---------------------------------------------------------------------------
# bf16 storage configurations: the same compositions with a rounding to
# bfloat16 at each storage point of the bf16 numerics contract (every matrix
# product input, e, the memory, the window keys/values after RoPE, the
# encoder's q/k/v after RoPE, and the encoder's unnormalised attention
# weights before they multiply the values).  Rounding uses torch's own
# float32 and bfloat16 conversions.

def bf16_rne(x):
    """float64 -> nearest bfloat16 value (ties to even) -> float64, through
    torch's float32 and bfloat16 conversions.  torch converts float64 through
    float32, which rounds twice; a value that the float32 step lands exactly
    on a bfloat16 tie is therefore moved one float32 ulp back towards itself
    first (the float32 step only carried it onto the tie), which makes the
    result the single rounding of x."""
    x = torch.as_tensor(x, dtype=D)
    f = x.to(torch.float32)
    back = f.to(D)
    tie = (f.view(torch.int32) & 0xFFFF) == 0x8000
    fix = tie & (back != x)
    toward = torch.where(x > back, torch.full_like(f, math.inf), torch.full_like(f, -math.inf))
    f = torch.where(fix, torch.nextafter(f, toward), f)
    return f.to(torch.bfloat16).to(D)


def encoder_bf16(cfg, W, tokens):
    """e [B,T,d] and memory [G,2,B,H,T,hd] of a bf16-storage config."""
    R = bf16_rne
    d, H, hd = cfg.d, cfg.n_heads, cfg.head_dim
    tok = torch.as_tensor(tokens, dtype=torch.long)
    B, P = tok.shape
    pos = torch.arange(P)
    causal = torch.ones(P, P, dtype=torch.bool).tril()
    h = F.embedding(tok, T(W["tok_emb"]))
    hidden = []
    for l in range(cfg.n_layers):
        a = R(F.rms_norm(h, (d,), weight=T(W["enc_attn_norm"][l]), eps=cfg.rms_eps))
        q, k, v = F.linear(a, T(W["W_qkv"][l])).split(d, dim=-1)
        q, k, v = _heads(q, H), _heads(k, H), R(_heads(v, H))
        q, k = R(rope_complex(q, pos, cfg.rope_theta)), R(rope_complex(k, pos, cfg.rope_theta))
        s = torch.matmul(q, k.transpose(-1, -2)).div(math.sqrt(hd)).masked_fill(~causal, -math.inf)
        w = torch.exp(s - s.amax(dim=-1, keepdim=True))
        o = torch.matmul(R(w), v) / w.sum(dim=-1, keepdim=True)
        h = h + F.linear(R(_merge_heads(o)), T(W["W_O"][l]))
        b = R(F.rms_norm(h, (d,), weight=T(W["enc_ffn_norm"][l]), eps=cfg.rms_eps))
        h = h + F.linear(R(F.silu(F.linear(b, T(W["W_1"][l]))) * F.linear(b, T(W["W_3"][l]))),
                         T(W["W_2"][l]))
        hidden.append(h)
    e = R(F.rms_norm(h, (d,), weight=T(W["enc_norm"]), eps=cfg.rms_eps))
    mem = []
    for g in range(cfg.mem_groups):
        src = R(F.rms_norm(hidden[g], (d,), weight=T(W["enc_norm"]), eps=cfg.rms_eps)) \
            if getattr(cfg, "mem_source", 0) == 1 else e
        mem.append(torch.stack([_heads(R(F.linear(src, T(W["W_K"][g]))), H),
                                _heads(R(F.linear(src, T(W["W_V"][g]))), H)]))
    return e.numpy(), torch.stack(mem).numpy()


def decoder_bf16(cfg, W, e, mem, n):
    """n recurrent steps of a bf16-storage config from H_0, with the window
    cache as a list per layer: the current entry is appended, attention runs
    over the last `window` entries, and the last window - 1 are kept.
    Returns s_n [B,d], the logits of every step [n][B,V] and the caches
    (per layer a list of (k, v) [B,H,hd], oldest first)."""
    R = bf16_rne
    d, H, hd, Wn = cfg.d, cfg.n_heads, cfg.head_dim, cfg.window
    e = T(e)
    B = e.shape[0]
    s = T(W["s_star"]).expand(B, d).clone()
    caches = [[] for _ in range(cfg.n_layers)]
    logits = []
    for p in range(n):
        et = e[:, p]
        if cfg.gate_mode == 1:
            z = torch.zeros_like(s)
        else:
            z = torch.sigmoid(F.linear(R(torch.cat([et, s], dim=-1)), T(W["W_g"]), T(W["b_g"])))
        h = z * s + (1.0 - z) * et
        for l in range(cfg.n_layers):
            a = R(F.rms_norm(h, (d,), weight=T(W["dec_attn_norm"][l]), eps=cfg.rms_eps))
            q, k, v = F.linear(a, T(W["W_qkv"][l])).split(d, dim=-1)
            q = rope_complex(q.reshape(B, H, 1, hd), [p], cfg.rope_theta)
            k = R(rope_complex(k.reshape(B, H, 1, hd), [p], cfg.rope_theta))
            v = R(v.reshape(B, H, 1, hd))
            entries = (caches[l] + [(k, v)])[-Wn:]
            o = F.scaled_dot_product_attention(q, torch.cat([x for x, _ in entries], dim=2),
                                               torch.cat([x for _, x in entries], dim=2))
            caches[l] = entries[1:] if len(entries) == Wn else entries
            h = h + F.linear(R(o.reshape(B, d)), T(W["W_O"][l]))
            c = R(F.rms_norm(h, (d,), weight=T(W["dec_xattn_norm"][l]), eps=cfg.rms_eps))
            qx = F.linear(c, T(W["W_Qx"][l])).reshape(B, H, 1, hd)
            g = 0 if cfg.mem_groups == 1 else l
            ox = F.scaled_dot_product_attention(qx, T(mem[g, 0, :, :, :p + 1]), T(mem[g, 1, :, :, :p + 1]))
            h = h + F.linear(R(ox.reshape(B, d)), T(W["W_Ox"][l]))
            b = R(F.rms_norm(h, (d,), weight=T(W["dec_ffn_norm"][l]), eps=cfg.rms_eps))
            h = h + F.linear(R(F.silu(F.linear(b, T(W["W_1"][l]))) * F.linear(b, T(W["W_3"][l]))),
                             T(W["W_2"][l]))
        s = h
        a = R(F.rms_norm(s, (d,), weight=T(W["head_norm"]), eps=cfg.rms_eps))
        logits.append(F.linear(a, T(W["W_o"])).numpy())
    caches = [[(k[:, :, 0].numpy(), v[:, :, 0].numpy()) for k, v in cl] for cl in caches]
    return s.numpy(), logits, caches
