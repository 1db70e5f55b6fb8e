"""Gradients of the RLT decoder recurrence (full and truncated BPTT), float64
on the CPU.

TEST INFRASTRUCTURE, like rlt_oracle.py: only the test suite may import it;
the product library never calls it.  It shares no code with the CUDA path.

What it computes.  The teacher-forced sequence loss of the recurrent decoder,

    L = - sum over steps t and sequences b of lp_t(a_{b,t}),

where step t consumes the token at position t-1 (merge with e_t, the decoder
layers with their window caches and cross-attention to the memory of
positions 1..t) and lp_t is the tempered (top-k) log-probability of the action
under the head of s_t - the same transition and scoring as rlt_oracle - and
its gradients with respect to the decoder's parameters, s_*, the encoder
output e and the memory M, through every path the state has:

* "Recurrent Looped Transformer: A New Architecture for Infinite Context
  Reasoning", "Training and Serving Considerations": training uses full
  backpropagation through time;
* "Princeton Researcher Proposes Recurrent Looped Transformer ...", training
  paragraph: the state-to-state Jacobian has cross terms through the decoder's
  keys and values, so detaching only s_t still leaves gradient paths through
  the window cache, and a truncated scheme has to name every tensor it
  detaches;
* "Understanding and Applying the Recurrent Looped Transformer Architecture",
  "Current-Policy Reinforcement Learning Replay": full gradients pass through
  the recurrent outputs, the decoder key-value entries and the encoder
  memory; detaching any of them is an approximation.

With model_gradients the encoder is part of the graph too (encode builds e
and M from the tokens, as rlt_oracle.encode does): gradients reach the token
embedding, the encoder norms and the memory projections, and each tied
attention / FFN matrix collects its encoder and its decoder use - the
full-sequence next-token training of the Princeton page's training paragraph.

Named detach points (each off by default = full BPTT):
  detach_s_every = k > 0: s_t is detached after every k-th step;
  detach_cache: the window's keys and values enter later steps as constants
      (the current step's own entry keeps its gradient);
  detach_memory: the memory enters every step as a constant.

The forward is written with torch float64 tensors so that the library's
automatic differentiation gives the gradients; it follows rlt_oracle's
decode_step term by term for float32-storage configurations (no bf16 rounding
points: rounding has no derivative) and is pinned to it and to central finite
differences in tests/test_bptt_pins.py.
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, Optional

import numpy as np
import torch

from oracle.rlt_oracle import Cfg

F = torch.float64

DECODER_PARAMS = ("W_g", "b_g", "W_qkv", "W_O", "W_Qx", "W_Ox", "W_1", "W_3", "W_2", "dec_attn_norm",
                  "dec_xattn_norm", "dec_ffn_norm", "head_norm", "W_o", "s_star")


def _rmsnorm(x, g, eps):
    return x / torch.sqrt(torch.mean(x * x, dim=-1, keepdim=True) + eps) * g


def _rope(x, p: int, theta: float):
    """Rotate-half RoPE of x [..., hd] at position p."""
    hd = x.shape[-1]
    i = torch.arange(hd // 2, dtype=F)
    ang = p * theta ** (-2.0 * i / hd)
    c, s = torch.cos(ang), torch.sin(ang)
    x1, x2 = x[..., : hd // 2], x[..., hd // 2:]
    return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1)


def _attend(q, ks, vs, hd):
    """q [B, H, hd] over entries ks, vs [B, H, n, hd]."""
    s = torch.einsum("bhd,bhnd->bhn", q, ks) / math.sqrt(hd)
    p = torch.softmax(s, dim=-1)
    return torch.einsum("bhn,bhnd->bhd", p, vs)


def _lp(logits, actions, temperature, top_k):
    """Tempered (top-k) log-probabilities of actions [B] (0 where action < 0)."""
    x = logits / temperature
    V = x.shape[-1]
    if 0 < top_k < V:
        ids = torch.arange(V)
        mask = torch.zeros_like(x, dtype=torch.bool)
        for b in range(x.shape[0]):
            order = np.lexsort((ids.numpy(), -x[b].detach().numpy()))  # value desc, id asc
            mask[b, torch.as_tensor(order[:top_k])] = True
        x = torch.where(mask, x, torch.full_like(x, -math.inf))
    lse = torch.logsumexp(x, dim=-1)
    a = torch.as_tensor(np.maximum(actions, 0), dtype=torch.long)
    lp = x.gather(1, a[:, None])[:, 0] - lse
    return torch.where(torch.as_tensor(actions >= 0), lp, torch.zeros_like(lp))


def sequence_loss(cfg: Cfg, P: Dict[str, torch.Tensor], e, mem, actions, n: Optional[int] = None,
                  temperature: float = 1.0, top_k: int = 0, detach_s_every: int = 0, detach_cache: bool = False,
                  detach_memory: bool = False, per_step: bool = False):
    """L over the first n steps (all of actions' columns by default).

    P: float64 tensors of the decoder parameters (DECODER_PARAMS); e [B, T, d],
    mem [G, 2, B, H, T, hd] float64 tensors; actions int [B, >= n].  With
    per_step, returns the list of step losses instead of their sum.
    """
    if cfg.bf16:
        raise ValueError("gradients are defined for float32-storage configurations")
    B = e.shape[0]
    d, H, hd, L = cfg.d, cfg.n_heads, cfg.head_dim, cfg.n_layers
    n = actions.shape[1] if n is None else n
    keep = cfg.window - 1
    M = mem.detach() if detach_memory else mem
    s = P["s_star"].expand(B, d)
    cache = [[] for _ in range(L)]
    losses = []
    for t in range(1, n + 1):
        p = t - 1
        e_t = e[:, p]
        if cfg.gate_mode == 1:
            z = torch.zeros_like(s)
        else:
            z = torch.sigmoid(torch.cat([e_t, s], dim=-1) @ P["W_g"].T + P["b_g"])
        h = z * s + (1.0 - z) * e_t
        for l in range(L):
            a = _rmsnorm(h, P["dec_attn_norm"][l], cfg.rms_eps)
            qkv = a @ P["W_qkv"][l].T
            q = _rope(qkv[:, :d].reshape(B, H, hd), p, cfg.rope_theta)
            k = _rope(qkv[:, d:2 * d].reshape(B, H, hd), p, cfg.rope_theta)
            v = qkv[:, 2 * d:].reshape(B, H, hd)
            entries = cache[l] + [(k, v)]
            ks = torch.stack([x[0] for x in entries], dim=2)
            vs = torch.stack([x[1] for x in entries], dim=2)
            h = h + _attend(q, ks, vs, hd).reshape(B, d) @ P["W_O"][l].T
            kept = entries[max(0, len(entries) - keep):] if keep > 0 else []
            cache[l] = [(kk.detach(), vv.detach()) for kk, vv in kept] if detach_cache else kept
            c = _rmsnorm(h, P["dec_xattn_norm"][l], cfg.rms_eps)
            qx = (c @ P["W_Qx"][l].T).reshape(B, H, hd)
            g = cfg.group_of(l)
            ox = _attend(qx, M[g, 0, :, :, :t], M[g, 1, :, :, :t], hd).reshape(B, d)
            h = h + ox @ P["W_Ox"][l].T
            bb = _rmsnorm(h, P["dec_ffn_norm"][l], cfg.rms_eps)
            gate = bb @ P["W_1"][l].T
            h = h + (gate * torch.sigmoid(gate) * (bb @ P["W_3"][l].T)) @ P["W_2"][l].T
        s = h
        logits = _rmsnorm(s, P["head_norm"], cfg.rms_eps) @ P["W_o"].T
        losses.append(-torch.sum(_lp(logits, np.asarray(actions)[:, p], temperature, top_k)))
        if detach_s_every > 0 and t % detach_s_every == 0:
            s = s.detach()
    return losses if per_step else torch.stack(losses).sum()


ENCODER_PARAMS = ("tok_emb", "enc_attn_norm", "enc_ffn_norm", "enc_norm", "W_K", "W_V")


def encode(cfg: Cfg, P: Dict[str, torch.Tensor], tokens):
    """The causal encoder and memory projection of rlt_oracle.encode in float64
    torch (float32-storage configurations): e [B, T, d] and mem
    [G, 2, B, H, T, hd] as functions of the encoder parameters, which include
    the attention and FFN weights it shares with the decoder (W_qkv, W_O, W_1,
    W_3, W_2)."""
    if cfg.bf16:
        raise ValueError("gradients are defined for float32-storage configurations")
    tok = torch.as_tensor(np.asarray(tokens), dtype=torch.long)
    B, T = tok.shape
    d, H, hd = cfg.d, cfg.n_heads, cfg.head_dim
    causal = torch.tril(torch.ones(T, T, dtype=torch.bool))
    h = P["tok_emb"][tok]
    sources = []
    for l in range(cfg.n_layers):
        a = _rmsnorm(h, P["enc_attn_norm"][l], cfg.rms_eps)
        qkv = a @ P["W_qkv"][l].T
        q = qkv[..., :d].reshape(B, T, H, hd).transpose(1, 2)
        k = qkv[..., d:2 * d].reshape(B, T, H, hd).transpose(1, 2)
        v = qkv[..., 2 * d:].reshape(B, T, H, hd).transpose(1, 2)
        q = torch.stack([_rope(q[:, :, p], p, cfg.rope_theta) for p in range(T)], dim=2)
        k = torch.stack([_rope(k[:, :, p], p, cfg.rope_theta) for p in range(T)], dim=2)
        sc = (q @ k.transpose(-1, -2)) / math.sqrt(hd)
        sc = torch.where(causal, sc, torch.full_like(sc, -math.inf))
        o = (torch.softmax(sc, dim=-1) @ v).transpose(1, 2).reshape(B, T, d)
        h = h + o @ P["W_O"][l].T
        bb = _rmsnorm(h, P["enc_ffn_norm"][l], cfg.rms_eps)
        gate = bb @ P["W_1"][l].T
        h = h + (gate * torch.sigmoid(gate) * (bb @ P["W_3"][l].T)) @ P["W_2"][l].T
        if cfg.mem_source == 1:
            sources.append(_rmsnorm(h, P["enc_norm"], cfg.rms_eps))
    e = _rmsnorm(h, P["enc_norm"], cfg.rms_eps)
    if cfg.mem_source != 1:
        sources = [e] * cfg.mem_groups
    mem = []
    for g in range(cfg.mem_groups):
        kk = (sources[g] @ P["W_K"][g].T).reshape(B, T, H, hd).transpose(1, 2)
        vv = (sources[g] @ P["W_V"][g].T).reshape(B, T, H, hd).transpose(1, 2)
        mem.append(torch.stack([kk, vv]))
    return e, torch.stack(mem)


def model_gradients(cfg: Cfg, W, tokens, actions, wrt: Iterable[str] = DECODER_PARAMS + ENCODER_PARAMS, **kw):
    """(loss, {name: gradient}) of the whole model's sequence loss: the encoder
    builds e and M from the tokens, the recurrent decoder consumes them; tied
    weights receive the gradients of both uses."""
    P = {k: torch.tensor(np.asarray(W[k], np.float64), dtype=F, requires_grad=True)
         for k in DECODER_PARAMS + ENCODER_PARAMS}
    e, mem = encode(cfg, P, tokens)
    loss = sequence_loss(cfg, P, e, mem, actions, **kw)
    names = list(wrt)
    grads = torch.autograd.grad(loss, [P[k] for k in names], allow_unused=True)
    return float(loss.detach()), {k: (np.zeros(tuple(P[k].shape)) if g is None else g.detach().numpy())
                                  for k, g in zip(names, grads)}


def leaves(W: Dict[str, np.ndarray], e, mem):
    """Float64 leaf tensors (requires_grad) of the decoder parameters, e and mem."""
    P = {k: torch.tensor(np.asarray(W[k], np.float64), dtype=F, requires_grad=True) for k in DECODER_PARAMS}
    et = torch.tensor(np.asarray(e, np.float64), dtype=F, requires_grad=True)
    mt = torch.tensor(np.asarray(mem, np.float64), dtype=F, requires_grad=True)
    return P, et, mt


def gradients(cfg: Cfg, W, e, mem, actions, wrt: Iterable[str] = DECODER_PARAMS + ("e", "mem"), **kw):
    """(loss, {name: gradient as float64 numpy}) of sequence_loss."""
    P, et, mt = leaves(W, e, mem)
    loss = sequence_loss(cfg, P, et, mt, actions, **kw)
    names = list(wrt)
    tensors = [et if k == "e" else mt if k == "mem" else P[k] for k in names]
    grads = torch.autograd.grad(loss, tensors, allow_unused=True)
    out = {}
    for k, gt, x in zip(names, grads, tensors):
        out[k] = np.zeros(tuple(x.shape)) if gt is None else gt.detach().numpy()
    return float(loss.detach()), out
