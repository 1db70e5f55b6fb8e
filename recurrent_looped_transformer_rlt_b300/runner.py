"""Convenience driver over the C ABI: allocates e, memory, state and workspace
with torch and issues rlt_encode / rlt_decode_steps.  Marshalling only."""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import (Model, State, rlt_decode_steps, rlt_encode, rlt_state_init, rlt_status)


@dataclass
class Buffers:
    e: torch.Tensor
    mem: torch.Tensor
    ws: torch.Tensor
    B: int
    T: int


def alloc_buffers(model: Model, B: int, T: int, stream=None) -> Buffers:
    c = model.cfg
    e = torch.empty(B, T, c.d, dtype=model.dtype, device="cuda")
    mem = torch.empty(c.mem_groups, 2, B, c.n_heads, T, c.head_dim, dtype=model.dtype, device="cuda")
    ws = model.workspace(B, T, stream)
    return Buffers(e, mem, ws, B, T)


def encode(model: Model, tokens: torch.Tensor, buf: Buffers, stream=None):
    B, T = tokens.shape
    rlt_encode(model.handle, tokens, B, T, buf.e, buf.mem, buf.ws, buf.ws.numel(), stream)


def new_state(model: Model, B: int, stream=None) -> State:
    st = State(model, B)
    rlt_state_init(model.handle, st.c, stream)
    return st


@dataclass
class StepOutputs:
    logp: torch.Tensor
    logp_full: torch.Tensor
    argmax: torch.Tensor
    logits: Optional[torch.Tensor]


def decode(model: Model, st: State, buf: Buffers, n: int, actions: Optional[torch.Tensor] = None,
           temperature: float = 1.0, top_k: int = 0, emit_steps: Sequence[int] = (),
           out: Optional[StepOutputs] = None, stream=None) -> StepOutputs:
    B = st.c.batch
    if out is None:
        out = StepOutputs(torch.empty(B, n, device="cuda"), torch.empty(B, n, device="cuda"),
                          torch.empty(B, n, dtype=torch.int32, device="cuda"),
                          torch.empty(len(emit_steps), B, model.cfg.vocab, device="cuda") if emit_steps else None)
    if actions is not None:
        actions = actions.contiguous()
        assert actions.shape == (B, n) and actions.dtype == torch.int32
    rlt_decode_steps(model.handle, st.c, buf.e, buf.mem, buf.T, n, actions, temperature, top_k, out.logp,
                     out.logp_full, out.argmax, list(emit_steps), out.logits, buf.ws, buf.ws.numel(), stream)
    return out


def status(buf: Buffers, stream=None) -> int:
    return rlt_status(buf.ws, stream)
