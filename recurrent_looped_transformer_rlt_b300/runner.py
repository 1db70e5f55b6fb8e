"""Convenience driver over the C ABI: allocates e, memory, state and workspace
with torch and issues rlt_encode / rlt_decode_steps.  Marshalling only."""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import (GRAD_FIELDS, RLT_BPTT_CORE_MEMGRAD, RLT_BPTT_NO_GRAPHS, RLT_DETACH_CACHE, RLT_DETACH_MEMORY,
               Model, State, rlt_bptt, rlt_bptt_workspace_size, rlt_decode_steps, rlt_encode, rlt_grads,
               rlt_state_init, rlt_status, rlt_workspace_init)


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


@dataclass
class BpttResult:
    loss: torch.Tensor           # [1] f32
    logp: torch.Tensor           # [B][n] f32
    grads: dict                  # name -> f32 tensor of the parameter's shape
    d_e: Optional[torch.Tensor]  # [B][T_mem][d] f32
    d_mem: Optional[torch.Tensor]


def bptt(model: Model, buf: Buffers, actions: torch.Tensor, temperature: float = 1.0, top_k: int = 0,
         detach_s_every: int = 0, detach_cache: bool = False, detach_memory: bool = False,
         want_inputs: bool = True, ws: Optional[torch.Tensor] = None, graphs: bool = True,
         core_memgrad: bool = False, stream=None) -> BpttResult:
    """Loss and gradients of the teacher-forced sequence (rlt_bptt) over the
    first n = actions.shape[1] positions of buf's encoder output and memory.
    core_memgrad: the memory gradient on CUDA cores (RLT_BPTT_CORE_MEMGRAD)."""
    B, n = actions.shape
    actions = actions.contiguous()
    assert actions.dtype == torch.int32 and B == buf.B
    t = model.t
    grads = {k: torch.empty_like(t[k], dtype=torch.float32) for k in GRAD_FIELDS}
    cg = rlt_grads(*[grads[k].data_ptr() for k in GRAD_FIELDS])
    d_e = torch.empty(buf.e.shape, dtype=torch.float32, device="cuda") if want_inputs else None
    d_mem = torch.empty(buf.mem.shape, dtype=torch.float32, device="cuda") if want_inputs else None
    if ws is None:
        nb = rlt_bptt_workspace_size(model.handle, B, n)
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        rlt_workspace_init(ws, nb, stream)
    loss = torch.empty(1, device="cuda")
    logp = torch.empty(B, n, device="cuda")
    flags = (RLT_DETACH_CACHE if detach_cache else 0) | (RLT_DETACH_MEMORY if detach_memory else 0)
    flags |= 0 if graphs else RLT_BPTT_NO_GRAPHS
    flags |= RLT_BPTT_CORE_MEMGRAD if core_memgrad else 0
    rlt_bptt(model.handle, buf.e, buf.mem, buf.T, B, n, actions, temperature, top_k, detach_s_every, flags, loss,
             logp, cg, d_e, d_mem, ws, ws.numel(), stream)
    return BpttResult(loss, logp, grads, d_e, d_mem)
