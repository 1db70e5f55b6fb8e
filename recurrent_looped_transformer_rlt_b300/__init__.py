"""Python binding of librlt.so, the B300 implementation of the RLT hot path.

Argument marshalling only: every computation runs in the library's CUDA
kernels.  The functions keep the C names (rlt_model_create, rlt_state_init,
rlt_encode, rlt_decode_steps, ...) and take torch tensors or raw pointers.
PyTorch provides the device memory and the stream.  There is no CPU path:
if the library is missing, importing this package raises.

Helpers ``Model`` and ``State`` hold the torch tensors behind the C structs
so that their pointers stay valid.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librlt.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"librlt.so not built at {LIB_PATH}: run "
                      "`python recurrent_looped_transformer_rlt_b300/build.py` (needs nvcc)")

_lib = ctypes.CDLL(LIB_PATH)

RLT_OK, RLT_EINVAL, RLT_ESTALE, RLT_ERANGE, RLT_ECUDA = 0, -1, -2, -3, -4
RLT_ETIMEOUT, RLT_EBOUNDS, RLT_EWORKSPACE, RLT_EUNSUPPORTED = -5, -6, -7, -8
RLT_F32, RLT_BF16 = 0, 1
RLT_GATE_LEARNED, RLT_GATE_DISCARD_S = 0, 1
RLT_MEM_FINAL, RLT_MEM_PER_LAYER = 0, 1

_p = ctypes.c_void_p
_i32 = ctypes.c_int32


class rlt_config(ctypes.Structure):
    _fields_ = [("d_model", _i32), ("n_layers", _i32), ("n_heads", _i32), ("head_dim", _i32),
                ("d_ffn", _i32), ("window", _i32), ("mem_groups", _i32), ("vocab", _i32),
                ("dtype", _i32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("gate_mode", _i32), ("mem_source", _i32)]


WEIGHT_FIELDS = ["tok_emb", "s_star", "W_g", "b_g", "W_qkv", "W_O", "W_1", "W_3", "W_2", "W_Qx",
                 "W_Ox", "W_K", "W_V", "W_o", "enc_attn_norm", "enc_ffn_norm", "enc_norm",
                 "dec_attn_norm", "dec_xattn_norm", "dec_ffn_norm", "head_norm"]


class rlt_weights(ctypes.Structure):
    _fields_ = [(n, _p) for n in WEIGHT_FIELDS]


class rlt_state(ctypes.Structure):
    _fields_ = [("batch", _i32), ("pos", _i32), ("version", ctypes.c_uint64), ("s", _p),
                ("ring_k", _p), ("ring_v", _p)]


GRAD_FIELDS = ["W_g", "b_g", "W_qkv", "W_O", "W_Qx", "W_Ox", "W_1", "W_3", "W_2", "W_o", "dec_attn_norm",
               "dec_xattn_norm", "dec_ffn_norm", "head_norm", "s_star"]
RLT_DETACH_CACHE, RLT_DETACH_MEMORY, RLT_BPTT_NO_GRAPHS, RLT_BPTT_CORE_MEMGRAD = 1, 2, 4, 8


class rlt_grads(ctypes.Structure):
    _fields_ = [(n, _p) for n in GRAD_FIELDS]


def _sig(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


_model_create = _sig("rlt_model_create", ctypes.c_int,
                     [ctypes.POINTER(rlt_config), ctypes.POINTER(rlt_weights), ctypes.c_uint64,
                      ctypes.POINTER(_p)])
_model_set_version = _sig("rlt_model_set_version", ctypes.c_int, [_p, ctypes.c_uint64])
_model_destroy = _sig("rlt_model_destroy", None, [_p])
_workspace_size = _sig("rlt_workspace_size", ctypes.c_int, [_p, _i32, _i32, ctypes.POINTER(ctypes.c_size_t)])
_workspace_init = _sig("rlt_workspace_init", ctypes.c_int, [_p, ctypes.c_size_t, _p])
_state_sizes = _sig("rlt_state_sizes", ctypes.c_int,
                    [_p, _i32, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)])
_state_init = _sig("rlt_state_init", ctypes.c_int, [_p, ctypes.POINTER(rlt_state), _p])
_encode = _sig("rlt_encode", ctypes.c_int, [_p, _p, _i32, _i32, _p, _p, _p, ctypes.c_size_t, _p])
_decode_steps = _sig("rlt_decode_steps", ctypes.c_int,
                     [_p, ctypes.POINTER(rlt_state), _p, _p, _i32, _i32, _p, ctypes.c_float, _i32, _p, _p,
                      _p, ctypes.POINTER(_i32), _i32, _p, _p, ctypes.c_size_t, _p])
_status = _sig("rlt_status", ctypes.c_int, [_p, _p])
_cross_attention = _sig("rlt_cross_attention", ctypes.c_int, [_p, _p, _p, _p, _i32, _i32, _i32, _p, _p,
                                                              ctypes.c_size_t, _p])
_cross_attention_noalloc = _sig("rlt_cross_attention_noalloc", ctypes.c_int,
                                [_p, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _p, _p])
_cross_attention_noalloc_status = _sig("rlt_cross_attention_noalloc_status", ctypes.c_int, [_p])
_linear = _sig("rlt_linear", ctypes.c_int, [_p, _p, _i32, _i32, _i32, _p, _p, _i32, _i32, _p, _i32, _p,
                                          ctypes.c_size_t, _p])
_encode_kv = _sig("rlt_encode_kv", ctypes.c_int, [_p, _p, _i32, _i32, _i32, _p, _p, _p, _p, ctypes.c_size_t, _p])
_generate = _sig("rlt_generate", ctypes.c_int,
                 [_p, ctypes.POINTER(rlt_state), _p, _p, _p, _i32, _i32, ctypes.c_uint64, ctypes.c_float, _i32, _p,
                  _p, _p, ctypes.c_size_t, _p])
_snapshot_size = _sig("rlt_snapshot_size", ctypes.c_int, [_p, _i32, _i32, _i32, ctypes.POINTER(ctypes.c_size_t)])
_snapshot_save = _sig("rlt_snapshot_save", ctypes.c_int,
                      [_p, ctypes.POINTER(rlt_state), _p, _p, _p, _i32, _p, ctypes.c_size_t, _p])
_snapshot_restore = _sig("rlt_snapshot_restore", ctypes.c_int,
                         [_p, _p, ctypes.c_size_t, ctypes.POINTER(rlt_state), _p, _p, _p, _i32, _p])
_bptt_workspace_size = _sig("rlt_bptt_workspace_size", ctypes.c_int,
                            [_p, _i32, _i32, ctypes.POINTER(ctypes.c_size_t)])
_bptt = _sig("rlt_bptt", ctypes.c_int,
             [_p, _p, _p, _i32, _i32, _i32, _p, ctypes.c_float, _i32, _i32, _i32, _p, _p,
              ctypes.POINTER(rlt_grads), _p, _p, _p, ctypes.c_size_t, _p])
_set_decode_path = _sig("rlt_set_decode_path", ctypes.c_int, [_p, _i32, _i32])
_fused_plan = _sig("rlt_fused_plan", ctypes.c_int, [_p, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32),
                                                   ctypes.POINTER(_i32), ctypes.POINTER(_i32)])
_timer_arm = _sig("rlt_timer_arm", ctypes.c_int, [_p, _i32, _i32])
_timer_read = _sig("rlt_timer_read", ctypes.c_int, [_p, ctypes.POINTER(ctypes.c_float), _i32, ctypes.POINTER(_i32)])
_strerror = _sig("rlt_strerror", ctypes.c_char_p, [ctypes.c_int])
_launch_count = _sig("rlt_launch_count", ctypes.c_uint64, [])
_abi_version = _sig("rlt_abi_version", ctypes.c_int, [])
_debug_withhold_copy = _sig("rlt_debug_withhold_copy", ctypes.c_int, [_p, _i32, ctypes.c_int64])

EXPORTED = ["rlt_model_create", "rlt_model_set_version", "rlt_model_destroy", "rlt_workspace_size",
            "rlt_workspace_init", "rlt_state_sizes", "rlt_state_init", "rlt_encode", "rlt_decode_steps",
            "rlt_status", "rlt_strerror", "rlt_launch_count", "rlt_abi_version", "rlt_timer_arm",
            "rlt_timer_read", "rlt_cross_attention", "rlt_cross_attention_noalloc", "rlt_linear",
            "rlt_snapshot_size", "rlt_snapshot_save", "rlt_snapshot_restore", "rlt_encode_kv", "rlt_generate",
            "rlt_bptt_workspace_size", "rlt_bptt", "rlt_set_decode_path", "rlt_fused_plan",
            "rlt_debug_withhold_copy", "rlt_cross_attention_noalloc_status"]
RLT_DECODE_AUTO, RLT_DECODE_GRAPH, RLT_DECODE_FUSED = 0, 1, 2
DECODE_PATHS = {"auto": RLT_DECODE_AUTO, "graph": RLT_DECODE_GRAPH, "fused": RLT_DECODE_FUSED}
RLT_TIMER_CLASSES = {"off": 0, "xattn": 1, "swa": 2, "gemm": 3, "head": 4, "step": 5}
RLT_KERNEL_XATTN, RLT_KERNEL_GEMM, RLT_KERNEL_NORM_PROJ = 1, 2, 3


class RLTError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {rlt_strerror(code)} ({code})")
        self.code = code


def _check(rc: int, where: str):
    if rc != RLT_OK:
        raise RLTError(rc, where)


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def rlt_strerror(code: int) -> str:
    return _strerror(code).decode()


def rlt_launch_count() -> int:
    return int(_launch_count())


def rlt_abi_version() -> int:
    return int(_abi_version())


# ---------------------------------------------------------------------------
# thin wrappers with the C names

def rlt_model_create(cfg: rlt_config, weights: rlt_weights, version: int = 0) -> int:
    h = _p()
    _check(_model_create(ctypes.byref(cfg), ctypes.byref(weights), version, ctypes.byref(h)), "rlt_model_create")
    return h.value


def rlt_model_set_version(model: int, version: int):
    _check(_model_set_version(model, version), "rlt_model_set_version")


def rlt_model_destroy(model: int):
    _model_destroy(model)


def rlt_workspace_size(model: int, B: int, T_max: int) -> int:
    n = ctypes.c_size_t()
    _check(_workspace_size(model, B, T_max, ctypes.byref(n)), "rlt_workspace_size")
    return n.value


def rlt_workspace_init(ws, nbytes: int, stream=None):
    _check(_workspace_init(_ptr(ws), nbytes, _stream_ptr(stream)), "rlt_workspace_init")


def rlt_state_sizes(model: int, B: int):
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    _check(_state_sizes(model, B, ctypes.byref(a), ctypes.byref(b)), "rlt_state_sizes")
    return a.value, b.value


def rlt_state_init(model: int, st: rlt_state, stream=None):
    _check(_state_init(model, ctypes.byref(st), _stream_ptr(stream)), "rlt_state_init")


def rlt_encode(model: int, tokens, B: int, T: int, e, mem, ws, ws_bytes: int, stream=None):
    _check(_encode(model, _ptr(tokens), B, T, _ptr(e), _ptr(mem), _ptr(ws), ws_bytes, _stream_ptr(stream)),
           "rlt_encode")


def rlt_decode_steps(model: int, st: rlt_state, e, mem, T_mem: int, n: int, actions=None,
                     temperature: float = 1.0, top_k: int = 0, logp=None, logp_full=None, argmax=None,
                     emit_steps: Sequence[int] = (), logits=None, ws=None, ws_bytes: int = 0, stream=None,
                     check: bool = True) -> int:
    ne = len(emit_steps)
    arr = (_i32 * max(ne, 1))(*emit_steps)
    rc = _decode_steps(model, ctypes.byref(st), _ptr(e), _ptr(mem), T_mem, n, _ptr(actions), float(temperature),
                       top_k, _ptr(logp), _ptr(logp_full), _ptr(argmax), arr if ne else None, ne, _ptr(logits),
                       _ptr(ws), ws_bytes, _stream_ptr(stream))
    if check:
        _check(rc, "rlt_decode_steps")
    return rc


def rlt_encode_kv(model: int, tokens, B: int, T: int, T_max: int, e, mem, enc_kv, ws, ws_bytes: int, stream=None):
    _check(_encode_kv(model, _ptr(tokens), B, T, T_max, _ptr(e), _ptr(mem), _ptr(enc_kv), _ptr(ws), ws_bytes,
                      _stream_ptr(stream)), "rlt_encode_kv")


def rlt_generate(model: int, st: rlt_state, e, mem, enc_kv, T_max: int, n: int, seed: int, temperature: float,
                 top_k: int, tokens, logp, ws, ws_bytes: int, stream=None, check: bool = True) -> int:
    rc = _generate(model, ctypes.byref(st), _ptr(e), _ptr(mem), _ptr(enc_kv), T_max, n, seed, temperature, top_k,
                   _ptr(tokens), _ptr(logp), _ptr(ws), ws_bytes, _stream_ptr(stream))
    if check:
        _check(rc, "rlt_generate")
    return rc


def rlt_snapshot_size(model: int, B: int, pos: int, with_enc_kv: bool = False) -> int:
    n = ctypes.c_size_t()
    _check(_snapshot_size(model, B, pos, int(bool(with_enc_kv)), ctypes.byref(n)), "rlt_snapshot_size")
    return n.value


def rlt_snapshot_save(model: int, st: rlt_state, e, mem, T_mem: int, snap, snap_bytes: int, stream=None,
                      check: bool = True, enc_kv=None) -> int:
    rc = _snapshot_save(model, ctypes.byref(st), _ptr(e), _ptr(mem), _ptr(enc_kv), T_mem, _ptr(snap), snap_bytes,
                        _stream_ptr(stream))
    if check:
        _check(rc, "rlt_snapshot_save")
    return rc


def rlt_snapshot_restore(model: int, snap, snap_bytes: int, st: rlt_state, e, mem, T_mem: int, stream=None,
                         check: bool = True, enc_kv=None) -> int:
    rc = _snapshot_restore(model, _ptr(snap), snap_bytes, ctypes.byref(st), _ptr(e), _ptr(mem), _ptr(enc_kv), T_mem,
                           _stream_ptr(stream))
    if check:
        _check(rc, "rlt_snapshot_restore")
    return rc


def rlt_status(ws, stream=None) -> int:
    return int(_status(_ptr(ws), _stream_ptr(stream)))


def rlt_cross_attention(model: int, q, mem_k, mem_v, B: int, T_mem: int, t: int, out, ws, ws_bytes: int,
                        stream=None):
    _check(_cross_attention(model, _ptr(q), _ptr(mem_k), _ptr(mem_v), B, T_mem, t, _ptr(out), _ptr(ws), ws_bytes,
                            _stream_ptr(stream)), "rlt_cross_attention")


def rlt_cross_attention_noalloc(q, mem_k, mem_v, B: int, n_heads: int, head_dim: int, dtype: int, T_mem: int,
                                t: int, out, stream=None, check: bool = True) -> int:
    """Same as rlt_cross_attention without a workspace (fixed scratch inside the library)."""
    rc = _cross_attention_noalloc(_ptr(q), _ptr(mem_k), _ptr(mem_v), B, n_heads, head_dim, dtype, T_mem, t,
                                  _ptr(out), _stream_ptr(stream))
    if check:
        _check(rc, "rlt_cross_attention_noalloc")
    return rc


def rlt_cross_attention_noalloc_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status of
    the allocation-free entry point's built-in array."""
    return int(_cross_attention_noalloc_status(_stream_ptr(stream)))


def rlt_linear(model: int, A, lda: int, M: int, K: int, W, W3, ldw: int, N: int, C, ldc: int, ws, ws_bytes: int,
               stream=None, check: bool = True) -> int:
    rc = _linear(model, _ptr(A), lda, M, K, _ptr(W), _ptr(W3), ldw, N, _ptr(C), ldc, _ptr(ws), ws_bytes,
                 _stream_ptr(stream))
    if check:
        _check(rc, "rlt_linear")
    return rc


def rlt_bptt_workspace_size(model: int, B: int, n: int) -> int:
    nb = ctypes.c_size_t()
    _check(_bptt_workspace_size(model, B, n, ctypes.byref(nb)), "rlt_bptt_workspace_size")
    return nb.value


def rlt_bptt(model: int, e, mem, T_mem: int, B: int, n: int, actions, temperature: float, top_k: int,
             detach_s_every: int, flags: int, loss, logp, grads: rlt_grads, d_e, d_mem, ws, ws_bytes: int,
             stream=None, check: bool = True) -> int:
    rc = _bptt(model, _ptr(e), _ptr(mem), T_mem, B, n, _ptr(actions), temperature, top_k, detach_s_every,
               flags, _ptr(loss), _ptr(logp), ctypes.byref(grads), _ptr(d_e), _ptr(d_mem), _ptr(ws), ws_bytes,
               _stream_ptr(stream))
    if check:
        _check(rc, "rlt_bptt")
    return rc


def rlt_set_decode_path(model: int, path: int, cluster_size: int = 0):
    _check(_set_decode_path(model, path, cluster_size), "rlt_set_decode_path")


def rlt_fused_plan(model: int, B: int):
    """(cluster_size, seqs_per_cluster, clusters, smem_bytes), or None when the
    fused decoder path does not take this model."""
    out = [_i32() for _ in range(4)]
    rc = _fused_plan(model, B, *[ctypes.byref(x) for x in out])
    if rc == RLT_EUNSUPPORTED:
        return None
    _check(rc, "rlt_fused_plan")
    return tuple(x.value for x in out)


def rlt_debug_withhold_copy(model: int, kernel: int, budget_cycles: int, check: bool = True) -> int:
    """Arms the bounded-wait give-up path for the next launch of `kernel` on
    this model: RLT_KERNEL_XATTN (rlt_cross_attention), RLT_KERNEL_GEMM
    (rlt_linear) or RLT_KERNEL_NORM_PROJ (the layer-0 QKV projection of the
    next rlt_decode_steps call)."""
    rc = _debug_withhold_copy(model, kernel, budget_cycles)
    if check:
        _check(rc, "rlt_debug_withhold_copy")
    return rc


def rlt_timer_arm(model: int, kernel_class: int, max_launches: int):
    _check(_timer_arm(model, kernel_class, max_launches), "rlt_timer_arm")


def rlt_timer_read(model: int, cap: int):
    buf = (ctypes.c_float * max(cap, 1))()
    n = _i32()
    _check(_timer_read(model, buf, cap, ctypes.byref(n)), "rlt_timer_read")
    return [float(buf[i]) for i in range(min(n.value, cap))]


# ---------------------------------------------------------------------------
# torch-side holders

def make_config(c, gate_mode: Optional[int] = None) -> rlt_config:
    """rlt_config from any object with the fields of rlt_inputs.RLTConfig."""
    return rlt_config(c.d, c.n_layers, c.n_heads, c.head_dim, c.d_ffn, c.window, c.mem_groups, c.vocab,
                      RLT_BF16 if c.dtype == "bf16" else RLT_F32, c.rms_eps, c.rope_theta,
                      c.gate_mode if gate_mode is None else gate_mode, getattr(c, "mem_source", RLT_MEM_FINAL))


class Model:
    """Device weights (torch tensors) plus the library's model handle."""

    MATRICES = {"tok_emb", "W_g", "W_qkv", "W_O", "W_1", "W_3", "W_2", "W_Qx", "W_Ox", "W_K", "W_V", "W_o"}

    def __init__(self, cfg, weights: Dict[str, object], device="cuda", version: int = 1):
        import torch
        self.cfg = cfg
        self.dtype = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
        self.t = {}
        for name in WEIGHT_FIELDS:
            w = weights[name]
            if not isinstance(w, torch.Tensor):
                w = torch.from_numpy(w)
            dt = self.dtype if name in self.MATRICES else torch.float32
            self.t[name] = w.to(device=device, dtype=dt).contiguous()
        self.cstruct = rlt_weights(*[self.t[n].data_ptr() for n in WEIGHT_FIELDS])
        self.ccfg = make_config(cfg)
        self.handle = rlt_model_create(self.ccfg, self.cstruct, version)
        self.version = version

    def set_version(self, v: int):
        rlt_model_set_version(self.handle, v)
        self.version = v

    def set_decode_path(self, path: str, cluster_size: int = 0):
        """'graph', 'fused' or 'auto' (rlt_set_decode_path)."""
        rlt_set_decode_path(self.handle, DECODE_PATHS[path], cluster_size)

    def fused_plan(self, B: int):
        return rlt_fused_plan(self.handle, B)

    def timer_arm(self, kernel_class: str, max_launches: int) -> bool:
        rlt_timer_arm(self.handle, RLT_TIMER_CLASSES[kernel_class], max_launches)
        self._timer_cap = max_launches
        return True

    def timer_read(self):
        return rlt_timer_read(self.handle, self._timer_cap)

    def workspace(self, B: int, T_max: int, stream=None):
        import torch
        n = rlt_workspace_size(self.handle, B, T_max)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        rlt_workspace_init(ws, n, stream)
        return ws

    def close(self):
        if self.handle:
            rlt_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class State:
    """Caller-owned state tensors of B sequences plus the C struct over them."""

    def __init__(self, model: Model, B: int):
        import torch
        c = model.cfg
        self.s = torch.empty(B, c.d, dtype=torch.float32, device="cuda")
        shape = (c.n_layers, B, c.n_heads, c.window, c.head_dim)
        self.ring_k = torch.empty(shape, dtype=model.dtype, device="cuda")
        self.ring_v = torch.empty(shape, dtype=model.dtype, device="cuda")
        self.c = rlt_state(B, 0, 0, self.s.data_ptr(), self.ring_k.data_ptr(), self.ring_v.data_ptr())

    @property
    def pos(self) -> int:
        return self.c.pos

    def clone(self) -> "State":
        other = State.__new__(State)
        other.s = self.s.clone()
        other.ring_k = self.ring_k.clone()
        other.ring_v = self.ring_v.clone()
        other.c = rlt_state(self.c.batch, self.c.pos, self.c.version, other.s.data_ptr(),
                            other.ring_k.data_ptr(), other.ring_v.data_ptr())
        return other
