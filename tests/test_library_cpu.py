"""The C-ABI library builds, loads and exports every declared symbol (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            txt = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"RLT_API\s+[\w\s\*]*?\b(rlt_\w+)\s*\(", txt))
    return names


def test_header_declares_the_boundary_calls():
    names = _declared()
    for n in ("rlt_state_init", "rlt_encode", "rlt_decode_steps", "rlt_model_create", "rlt_status"):
        assert n in names


def test_library_loads_and_exports_every_declared_symbol():
    import recurrent_looped_transformer_rlt_b300 as rlt
    lib = ctypes.CDLL(rlt.LIB_PATH)
    for n in _declared():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", rlt.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.strip()}
    assert _declared() <= exported
    assert set(rlt.EXPORTED) == _declared()


def test_library_is_built_for_sm_103a():
    import recurrent_looped_transformer_rlt_b300 as rlt
    out = subprocess.run(["cuobjdump", "--list-elf", rlt.LIB_PATH], capture_output=True, text=True).stdout
    assert "sm_103a" in out


def test_abi_version_and_strerror():
    import recurrent_looped_transformer_rlt_b300 as rlt
    assert rlt.rlt_abi_version() == 200
    assert rlt.rlt_strerror(rlt.RLT_ESTALE).startswith("state built")
    assert rlt.rlt_strerror(12345) == "unknown error"


@pytest.mark.parametrize("field,value,code", [
    ("d_model", 100, -1),        # d != H * hd
    ("mem_groups", 3, -1),       # neither 1 nor L
    ("dtype", 7, -1),
    ("head_dim", 24, -1),        # d mismatch first
    ("gate_mode", 5, -1),
    ("vocab", 0, -1),
    ("mem_source", 2, -1),
    ("mem_source", 1, -1),       # per-layer memory needs one group per layer (tiny has G = 1, L = 2)
])
def test_model_create_rejects_bad_config_without_gpu(field, value, code):
    import recurrent_looped_transformer_rlt_b300 as rlt
    import rlt_inputs as ri
    cfg = rlt.make_config(ri.preset("tiny").cfg)
    setattr(cfg, field, value)
    w = rlt.rlt_weights(*([16] * len(rlt.WEIGHT_FIELDS)))
    h = ctypes.c_void_p()
    rc = rlt._model_create(ctypes.byref(cfg), ctypes.byref(w), 0, ctypes.byref(h))
    assert rc == code and not h.value


def test_model_create_rejects_null_and_misaligned_weights():
    import recurrent_looped_transformer_rlt_b300 as rlt
    import rlt_inputs as ri
    cfg = rlt.make_config(ri.preset("tiny").cfg)
    h = ctypes.c_void_p()
    w = rlt.rlt_weights(*([16] * len(rlt.WEIGHT_FIELDS)))
    w.W_O = None
    assert rlt._model_create(ctypes.byref(cfg), ctypes.byref(w), 0, ctypes.byref(h)) == rlt.RLT_EINVAL
    w = rlt.rlt_weights(*([16] * len(rlt.WEIGHT_FIELDS)))
    w.W_2 = 18
    assert rlt._model_create(ctypes.byref(cfg), ctypes.byref(w), 0, ctypes.byref(h)) == rlt.RLT_EINVAL


def test_unsupported_head_dim_reported():
    import recurrent_looped_transformer_rlt_b300 as rlt
    import rlt_inputs as ri
    cfg = rlt.make_config(ri.preset("tiny").cfg)
    cfg.head_dim, cfg.n_heads, cfg.d_model = 12, 4, 48
    w = rlt.rlt_weights(*([16] * len(rlt.WEIGHT_FIELDS)))
    h = ctypes.c_void_p()
    assert rlt._model_create(ctypes.byref(cfg), ctypes.byref(w), 0, ctypes.byref(h)) == rlt.RLT_EUNSUPPORTED


def test_decode_path_calls_reject_bad_arguments_without_gpu():
    """rlt_set_decode_path and rlt_fused_plan validate on the host: a null
    model, an unknown path, a cluster size that is not 0, 1, 2, 4, 8 or 16, a
    non-positive batch."""
    import recurrent_looped_transformer_rlt_b300 as rlt
    assert rlt._set_decode_path(None, rlt.RLT_DECODE_FUSED, 0) == rlt.RLT_EINVAL
    out = [ctypes.c_int32() for _ in range(4)]
    assert rlt._fused_plan(None, 8, *[ctypes.byref(x) for x in out]) == rlt.RLT_EINVAL
    # a fake (non-null) handle is never dereferenced before the argument checks fail
    fake = ctypes.c_void_p(16)
    assert rlt._set_decode_path(fake, 3, 0) == rlt.RLT_EINVAL
    assert rlt._set_decode_path(fake, rlt.RLT_DECODE_FUSED, 3) == rlt.RLT_EINVAL
    assert rlt._set_decode_path(fake, rlt.RLT_DECODE_FUSED, 32) == rlt.RLT_EINVAL
    assert rlt._fused_plan(fake, 0, *[ctypes.byref(x) for x in out]) == rlt.RLT_EINVAL


def test_withhold_copy_rejects_bad_arguments_without_gpu():
    """rlt_debug_withhold_copy validates before touching the model: a null
    model, an unknown kernel class, a wait budget outside 1e3 .. 4e9 cycles."""
    import recurrent_looped_transformer_rlt_b300 as rlt
    assert rlt.rlt_debug_withhold_copy(None, rlt.RLT_KERNEL_XATTN, 10 ** 6, check=False) == rlt.RLT_EINVAL
    fake = ctypes.c_void_p(16)
    assert rlt._debug_withhold_copy(fake, 0, 10 ** 6) == rlt.RLT_EINVAL
    assert rlt._debug_withhold_copy(fake, 4, 10 ** 6) == rlt.RLT_EINVAL
    assert rlt._debug_withhold_copy(fake, rlt.RLT_KERNEL_NORM_PROJ, 999) == rlt.RLT_EINVAL
    assert rlt._debug_withhold_copy(fake, rlt.RLT_KERNEL_XATTN, 999) == rlt.RLT_EINVAL
    assert rlt._debug_withhold_copy(fake, rlt.RLT_KERNEL_GEMM, 4 * 10 ** 9 + 1) == rlt.RLT_EINVAL
