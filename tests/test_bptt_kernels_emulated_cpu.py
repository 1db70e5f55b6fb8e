"""The backward's device kernels, run under a host emulation of the CUDA
execution model (tests/simt_emu), against the float64 autograd oracle.

bptt.cuh's kernels are compiled with g++ against stand-in CUDA headers (one
host thread per CUDA thread, barriers for __syncthreads and warp shuffles)
and driven by the device Ops of bptt_api.cuh with each launch rewritten to
the emulator's launcher: the same grids, blocks and arguments as on the GPU.
The projections run as a reference loop into the same epilogue functors
(the GEMM kernels themselves are covered by the forward's GPU tests).  This
checks the kernels' index arithmetic, launch configurations and lane
pairings without a GPU; the results are not GPU parity (the GPU tests are).
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
from oracle import rlt_bptt as BP
from oracle import rlt_oracle as O
from tests import test_bptt_schedule_cpu as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "recurrent_looped_transformer_rlt_b300", "csrc")
EMU = os.path.join(ROOT, "tests", "simt_emu")


def _generate(out_dir):
    """bptt.cuh with the dynamic shared array from the emulator, and the
    device Ops with every `kernel<<<grid, block, smem, st>>>(args);` launch
    rewritten as `emu_launch(grid, block, smem, kernel, args);`."""
    src = open(os.path.join(CSRC, "bptt.cuh")).read()
    src, n = re.subn(r"extern __shared__ float (\w+)\[\];", r"float* \1 = emu_dyn_smem<float>();", src)
    assert n == 1
    open(os.path.join(out_dir, "bptt_emu.cuh"), "w").write(src)
    api = open(os.path.join(CSRC, "bptt_api.cuh")).read()
    a = api.index("template <typename T_>\nstruct BpttOps {")
    b = api.index("};", api.index("  int loss_sum(")) + 2
    ops, n = re.subn(r"([\w:<>]+)<<<(.*?), st>>>\((.*?)\);", r"emu_launch(\2, \1, \3);", api[a:b], flags=re.S)
    assert n >= 15 and "<<<" not in ops
    open(os.path.join(out_dir, "emu_ops.inc"), "w").write(ops.replace("BpttOps", "EmuOps"))


@pytest.fixture(scope="module")
def emu(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not available")
    d = str(tmp_path_factory.mktemp("simt_emu"))
    _generate(d)
    lib = os.path.join(d, "libemu.so")
    # keys per warp of the split memory attention: 3, so that the short test
    # sequences take both the single-warp and the split-and-combine paths
    r = subprocess.run([cxx, "-std=c++20", "-O1", "-shared", "-fPIC", "-pthread", "-DRLT_BPTT_ATTN_CHUNK=3", "-I", d,
                        "-I", EMU, "-I", CSRC, "-o", lib, os.path.join(EMU, "emu_harness.cpp")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    h = ctypes.CDLL(lib)
    h.bptt_emu.restype = ctypes.c_int
    return h


def _run(h, c, W, e, mem, acts, block=4, bf16=False, **kw):
    B, n = acts.shape
    sh = [B, n, e.shape[1], c.d, c.n_heads, c.head_dim, c.d_ffn, c.n_layers, c.window, c.vocab, c.mem_groups,
          1 if c.gate_mode == 0 else 0, kw.get("k", 0), kw.get("s_every", 0), int(kw.get("cache", False)),
          int(kw.get("memory", False)), block, int(bf16)]
    arrs = [np.ascontiguousarray(np.asarray(W[p], np.float32)) for p in S.PARAMS]
    arrs += [np.ascontiguousarray(e, np.float32), np.ascontiguousarray(mem, np.float32),
             np.ascontiguousarray(acts, np.int32)]
    loss, logp = np.zeros(1, np.float32), np.zeros((B, n), np.float32)
    grads = {g: np.zeros(np.shape(W[g]), np.float32) for g in S.GRADS}
    d_e, d_mem = np.zeros(e.shape, np.float32), np.zeros(mem.shape, np.float32)
    arrs += [loss, logp] + [grads[g] for g in S.GRADS] + [d_e, d_mem]
    ptrs = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    nel = (ctypes.c_size_t * len(arrs))(*[a.size for a in arrs])
    rc = h.bptt_emu((ctypes.c_int * len(sh))(*sh), (ctypes.c_float * 3)(c.rms_eps, c.rope_theta, kw.get("tau", 1.0)),
                    ptrs, nel)
    assert rc == 0
    return float(loss[0]), grads, d_e, d_mem


def _worst(loss, g, d_e, d_mem, lref, gref):
    w = abs(loss - lref) / max(1.0, abs(lref))
    for name, x in list(g.items()) + [("e", d_e), ("mem", d_mem)]:
        scale = np.abs(gref[name]).max()
        w = max(w, np.abs(x - gref[name]).max() / scale if scale > 0 else np.abs(x).max())
    return w


@pytest.mark.parametrize("setup_kw,kw", [
    ({"G": 2}, {}),                                        # ring wraps, one memory group per layer
    ({"T": 9}, {"s_every": 3, "cache": True, "memory": True}),
    ({"T": 9, "window": 7}, {}),                           # window and records over several 3-key chunks
])
def test_emulated_kernels_fp32(emu, setup_kw, kw):
    c, W, e, mem, acts = S._setup(**setup_kw)
    loss, g, d_e, d_mem = _run(emu, c, W, e, mem, acts, **kw)
    lref, gref = BP.gradients(O.Cfg.of(c), W, e, mem, acts, detach_s_every=kw.get("s_every", 0),
                              detach_cache=kw.get("cache", False), detach_memory=kw.get("memory", False))
    assert _worst(loss, g, d_e, d_mem, lref, gref) < 1e-4


@pytest.mark.parametrize("hd", [64, 128])
def test_emulated_kernels_wide_heads(emu, hd):
    """Head widths >= 64: RoPE partners in the same lane's registers."""
    c = ri.RLTConfig(d=2 * hd, n_layers=1, n_heads=2, head_dim=hd, d_ffn=48, window=3, mem_groups=1, vocab=9,
                     dtype="f32")
    W = ri.make_weights(c, 41, norm_jitter=0.1)
    for k in W:
        if W[k].ndim >= 2:
            W[k] = W[k] * 2.0
    B, T = 1, 4
    e, mem = ri.make_decoder_inputs(c, B, T, 48, mem_scale=0.5)
    acts = (np.arange(B * T).reshape(B, T) % c.vocab).astype(np.int32)
    loss, g, d_e, d_mem = _run(emu, c, W, e, mem, acts)
    lref, gref = BP.gradients(O.Cfg.of(c), W, e, mem, acts)
    assert _worst(loss, g, d_e, d_mem, lref, gref) < 1e-4


def test_emulated_kernels_bf16(emu):
    """The kernels' bf16 instantiations (projections by a reference loop):
    within bf16 rounding of the oracle on the same bf16 weights and inputs."""
    c = ri.RLTConfig(d=256, n_layers=1, n_heads=8, head_dim=32, d_ffn=512, window=2, mem_groups=1, vocab=64,
                     dtype="bf16")
    W = ri.make_weights(c, 41, norm_jitter=0.1)
    B, T = 2, 3
    e, mem = ri.make_decoder_inputs(c, B, T, 48, mem_scale=0.5)
    acts = (np.arange(B * T).reshape(B, T) * 7 % c.vocab).astype(np.int32)
    loss, g, d_e, d_mem = _run(emu, c, W, e, mem, acts, block=16, bf16=True)
    cfg = O.Cfg.of(ri.RLTConfig(**{**c.__dict__, "dtype": "f32"}))
    lref, gref = BP.gradients(cfg, W, e, mem, acts)
    assert abs(loss - lref) <= 1e-3 * abs(lref)
    for name, x in list(g.items()) + [("e", d_e), ("mem", d_mem)]:
        r = gref[name]
        assert np.linalg.norm((x - r).ravel()) <= 1e-2 * np.linalg.norm(r.ravel()), name


@pytest.fixture(scope="module")
def emu64(tmp_path_factory):
    """The kernels with the library's own key chunk (64 keys per warp)."""
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not available")
    d = str(tmp_path_factory.mktemp("simt_emu64"))
    _generate(d)
    lib = os.path.join(d, "libemu.so")
    r = subprocess.run([cxx, "-std=c++20", "-O2", "-shared", "-fPIC", "-pthread", "-I", d, "-I", EMU, "-I", CSRC,
                        "-o", lib, os.path.join(EMU, "emu_harness.cpp")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    h = ctypes.CDLL(lib)
    h.bptt_emu.restype = ctypes.c_int
    return h


def test_emulated_kernels_production_chunk(emu64):
    """67 steps with the library's 64-key chunk: the last steps' memory
    attention is split in two and combined, the last 16-step block is ragged
    (67 = 4 x 16 + 3)."""
    c = ri.RLTConfig(d=64, n_layers=1, n_heads=2, head_dim=32, d_ffn=96, window=16, mem_groups=1, vocab=40,
                     dtype="f32")
    W = ri.make_weights(c, 41, norm_jitter=0.1)
    for k in W:
        if W[k].ndim >= 2:
            W[k] = W[k] * 2.0
    B, T = 1, 67
    e, mem = ri.make_decoder_inputs(c, B, T, 48, mem_scale=0.5)
    acts = (np.arange(B * T).reshape(B, T) * 7 % c.vocab).astype(np.int32)
    loss, g, d_e, d_mem = _run(emu64, c, W, e, mem, acts, block=16)
    lref, gref = BP.gradients(O.Cfg.of(c), W, e, mem, acts)
    assert _worst(loss, g, d_e, d_mem, lref, gref) < 1e-4


def test_emulated_kernels_have_no_unordered_shared_accesses(emu, tmp_path):
    """Two runs with EMU_JITTER=1 (a random sleep after every block barrier,
    so that an access no barrier orders gives run-dependent results) are
    bitwise identical: an fp32 model, and a bf16 model (tensor-core memory
    gradient)."""
    lib = emu._name
    script = tmp_path / "jitter.py"
    script.write_text(
        "import ctypes, sys\n"
        "import numpy as np\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "from tests import test_bptt_kernels_emulated_cpu as E\n"
        "from tests import test_bptt_schedule_cpu as S\n"
        f"h = ctypes.CDLL({lib!r})\n"
        "h.bptt_emu.restype = ctypes.c_int\n"
        "import rlt_inputs as ri\n"
        "c, W, e, mem, acts = S._setup(T=9, window=7)\n"
        "cb = ri.RLTConfig(d=64, n_layers=1, n_heads=2, head_dim=32, d_ffn=96, window=3, mem_groups=1, vocab=32,\n"
        "                  dtype='bf16')\n"
        "Wb = ri.make_weights(cb, 41, norm_jitter=0.1)\n"
        "eb, mb = ri.make_decoder_inputs(cb, 2, 5, 48, mem_scale=0.5)\n"
        "ab = (np.arange(10).reshape(2, 5) * 5 % 32).astype(np.int32)\n"
        "for args, kw in (((c, W, e, mem, acts), {}), ((cb, Wb, eb, mb, ab), dict(block=16, bf16=True))):\n"
        "    a = E._run(h, *args, **kw)\n"
        "    b = E._run(h, *args, **kw)\n"
        "    assert a[0] == b[0]\n"
        "    for k in a[1]:\n"
        "        assert np.array_equal(a[1][k], b[1][k]), k\n"
        "    assert np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3])\n")
    env = dict(os.environ, EMU_JITTER="1")
    r = subprocess.run([sys.executable, str(script)], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]


@pytest.mark.parametrize("hd", [64, 128])
def test_emulated_tensor_core_memory_gradient_wide_heads(emu, hd):
    """bf16 models take the tensor-core memory gradient (one template per head
    width): at widths 64 and 128, within bf16 rounding of the oracle."""
    c = ri.RLTConfig(d=2 * hd, n_layers=1, n_heads=2, head_dim=hd, d_ffn=128, window=2, mem_groups=1, vocab=32,
                     dtype="bf16")
    W = ri.make_weights(c, 41, norm_jitter=0.1)
    B, T = 2, 5
    e, mem = ri.make_decoder_inputs(c, B, T, 48, mem_scale=0.5)
    acts = (np.arange(B * T).reshape(B, T) * 5 % c.vocab).astype(np.int32)
    loss, g, d_e, d_mem = _run(emu, c, W, e, mem, acts, block=16, bf16=True)
    cfg = O.Cfg.of(ri.RLTConfig(**{**c.__dict__, "dtype": "f32"}))
    lref, gref = BP.gradients(cfg, W, e, mem, acts)
    assert np.linalg.norm((d_mem - gref["mem"]).ravel()) <= 1e-2 * np.linalg.norm(gref["mem"].ravel())
    assert abs(loss - lref) <= 1e-3 * abs(lref)
