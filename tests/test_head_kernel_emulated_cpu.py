"""The forward head kernel (head_reduce_kernel: tempered log-softmax with the
action's log-probability, the top-k set by radix select with ties to the lower
id, the argmax, and the sampling draw of generation) run under the host
emulation of the CUDA execution model (tests/simt_emu), against the oracle's
scoring and sampling on tie-heavy logits.

The kernel is compiled with g++ against stand-in CUDA headers (one host
thread per CUDA thread, barriers for __syncthreads and warp shuffles) and
launched with the library's grid and block (one 1024-thread block per row).
This checks the selection and tie logic without a GPU; the GPU tests check the
same kernel on the device.
"""
import ctypes
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

from oracle import rlt_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "recurrent_looped_transformer_rlt_b300", "csrc")
EMU = os.path.join(ROOT, "tests", "simt_emu")


@pytest.fixture(scope="module")
def head(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not available")
    d = str(tmp_path_factory.mktemp("head_emu"))
    src = open(os.path.join(CSRC, "kernels.cuh")).read()
    src, n = re.subn(r'#include "ptx.cuh"', "namespace rlt { inline void pdl_wait() {} inline void pdl_trigger() {} }",
                     src)
    assert n == 1
    src, n = re.subn(r"extern __shared__ float (\w+)\[\];", r"float* \1 = emu_dyn_smem<float>();", src)
    assert n >= 1
    open(os.path.join(d, "kernels_emu.cuh"), "w").write(src)
    lib = os.path.join(d, "libhead.so")
    r = subprocess.run([cxx, "-std=c++20", "-O1", "-shared", "-fPIC", "-pthread", "-I", d, "-I", EMU, "-I", CSRC,
                        "-o", lib, os.path.join(EMU, "head_harness.cpp")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    h = ctypes.CDLL(lib)
    h.head_emu.restype = ctypes.c_int
    return h


def _run(h, lg, act, tau, k, sample=False, seed=0, pos=0):
    B, V = lg.shape
    lg = np.ascontiguousarray(lg, np.float32)
    act = np.ascontiguousarray(act, np.int32)
    lp, lf = np.zeros(B, np.float32), np.zeros(B, np.float32)
    am, tok = np.zeros(B, np.int32), np.full(B, -1, np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    rc = h.head_emu(p(lg), p(act), B, V, ctypes.c_float(1.0 / tau), k, int(sample), ctypes.c_ulonglong(seed), pos,
                    p(lp), p(lf), p(am), p(tok))
    assert rc == 0
    return lp, lf, am, tok


def _logits(rng, kind, B, V):
    if kind == "equal":
        x = np.zeros((B, V))
    elif kind == "integers":          # many ties at every value, the k-th included
        x = rng.integers(-3, 3, (B, V)).astype(float)
    elif kind == "duplicates":        # every 7th id repeats the first logit
        x = rng.standard_normal((B, V))
        x[:, ::7] = x[:, :1]
    else:
        x = 3.0 * rng.standard_normal((B, V))
    return x.astype(np.float32)


CASES = [(kind, V, k) for kind in ("equal", "integers", "duplicates", "normal")
         for V, k in ((5, 0), (37, 1), (37, 36), (37, 37), (37, 40), (700, 11), (1500, 100), (3000, 1024))]


@pytest.mark.parametrize("kind,V,k", CASES)
def test_scoring_matches_the_oracle(head, kind, V, k):
    """lp over the top-k set (-inf outside it), lp_full over the vocabulary and
    the argmax (lowest id on ties) equal the oracle's on the same tempered
    fp32 logits; membership of tied actions follows the lower-id rule."""
    rng = np.random.default_rng(V * 31 + k)
    B, tau = 4, 0.7
    lg = _logits(rng, kind, B, V)
    x = lg * np.float32(1.0 / tau)            # the kernel's tempered logits, fp32
    order = np.argsort(-x[0], kind="stable")
    # actions at both sides of the k-th place, so ties at the boundary are hit
    act = np.array([order[min(max(k - 1, 0), V - 1)], order[min(k, V - 1)], rng.integers(V), order[0]], np.int32)
    lp, lf, am, _ = _run(head, lg, act, tau, k)
    lpr, lfr = O.score(x.astype(np.float64), act, 1.0, k)
    np.testing.assert_allclose(lf, lfr, rtol=0, atol=2e-5 * max(1.0, np.abs(lfr).max()))
    assert np.array_equal(np.isinf(lp), np.isinf(lpr))
    fin = np.isfinite(lpr)
    np.testing.assert_allclose(lp[fin], lpr[fin], rtol=0, atol=2e-5 * max(1.0, np.abs(lpr[fin]).max(initial=0)))
    assert np.array_equal(am, np.argmax(lg, axis=1))


@pytest.mark.parametrize("kind,V,k", [c for c in CASES if c[1] >= 37])
def test_sampling_matches_the_oracle(head, kind, V, k):
    """The drawn token is the oracle's sample_token for the same uniform
    number (SplitMix64 of seed, row and position), except where u lies within
    fp32 summation error of a cumulative-probability boundary, where either
    neighbour is correct; the token's lp equals the oracle's score of it."""
    rng = np.random.default_rng(V * 17 + k)
    B, tau, seed, pos = 6, 0.9, 0x1234ABCD, 5
    lg = _logits(rng, kind, B, V)
    x = lg * np.float32(1.0 / tau)
    _, _, _, tok = _run(head, lg, np.zeros(B, np.int32), tau, k, sample=True, seed=seed, pos=pos)
    for b in range(B):
        u = O.uniform24(seed, b, pos)
        want = O.sample_token(x[b].astype(np.float64), u, 1.0, k)
        if tok[b] != want:
            c = np.cumsum(O.sampling_distribution(x[b].astype(np.float64), 1.0, k))
            near = np.abs(c - u).min()
            assert near < 1e-5, (b, tok[b], want, near)
        p = O.sampling_distribution(x[b].astype(np.float64), 1.0, k)
        assert p[tok[b]] > 0, "drawn token outside the top-k set"
