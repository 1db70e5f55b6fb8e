"""The persistent decoder's plan (csrc/fused_plan.h), host logic on the CPU:
which cluster size and how many sequences per cluster the library picks for
a model and a batch, given how many clusters the device holds at once, and
which shapes it rejects.  The co-resident cluster counts are inputs here (on
the device they come from cudaOccupancyMaxActiveClusters)."""
import ctypes
import os
import shutil
import subprocess

import pytest

import rlt_inputs as ri

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "recurrent_looped_transformer_rlt_b300", "csrc")
KEYS = ("CS", "Bc", "nclu", "cols", "hpc", "gph", "npairs", "smem")
SMEM_MAX = 232448


@pytest.fixture(scope="module")
def shim(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not available")
    lib = str(tmp_path_factory.mktemp("plan") / "libplan.so")
    subprocess.run([cxx, "-std=c++17", "-O1", "-shared", "-fPIC", "-I", CSRC, "-o", lib,
                    os.path.join(ROOT, "tests", "fused_plan_shim.cpp")], check=True, capture_output=True)
    return ctypes.CDLL(lib)


def _shape(c):
    return (ctypes.c_int * 9)(c.d, c.n_heads, c.head_dim, c.d_ffn, c.n_layers, c.window, c.vocab, c.mem_groups,
                              1 if c.gate_mode == 0 else 0)


def choose(h, c, B, mac=(148, 74, 37, 18, 8), force=0):
    out = (ctypes.c_longlong * 8)()
    rc = h.plan_choose(_shape(c), B, force, (ctypes.c_int * 5)(*mac), out)
    return None if rc else dict(zip(KEYS, out))


def make(h, c, B, CS, Bc):
    out = (ctypes.c_longlong * 8)()
    rc = h.plan_make(_shape(c), B, CS, Bc, out)
    return None if rc else dict(zip(KEYS, out))


def test_small_model_on_a_full_device(shim):
    """Eight co-resident 16-CTA clusters: 8 clusters of 8 sequences, one wave,
    two CTAs per head (four (sequence, head) pairs each), within 227 KB."""
    c = ri.preset("small").cfg
    p = choose(shim, c, 64)
    assert (p["CS"], p["Bc"], p["nclu"], p["cols"], p["gph"], p["npairs"]) == (16, 8, 8, 8, 2, 4)
    assert p["smem"] <= SMEM_MAX


def test_fewer_coresident_clusters_take_more_sequences_per_cluster_or_waves(shim):
    c = ri.preset("small").cfg
    largest = max(bc for bc in range(1, 17) if make(shim, c, 64, 16, bc) is not None)
    p = choose(shim, c, 64, mac=(148, 74, 37, 18, 7))
    assert p["CS"] == 16 and p["Bc"] == min(largest, 10)
    waves = -(-p["nclu"] // 7)
    assert waves == (1 if largest >= 10 else 2)


def test_small_batches_spread_over_clusters(shim):
    c = ri.preset("small").cfg
    p = choose(shim, c, 3)
    assert p["CS"] == 16 and p["Bc"] == 1 and p["nclu"] == 3


def test_forced_cluster_sizes(shim):
    c = ri.preset("small").cfg
    assert choose(shim, c, 64, force=16)["CS"] == 16
    # 8 CTAs per cluster: each CTA's W_1/W_3 rows (96 units) exceed what a
    # stage half can hold next to the doubled window ring, so the phase runs
    # in parts; the plan still fits
    p = choose(shim, c, 64, force=8)
    assert (p["CS"], p["Bc"], p["nclu"]) == (8, 4, 16) and p["smem"] <= SMEM_MAX   # 18 clusters fit: spread
    assert make(shim, c, 64, 8, 8)["smem"] <= SMEM_MAX
    p4 = choose(shim, c, 64, force=4)                # two heads per CTA: only 2 sequences per cluster fit
    assert (p4["CS"], p4["Bc"], p4["nclu"]) == (4, 2, 32)


def test_fewer_16_cta_clusters_take_more_sequences_each(shim):
    """With only 7 co-resident 16-CTA clusters, the weight phases run in
    parts so that 10 sequences fit a cluster: 7 clusters, one wave."""
    c = ri.preset("small").cfg
    p = choose(shim, c, 64, mac=(148, 74, 37, 16, 7))
    assert (p["CS"], p["Bc"], p["nclu"]) == (16, 10, 7) and p["smem"] <= SMEM_MAX


def test_shapes_the_plan_rejects(shim):
    for name in ("medium", "refdep", "rlreplay"):    # weights far beyond one cluster's shared memory
        assert choose(shim, ri.preset(name).cfg, ri.preset(name).B) is None
    c = ri.RLTConfig(d=80, n_layers=1, n_heads=5, head_dim=16, d_ffn=96, window=4, mem_groups=1, vocab=40,
                     dtype="bf16")
    assert choose(shim, c, 8) is None                # d not a multiple of 32
    c = ri.RLTConfig(d=64, n_layers=1, n_heads=1, head_dim=64, d_ffn=100, window=4, mem_groups=1, vocab=40,
                     dtype="bf16")
    assert make(shim, c, 8, 2, 8) is None            # f not a multiple of 8
    c = ri.RLTConfig(d=64, n_layers=1, n_heads=2, head_dim=32, d_ffn=96, window=4, mem_groups=1, vocab=40,
                     dtype="bf16")
    assert make(shim, c, 8, 3, 8) is None            # 3 CTAs: neither a multiple nor a divisor of 2 heads
    assert make(shim, c, 8, 2, 17) is None           # more than 16 sequences per cluster
    assert choose(shim, c, 8, mac=(0, 0, 0, 0, 0)) is None   # nothing fits on the device
