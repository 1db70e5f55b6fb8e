"""GPU parity of the persistent cluster decoder (rlt_set_decode_path(...,
RLT_DECODE_FUSED)).  The same kernel is also checked on the CPU under the
host emulation of the CUDA execution model
(tests/test_fused_decoder_emulated_cpu.py).

Small bf16 model against the oracle with the bf16 tolerances of the other
parity tests (relative logit error, argmax agreement), against the graph path
on the same inputs, call-split bitwise invariance within the path, every
cluster size the plan accepts, and the full-size workload on sampled rows.
"""
import numpy as np
import pytest

import rlt_inputs as ri
from tests.gpu_common import BF16_REL_LOGIT, gpu_run, oracle_run, rel_logit_err
from tests.test_gpu_parity import _check_bf16, _inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,T", [(8, 160), (3, 37), (21, 24)])
def test_fused_small_bf16_parity(B, T):
    wl, W, tok, acts = _inputs("small", B=B, T=T)
    emit = list(range(T))
    g = gpu_run(wl, W, tok, acts, emit=emit, decode_path="fused")
    o = oracle_run(wl, W, tok, acts, emit=emit)
    assert g["status"] == 0
    _check_bf16(g, o, emit)


@pytest.mark.parametrize("cs", [16, 8, 4, 2, 1])
def test_fused_every_cluster_size(cs):
    """Each cluster size the plan takes, forced, against the oracle."""
    import recurrent_looped_transformer_rlt_b300 as rlt
    wl, W, tok, acts = _inputs("small", B=19, T=40)
    m = rlt.Model(wl.cfg, W)
    m.set_decode_path("fused", cs)
    plan = m.fused_plan(19)
    m.close()
    if plan is None:
        pytest.skip(f"cluster size {cs} not schedulable with this shape")
    assert plan[0] == cs and plan[1] <= 16 and plan[1] * plan[2] >= 19
    emit = [0, 17, 39]
    g = gpu_run(wl, W, tok, acts, emit=emit, decode_path="fused", cluster_size=cs)
    o = oracle_run(wl, W, tok, acts, emit=emit)
    assert g["status"] == 0
    _check_bf16(g, o, emit)


def test_fused_agrees_with_graph_path():
    wl, W, tok, acts = _inputs("small", B=16, T=96)
    emit = [0, 47, 95]
    f = gpu_run(wl, W, tok, acts, emit=emit, decode_path="fused")
    g = gpu_run(wl, W, tok, acts, emit=emit, decode_path="graph")
    for i in emit:
        assert rel_logit_err(f["logits"][i], g["logits"][i]).max() <= BF16_REL_LOGIT
    assert np.mean(f["argmax"] == g["argmax"]) >= 0.99
    assert np.abs(f["s"] - g["s"]).max() <= BF16_REL_LOGIT * np.abs(g["s"]).max()


def test_fused_split_invariance_bitwise():
    wl, W, tok, acts = _inputs("small", B=16, T=96)
    a = gpu_run(wl, W, tok, acts, emit=[95], decode_path="fused")
    b = gpu_run(wl, W, tok, acts, n_split=[5, 17, 64], emit=[95], decode_path="fused")
    for k in ("s", "ring_k", "ring_v", "argmax", "logp", "logp_full"):
        assert np.array_equal(a[k], b[k], equal_nan=True), k
    assert np.array_equal(a["logits"][95], b["logits"][95])


def test_fused_top_k_and_gate_discard():
    wl, W, tok, acts = _inputs("small", B=6, T=30)
    emit = list(range(30))
    for kw in (dict(temperature=0.7, top_k=5), dict(gate_mode=1)):
        g = gpu_run(wl, W, tok, acts, emit=emit, decode_path="fused", **kw)
        o = oracle_run(wl, W, tok, acts, emit=emit, **kw)
        assert g["status"] == 0
        _check_bf16(g, o, emit, kw.get("top_k", 0), acts, kw.get("temperature", 1.0))


def test_fused_full_size_sampled_rows():
    """Full small workload (B=64, T=512) through the fused path; four sequences
    against the oracle."""
    wl, W, tok, acts = _inputs("small", jitter=0.0)
    T = wl.T
    emit = [0, 1, 15, 16, 255, 511]
    g = gpu_run(wl, W, tok, acts, emit=emit, decode_path="fused")
    assert g["status"] == 0
    rows = [0, 21, 42, 63]
    o = oracle_run(wl, W, tok[rows], acts[rows], emit=emit)
    for i in emit:
        assert rel_logit_err(g["logits"][i][rows], o["logits"][i]).max() <= BF16_REL_LOGIT


def test_fused_rejects_fp32_models():
    import recurrent_looped_transformer_rlt_b300 as rlt
    wl = ri.preset("tiny")
    m = rlt.Model(wl.cfg, ri.make_weights(wl.cfg, wl.seed))
    assert m.fused_plan(8) is None
    m.close()


def test_fused_generation_matches_the_oracle():
    """rlt_generate on the fused path under the graph path's generation
    contract: encoder rows, memory rows, state and behaviour log-probabilities
    against the oracle's teacher-forced run over the generated tokens, each
    draw at its uniform number."""
    from tests import test_gpu_generate as TG
    TG.test_generation_matches_the_oracle_on_the_generated_sequence(path="fused")


def test_fused_generation_call_split_bitwise():
    from tests import test_gpu_generate as TG
    TG.test_generation_does_not_depend_on_the_call_split(path="fused")


def test_fused_plan_of_the_small_workload():
    """The plan the bench's workload gets: 16-CTA clusters of 8 sequences,
    8 clusters (one per GPC, one wave); with only 7 resident 16-CTA clusters
    the plan takes 10 sequences each (weight phases in parts)."""
    import recurrent_looped_transformer_rlt_b300 as rlt
    wl = ri.preset("small")
    m = rlt.Model(wl.cfg, ri.make_weights(wl.cfg, wl.seed))
    m.set_decode_path("fused")
    plan = m.fused_plan(wl.B)
    m.close()
    assert plan is not None
    cs, bc, ncl, smem = plan
    assert (cs, bc, ncl) in ((16, 8, 8), (16, 10, 7)), plan
    assert smem <= 232448
