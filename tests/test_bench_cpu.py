"""The bench's roofline arithmetic, CPU only.

The per-step roofline behind `decode_roofline_frac` is the sum over steps of
max(bytes_t / HBM, flops_t / tensor peak).  These figures were computed
independently from the per-step byte and flop formulas (weights once per
step, the window read, the memory read per layer, the state I/O; 2 flops per
weight per sequence plus the attention) at the nominal 8 TB/s and 2.25
PFLOP/s, before the bench was written; the bench must reproduce them.
"""
import pytest

import bench
import rlt_inputs as ri

# name: (bytes at t = 1 [GB], bytes at t = T [GB], roofline of the whole decode [s], tokens/s, flops at t = 1 [GF])
EXPECTED = {
    "small": (0.008, 0.146, 0.0051, 6.46e6, None),
    "medium": (0.44, 14.1, 1.96, 134e3, None),
    "refdep": (5.94, 115.0, 32.6, 8040.0, None),
    "rlreplay": (0.99, 33.0, 0.62, 422e3, 806.0),
}


@pytest.mark.parametrize("name", sorted(EXPECTED))
def test_roofline_figures(name):
    wl = ri.preset(name)
    c, B, T = wl.cfg, wl.B, wl.T
    b1, bT, roof, tps, gf = EXPECTED[name]
    assert bench.step_bytes(c, B, 1) / 1e9 == pytest.approx(b1, rel=0.05)  # "8 MB": one significant digit
    assert bench.step_bytes(c, B, T) / 1e9 == pytest.approx(bT, rel=0.01)
    r = bench.decode_roofline_s(c, B, T, 8e12, 2.25e15)
    assert r == pytest.approx(roof, rel=0.01)
    assert B * T / r == pytest.approx(tps, rel=0.01)
    if gf is not None:
        assert bench.step_flops(c, B, 1) / 1e9 == pytest.approx(gf, rel=0.01)


def test_roofline_is_bytes_bound_for_the_memory_heavy_configs():
    for name in ("small", "medium", "refdep"):
        wl = ri.preset(name)
        c, B = wl.cfg, wl.B
        for t in (1, wl.T // 2, wl.T):
            assert bench.step_bytes(c, B, t) / 8e12 >= bench.step_flops(c, B, t) / 2.25e15


def test_job_throughput_counts_every_rank():
    assert bench.job_throughput(64, 512, 1, 0.1) == pytest.approx(327680.0)
    assert bench.job_throughput(64, 512, 4, 0.1) == pytest.approx(4 * 327680.0)


@pytest.mark.parametrize("name", ["small", "medium", "refdep", "rlreplay"])
def test_projection_bytes_cover_every_weight_once_per_step(name):
    c = ri.preset(name).cfg
    per = bench.projection_bytes(c, 0)  # no sequences: weights only
    assert len(per) == 6 * c.n_layers + 2
    assert sum(per) == bench.decoder_weight_bytes(c)
    with_rows = bench.projection_bytes(c, 64)
    assert all(a > b for a, b in zip(with_rows, per))


def test_projection_roofline_maps_launches_in_step_order():
    wl = ri.preset("small")
    per = bench.projection_bytes(wl.cfg, wl.B)
    ms = [0.005] * (2 * len(per))  # two steps of 5 us launches
    r = bench.projection_roofline(wl, ms, 6.5e12, "measured")
    assert r["launches"] == 2 * len(per)
    assert r["achieved"] == pytest.approx(2 * sum(per) / (sum(ms) / 1e3) / 1e9, rel=1e-3)
    assert bench.projection_roofline(wl, [], 6.5e12, "measured") is None


def test_bptt_byte_and_flop_accounting():
    """rlt_bptt's algorithmic bytes: with a one-position window and memory
    (n = 1) the call is its weight traffic (recording without the head,
    reverse twice, one block flush of fp32 gradients) plus the small
    activation terms; the block flush is paid once per block of steps; flops
    are four decoder GEMM passes and three attention passes per step."""
    import bench
    c = ri.preset("small").cfg
    B = 64
    es = 2
    wb = bench.decoder_weight_bytes(c)
    head = es * c.vocab * c.d
    params = bench.decoder_params(c)
    assert wb == es * params
    one = bench.bptt_bytes(c, B, 1)
    weights_only = (wb - head) + 2 * wb - es * c.d * c.d_ffn + 8 * params
    assert weights_only < one < weights_only * 1.3
    # the block flush: one per block of S steps
    n = 40
    per_block = [bench.bptt_bytes(c, B, n, S) for S in (1, 8, 40)]
    assert per_block[0] > per_block[1] > per_block[2]
    assert per_block[0] - per_block[2] >= 39 * 8 * params
    # each step costs more than a forward step and less than four
    for t in (1, 64, 512):
        d1 = bench.bptt_bytes(c, B, t + 1, 10 ** 9) - bench.bptt_bytes(c, B, t, 10 ** 9)
        assert bench.step_bytes(c, B, t + 1) < d1 < 4 * bench.step_bytes(c, B, t + 1)
    f1 = bench.bptt_flops(c, B, 1)
    gemm = 2 * B * params
    attn = 4 * B * c.d * c.n_layers * 2
    assert f1 == 4 * gemm + 3 * attn


def test_fused_roofline_counts_every_step_once():
    """The persistent decoder's roofline object: one launch for the whole
    decode call, whose algorithmic bytes are the sum of the per-step bytes;
    at the roofline time (bytes / HBM) the fraction is 1."""
    wl = ri.preset("small")
    c, B, T = wl.cfg, wl.B, wl.T
    total = sum(bench.step_bytes(c, B, t) for t in range(1, T + 1))
    # the small decode moves ~39 GB: ~0.146 GB at t = T, ~0.008 GB at t = 1, linear in t
    assert total / 1e9 == pytest.approx((0.008 + 0.146) / 2 * T, rel=0.03)
    bw = 7.0e12
    r = bench.fused_roofline(wl, total / bw, bw, "test")
    assert r["frac"] == pytest.approx(1.0, abs=1e-3) and r["launches"] == 1 and r["bound"] == "hbm"
    assert bench.fused_roofline(wl, 2 * total / bw, bw, "test")["frac"] == pytest.approx(0.5, abs=1e-3)


def test_fused_case_bytes_are_the_steps_it_runs():
    """--profile-case fused times n steps from p0 = T/2 - n/2: its bytes are
    those of steps p0 + 1 .. p0 + n, the decoder weights once per step plus
    the memory read growing with t."""
    wl = ri.preset("small")
    c, B, T = wl.cfg, wl.B, wl.T
    n = 32
    p0 = T // 2 - n // 2
    total = sum(bench.step_bytes(c, B, p + 1) for p in range(p0, p0 + n))
    mid = bench.step_bytes(c, B, p0 + n // 2)
    assert total == pytest.approx(n * mid, rel=0.02)     # linear in t: the mean is the middle step
    assert bench.step_bytes(c, B, p0 + n) - bench.step_bytes(c, B, p0 + 1) == \
        (n - 1) * c.n_layers * bench.xattn_bytes(c, B, 1)


def test_segments_cover_every_position_once():
    """The K bench steps are consecutive rlt_decode_steps ranges that consume
    positions 0..T-1 exactly once, in order, with lengths differing by at
    most one."""
    for T, K in [(4096, 20), (512, 20), (64, 64), (7, 3), (5, 1)]:
        segs = bench.segments(T, K)
        assert len(segs) == K
        p = 0
        for p0, n in segs:
            assert p0 == p and n >= 1
            p += n
        assert p == T
        assert max(n for _, n in segs) - min(n for _, n in segs) <= 1
    with pytest.raises(SystemExit):
        bench.segments(10, 11)


def test_config_names_the_step():
    import rlt_inputs as ri
    cfg = bench.workload_config(ri.preset("refdep"), 1, 20)
    assert cfg["T"] == 4096 and cfg["B_per_gpu"] == 64
    assert "205 positions" in cfg["step"] and "1..4096" in cfg["step"]
