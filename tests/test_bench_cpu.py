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
