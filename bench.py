"""Throughput of the RLT hot path on one B300 (or N replicas).

One pass of the hot path over one batch of synthetic sequences is: state
init (H_0), the token-parallel encode with memory projection of all T
positions, and the batched recurrent decoder over positions 1..T with
teacher-forced scoring of every next token (tempered top-k log-probabilities
for the replay workload).  A bench step is one rlt_decode_steps call over the
next T/K positions of all B sequences with the state carried, so the K timed
steps make one pass (Proposition 3.1: the split into calls does not change the
state); the encode runs once at the start of the timed region and is timed on
its own.  The default workload is the reference-depth model (d = 2048, 48
tied layers, B = 64, T = 4096).  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload refdep]
  python bench.py --impl reference ...   # the CPU oracle on bounded samples

Multi-GPU: sequences are sharded by index (each rank its own B sequences,
weak scaling); there is no collective on the data path, only a barrier and
a max-over-ranks reduction of the timings.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import rlt_inputs as ri  # noqa: E402

METRIC = "decoder tokens/s (B seqs x steps/s) on 1 B300; % of per-step HBM/TC roofline"
UNIT = "tokens/s"
L2_BYTES = 126 * 2 ** 20


# ---------------------------------------------------------------------------
# roofline arithmetic (algorithmic bytes / flops of the decoder)

def decoder_weight_bytes(c) -> int:
    es = 2 if c.dtype == "bf16" else 4
    d, f, L, V = c.d, c.d_ffn, c.n_layers, c.vocab
    return es * (L * (6 * d * d + 3 * d * f) + 2 * d * d + V * d)


def xattn_bytes(c, B, t) -> int:
    """Memory K and V of positions 1..t read by one layer's cross-attention (per step)."""
    es = 2 if c.dtype == "bf16" else 4
    return es * B * t * 2 * c.d


def step_bytes(c, B, t) -> int:
    es = 2 if c.dtype == "bf16" else 4
    n_win = min(c.window, t)
    swa = es * B * c.n_layers * (n_win - 1 + 1) * 2 * c.d
    mem = c.n_layers * xattn_bytes(c, B, t)
    io = B * c.d * 4 * 2 + B * c.d * es + B * 4 * 3
    return decoder_weight_bytes(c) + swa + mem + io


def step_flops(c, B, t) -> int:
    d, f, L, V = c.d, c.d_ffn, c.n_layers, c.vocab
    gemm = 2 * B * (L * (6 * d * d + 3 * d * f) + 2 * d * d + V * d)
    attn = 4 * B * d * L * (min(c.window, t) + t)
    return gemm + attn


def decode_roofline_s(c, B, T, bw, peak) -> float:
    return sum(max(step_bytes(c, B, t) / bw, step_flops(c, B, t) / peak) for t in range(1, T + 1))


def decoder_params(c) -> int:
    d, f, L, V = c.d, c.d_ffn, c.n_layers, c.vocab
    return L * (6 * d * d + 3 * d * f) + 2 * d * d + V * d


BPTT_BLOCK = 16   # steps per weight/memory-gradient block of rlt_bptt


def bptt_bytes(c, B, n, S=BPTT_BLOCK):
    """Algorithmic HBM bytes of one rlt_bptt call over n steps (full BPTT,
    memory gradient included), as its schedule moves them:
      recording step t: the forward step without the head, plus the writes of
        position t's keys/values, every layer's cross-attention output and LSE;
      reverse step t: the decoder weights twice (recomputation with the head
        but without the last layer's W_2, whose output s_t is recorded, and
        the transposed copies of dX = dY W), the window keys/values twice
        (recomputation and backward), the fp32 query-side records (query and
        output gradient) of the min(W, n - t + 1) positions whose queries read
        position t's key, the recorded cross-attention outputs, the memory
        keys/values of positions 1..t per layer (the query gradient);
      per block of S steps: every fp32 weight gradient read and written, and
        per memory group the memory keys/values of positions 1..p_hi read once
        and their fp32 gradient read and written."""
    es = 2 if c.dtype == "bf16" else 4
    d, L, H, V, W = c.d, c.n_layers, c.n_heads, c.vocab, c.window
    wb = decoder_weight_bytes(c)
    head = es * V * d
    total = 0
    for t in range(1, n + 1):
        win = min(W, t)
        swa = es * B * L * win * 2 * d
        mem = L * xattn_bytes(c, B, t)
        rec = (wb - head) + swa + mem + es * B * L * (2 * d + d) + 4 * B * L * H + 4 * B * d * 2
        nrec = min(W, n - t + 1)
        rev = 2 * wb - es * d * c.d_ffn + 2 * swa + 8 * B * L * nrec * d + es * B * L * d + mem + 4 * B * d * 2
        total += rec + rev
    for p_hi in range(n - 1, -1, -S):
        total += 8 * decoder_params(c) + c.mem_groups * 2 * B * (p_hi + 1) * d * (es + 8)
    return total


def bptt_flops(c, B, n):
    """Algorithmic flops of one rlt_bptt call: the decoder GEMMs four times per
    step (recording, recomputation, dX = dY W, dW += dY^T X) and the
    attention three times (forward, the backward's two products per key, the
    memory gradient's two per key)."""
    d, f, L, V = c.d, c.d_ffn, c.n_layers, c.vocab
    gemm = 2 * B * (L * (6 * d * d + 3 * d * f) + 2 * d * d + V * d)
    tot = 0
    for t in range(1, n + 1):
        attn = 4 * B * d * L * (min(c.window, t) + t)
        tot += 4 * gemm + 3 * attn
    return tot


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return j["hbm_gbs"] * 1e9, j["bf16_tflops"] * 1e12, "measured"
    return 6.4e12, 1.8e15, "fallback"


# ---------------------------------------------------------------------------
# clocks sampling during the timed region

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ---------------------------------------------------------------------------
# the GPU arm

# ---------------------------------------------------------------------------
# replicas: host-side logic of the N > 1 path (also run with gloo on CPU)

RANK_SEED_STRIDE = 7919


def rank_inputs(wl, rank):
    """This rank's sequences: tokens, prompt/response splits and the scored
    actions (teacher-forced next tokens), from a seed offset by the rank, so
    that ranks hold disjoint draws of the same workload (weak scaling)."""
    seed = wl.seed + RANK_SEED_STRIDE * rank
    tok = ri.make_tokens(wl, seed=seed)
    prompt = ri.make_splits(wl, seed=seed)
    acts = ri.teacher_actions(tok, 0, wl.T, None if wl.score_prompt else prompt)
    return tok, prompt, acts


def max_over_ranks(values, world, device=None):
    """Element-wise maximum of a list of per-rank timings over all ranks (the
    slowest rank times the job)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    v = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(v, op=dist.ReduceOp.MAX)
    return v.tolist()


def segments(T, K):
    """K consecutive position ranges (p0, n) that cover positions 0..T-1 once:
    one bench step is one rlt_decode_steps call over a range, with the state
    carried from the previous step (Proposition 3.1: splitting a decode into
    calls leaves the state unchanged).  The first T % K ranges are one longer."""
    if not 1 <= K <= T:
        raise SystemExit(f"--steps must be between 1 and T = {T}")
    q, r = divmod(T, K)
    out, p = [], 0
    for k in range(K):
        n = q + (1 if k < r else 0)
        out.append((p, n))
        p += n
    return out


def workload_config(wl, world, steps):
    """The `config` object of the bench line (both arms)."""
    c = wl.cfg
    n = -(-wl.T // steps)
    return {"workload": f"{wl.name}: d={c.d} L_E=L_D={c.n_layers} H={c.n_heads}x{c.head_dim} f={c.d_ffn}"
                        f" W={c.window} G={c.mem_groups} V={c.vocab}",
            "B_per_gpu": wl.B, "T": wl.T, "global_batch": wl.B * world, "parallelism": f"replicas{world}",
            "step": f"one rlt_decode_steps call advancing all B sequences by <= {n} positions with the state "
                    f"carried, so the {steps} timed steps consume positions 1..{wl.T} exactly once; the token-"
                    f"parallel encode of all {wl.T} positions runs once at the start of the timed region",
            "l2": "flushed before the encode and before every step (256 MB write)"}


def job_throughput(B, T, world, t_step):
    """Whole-job decoder tokens/s: every rank's B x T tokens over the slowest
    rank's step time."""
    return B * T * world / t_step


def run_gpu(args, rank, world, local_rank):
    """The GPU arm.  The timed region is one pass over the workload: state
    init and the token-parallel encode of all T positions (timed on their
    own), then K steps, each one rlt_decode_steps call over the next range of
    positions of all B sequences with the state carried, so the K steps
    consume positions 1..T exactly once.  Warm-up steps run the first ranges
    on a separate state."""
    import torch
    import torch.distributed as dist
    import recurrent_looped_transformer_rlt_b300 as rlt
    from recurrent_looped_transformer_rlt_b300 import runner

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = ri.preset(args.workload)
    c = wl.cfg
    B, T = wl.B, wl.T
    segs = segments(T, args.steps)
    # weights: seeded numpy draws (identical on every rank); tokens: this rank's sequences
    W = ri.make_weights(c, wl.seed)
    tok, prompt, acts = rank_inputs(wl, rank)
    model = rlt.Model(c, W, device=dev)
    del W
    model.set_decode_path(args.decode_path)
    if args.decode_path == "fused" and model.fused_plan(B) is None:
        raise SystemExit(f"the fused decoder does not take the {wl.name} model (rlt_fused_plan)")
    stream = torch.cuda.current_stream()
    buf = runner.alloc_buffers(model, B, T)
    tok_d = torch.from_numpy(tok).to(dev)
    # per step: its actions [B][n] and outputs (rlt_decode_steps takes row pitch n)
    acts_d = [torch.from_numpy(np.ascontiguousarray(acts[:, p0:p0 + n])).to(dev) for p0, n in segs]
    outs = [runner.StepOutputs(torch.empty(B, n, device=dev), torch.empty(B, n, device=dev),
                               torch.empty(B, n, dtype=torch.int32, device=dev), None) for _, n in segs]
    st = rlt.State(model, B)
    st_w = rlt.State(model, B)   # warm-up and instrumented passes
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def encode(state, tok_dev):
        rlt.rlt_state_init(model.handle, state.c, stream)
        rlt.rlt_encode(model.handle, tok_dev, B, T, buf.e, buf.mem, buf.ws, buf.ws.numel(), stream)

    def step(state, k, act_dev=None):
        p0, n = segs[k]
        assert state.c.pos == p0
        o = outs[k]
        rlt.rlt_decode_steps(model.handle, state.c, buf.e, buf.mem, T, n,
                             acts_d[k] if act_dev is None else act_dev, wl.temperature, wl.top_k,
                             o.logp, o.logp_full, o.argmax, (), None, buf.ws, buf.ws.numel(), stream)

    def full_pass(state):
        encode(state, tok_d)
        for k in range(len(segs)):
            step(state, k)

    # warm-up: the first ranges on a separate state (a fresh pass whenever one ends)
    k = len(segs)
    for _ in range(args.warmup):
        if k == len(segs):
            encode(st_w, tok_d)
            k = 0
        step(st_w, k)
        k += 1
    torch.cuda.synchronize()
    if rlt.rlt_status(buf.ws, stream) != 0:
        raise RuntimeError("device status flag set during warm-up")

    def barrier():
        if world > 1:
            dist.barrier()

    # timed region: the encode, then K steps; inputs resident in HBM, L2
    # flushed before the encode and before every step, CUDA events on the
    # launching stream around each
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(len(segs) + 1)]
    launches0 = rlt.rlt_launch_count()
    with ClockSampler(local_rank) as clk:
        barrier()
        torch.cuda.synchronize()
        flush.fill_(1.0)
        ev[0][0].record(stream)
        encode(st, tok_d)
        ev[0][1].record(stream)
        for k in range(len(segs)):
            flush.fill_(1.0)
            ev[k + 1][0].record(stream)
            step(st, k)
            ev[k + 1][1].record(stream)
        torch.cuda.synchronize()
        barrier()
    launches = rlt.rlt_launch_count() - launches0
    t_enc = ev[0][0].elapsed_time(ev[0][1]) / 1e3
    times = [a.elapsed_time(b) / 1e3 for a, b in ev[1:]]
    if rlt.rlt_status(buf.ws, stream) != 0:
        raise RuntimeError("device status flag set in the timed region")
    assert st.c.pos == T
    lp = np.concatenate([o.logp.cpu().numpy() for o in outs], axis=1)
    assert np.isfinite(lp[acts >= 0]).sum() > 0
    # per-launch durations of the roofline kernel: one more pass with CUDA
    # events around each launch of that kernel class, outside the timed steps
    # (an event between two kernels of the step graph suspends their
    # programmatic overlap, so the instrumented pass runs slower than the
    # timed one)
    kernel_ms = []
    fused = args.decode_path == "fused"
    if args.kernel_class and not fused:  # the per-launch timers instrument the graph path's step
        model.timer_arm(args.kernel_class, min(T * c.n_layers, 1 << 18))  # one launch per layer and step
        full_pass(st_w)
        torch.cuda.synchronize()
        kernel_ms = model.timer_read()  # reading disarms the timer
    # the projections' per-launch durations too, when a decoder step is cheap
    # (the projections dominate the small workload's step time); a failure
    # here only drops the extra object
    proj_ms = []
    if args.kernel_class and not fused and c.dtype == "bf16" and sum(times) / T < 1e-3:
        try:
            model.timer_arm("gemm", min(T * (6 * c.n_layers + 2), 1 << 18))
            full_pass(st_w)
            torch.cuda.synchronize()
            proj_ms = model.timer_read()
        except Exception:  # noqa: BLE001
            proj_ms = []
            try:
                rlt.rlt_timer_arm(model.handle, 0, 0)  # leave the timer off for the end-to-end pass
            except Exception:  # noqa: BLE001
                pass

    # end to end through the public API, the same pass: host tokens in (pinned),
    # then per step its host actions in and its host log-probabilities out
    tok_h = torch.from_numpy(tok).pin_memory()
    acts_h = [torch.from_numpy(np.ascontiguousarray(acts[:, p0:p0 + n])).pin_memory() for p0, n in segs]
    lp_h = [torch.empty(B, n, dtype=torch.float32).pin_memory() for _, n in segs]
    tok_e = torch.empty_like(tok_d)
    acts_e = [torch.empty_like(a) for a in acts_d]
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    tok_e.copy_(tok_h, non_blocking=True)
    encode(st_w, tok_e)
    for k in range(len(segs)):
        acts_e[k].copy_(acts_h[k], non_blocking=True)
        step(st_w, k, acts_e[k])
        lp_h[k].copy_(outs[k].logp, non_blocking=True)
    torch.cuda.synchronize()
    t_e2e = time.perf_counter() - t0
    barrier()
    if rlt.rlt_status(buf.ws, stream) != 0:
        raise RuntimeError("device status flag set in the end-to-end pass")

    t_dec = float(sum(times))
    t_dec, t_enc, t_e2e, t_max_step = max_over_ranks([t_dec, t_enc, t_e2e, max(times)], world, dev)
    K = len(segs)
    res = dict(t_step=(t_enc + t_dec) / K, t_dec=t_dec, t_enc=t_enc, t_e2e=t_e2e, t_max_step=t_max_step,
               launches=launches // K, clocks=clk.summary(), kernel_ms=kernel_ms, proj_ms=proj_ms, B=B, T=T, wl=wl,
               K=K, h2d=(tok.nbytes + acts.nbytes) / K, d2h=B * T * 4 / K)
    model.close()
    return res


# DRAM traffic of the cross-attention kernel, from one ncu capture of the
# current kernel build at the workload's shapes (bench.py --profile-case xattn;
# summaries in profiles/): (dram__bytes_read.sum + dram__bytes_write.sum,
# algorithmic bytes of that launch).  The bench reports traffic per launch as
# its average algorithmic bytes times this ratio.
XATTN_TRAFFIC = {
    "refdep": (1075496192 + 3594496, 1074528256),   # t = 2048, ring depth 2
}


def kernel_roofline(wl, kernel_ms, kernel_class, bw, peak, src):
    """Roofline object of the timed kernel class from its per-launch CUDA-event durations."""
    if not kernel_ms:
        return None
    c, B, T = wl.cfg, wl.B, wl.T
    L = c.n_layers
    if kernel_class == "xattn":
        # launch j of the timed region: step t = j // L + 1 (steps cycle 1..T per pass)
        byts = [xattn_bytes(c, B, (j // L) % T + 1) + B * c.d * 4 + B * c.d * 2 for j in range(len(kernel_ms))]
    else:
        return None
    ach = sum(byts) / (sum(kernel_ms) / 1e3)
    traffic = None
    if wl.name in XATTN_TRAFFIC:
        dram, alg = XATTN_TRAFFIC[wl.name]
        traffic = int(round(float(np.mean(byts)) * dram / alg))
    return {"bound": "hbm", "achieved": round(ach / 1e9, 1), "peak": round(bw / 1e9, 1), "unit": "GB/s",
            "frac": round(ach / bw, 4), "traffic": traffic, "kernel": "dec_xattn (partial + combine)",
            "launches": len(kernel_ms), "avg_us": round(1e3 * float(np.mean(kernel_ms)), 2),
            "peak_source": src, "durations": "CUDA events around every launch of one extra pass over all T positions "
                                             "after the timed steps"}


def fused_roofline(wl, t_dec, bw, src, launches=1):
    """Roofline object of the persistent decoder kernel: one launch runs a
    whole decode call, so the algorithmic bytes of the launches of one pass
    are every step's (weights, memory K/V of positions 1..t, window, state)
    and their duration is the decode part of the pass (CUDA events around the
    decode calls)."""
    c, B, T = wl.cfg, wl.B, wl.T
    byts = sum(step_bytes(c, B, t) for t in range(1, T + 1))
    ach = byts / t_dec
    return {"bound": "hbm", "achieved": round(ach / 1e9, 1), "peak": round(bw / 1e9, 1), "unit": "GB/s",
            "frac": round(ach / bw, 4), "traffic": None, "kernel": "dec_fused (all steps of the call)",
            "launches": launches, "avg_us": round(1e6 * t_dec / launches, 2), "peak_source": src,
            "durations": "CUDA events around the decode calls of the timed steps"}


def projection_bytes(c, B):
    """Algorithmic bytes of each decoder projection launch of one bf16 step, in
    launch order: the gate, then per layer QKV, O, Qx, Ox, W_1/W_3, W_2, then
    the head.  Weights once, the A operand once, the outputs once, and the
    residual stream read and written by the residual projections."""
    d, f, V, L = c.d, c.d_ffn, c.vocab, c.n_layers
    res = 2 * B * d * 4
    per = [d * 2 * d * 2 + B * 2 * d * 2 + B * d * 2 + res]                  # gate + merge (e in, s in/h out)
    per += [3 * d * d * 2 + B * d * 2 + B * d * 4 + 2 * B * d * 2,          # QKV: q fp32, k and v to the ring
            d * d * 2 + B * d * 2 + res,                                    # O + residual
            d * d * 2 + B * d * 2 + B * d * 4,                              # Qx
            d * d * 2 + B * d * 2 + res,                                    # Ox + residual
            2 * f * d * 2 + B * d * 2 + B * f * 2,                          # W_1, W_3 + SwiGLU
            d * f * 2 + B * f * 2 + res] * L                                # W_2 + residual
    per += [V * d * 2 + B * d * 2 + B * V * 4]                              # head
    return per


def projection_roofline(wl, kernel_ms, bw, src):
    """Roofline object of the decoder projections from per-launch durations in
    launch order (every projection launch of whole steps)."""
    if not kernel_ms:
        return None
    per = projection_bytes(wl.cfg, wl.B)
    byts = [per[j % len(per)] for j in range(len(kernel_ms))]
    ach = sum(byts) / (sum(kernel_ms) / 1e3)
    return {"bound": "hbm", "achieved": round(ach / 1e9, 1), "peak": round(bw / 1e9, 1), "unit": "GB/s",
            "frac": round(ach / bw, 4), "traffic": None, "kernel": "gemm_tc_kernel (all decoder projections)",
            "launches": len(kernel_ms), "avg_us": round(1e3 * float(np.mean(kernel_ms)), 2),
            "peak_source": src, "durations": "CUDA events around every projection launch of one extra step"}


# ---------------------------------------------------------------------------
# the CPU oracle (baseline / reference arm)

# Bounded oracle samples (sequences, positions from the start of a sequence)
# per workload: the GPU arm's cpu_baseline (about 10-30 s of host work on
# 16 cores) and each step of the reference arm (a few seconds).  The float64
# oracle converts every weight matrix it touches per step, so the deep
# configurations get short prefixes.
ORACLE_BASELINE = {"tiny": (8, 64), "small": (2, 512), "medium": (1, 96), "refdep": (1, 6), "rlreplay": (1, 64)}
ORACLE_STEP = {"tiny": (8, 64), "small": (1, 128), "medium": (1, 16), "refdep": (1, 2), "rlreplay": (1, 16)}


class OracleSampler:
    """The oracle, as it stands, on bounded samples of a workload: the weights
    are drawn once; each sample encodes, decodes and scores B_sub sequences of
    T_sub positions (the workload's temperature and top-k)."""

    def __init__(self, wl):
        from oracle import rlt_oracle as O
        self.O = O
        self.wl = wl
        self.c = O.Cfg.of(wl.cfg)
        self.W = ri.make_weights(wl.cfg, wl.seed)

    def run(self, B_sub, T_sub):
        wl = self.wl
        tok = ri.make_tokens(wl, B=B_sub, T=T_sub)
        acts = ri.teacher_actions(tok, 0, T_sub)
        t0 = time.perf_counter()
        self.O.run_sequence(self.c, self.W, tok, acts, wl.temperature, wl.top_k)
        dt = time.perf_counter() - t0
        return B_sub * T_sub / dt, f"{B_sub} seq x {T_sub} positions (encode + decode + scoring), float64 numpy", dt


def oracle_sample(wl):
    """Time the oracle on the cpu_baseline sample of the workload.  Returns
    tokens/s, the sample and its duration."""
    return OracleSampler(wl).run(*ORACLE_BASELINE[wl.name])


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args, rank):
    """The reference arm: the oracle on the host cores (rank 0 only), each
    step one bounded sample of the workload (ORACLE_STEP), the weights drawn
    once before the timed steps."""
    wl = ri.preset(args.workload)
    if rank != 0:
        return
    sampler = OracleSampler(wl)
    B_sub, T_sub = ORACLE_STEP[wl.name]
    vals, dts = [], []
    sample = ""
    for _ in range(max(args.steps, 1)):
        v, sample, dt = sampler.run(B_sub, T_sub)
        vals.append(v)
        dts.append(dt)
    v = B_sub * T_sub * len(dts) / float(np.sum(dts))
    line = {"metric": METRIC, "value": round(v, 3), "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * float(np.mean(dts)), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": workload_config(wl, args.gpus, min(max(args.steps, 1), wl.T)),
            "cpu_baseline": {"value": round(v, 3), "unit": UNIT, "cores": cores_used(), "kind": "oracle",
                             "sample": sample + " per step"},
            "e2e": {"value": round(v, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# single-kernel cases (for profiler captures): one decoder-step launch of the
# chosen kernel at the workload's shapes, through the public entry points

def run_profile_case(args):
    """Cross-attention ("xattn", memory positions 1..T/2), window attention
    ("swa", the ring of W entries) or a projection ("proj": W_qkv at M = B,
    "glu": the W_1/W_3 pair) of the workload, timed over --steps launches
    after --warmup; prints one JSON line with the algorithmic bytes per launch
    and the achieved bandwidth."""
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    wl = ri.preset(args.workload)
    c, B = wl.cfg, wl.B
    if c.dtype != "bf16":
        raise SystemExit("profile cases cover bf16 workloads")
    # a one-layer model of the workload's widths (the cases do not use the other layers)
    c1 = ri.preset(args.workload, n_layers=1, mem_groups=1, vocab=256).cfg
    g = torch.Generator(device="cuda").manual_seed(0)
    W = {}
    for n_, shape, kind in ri.weight_specs(c1):
        if kind == "mat":
            W[n_] = (torch.randn(shape, device="cuda", generator=g) * c1.sigma).to(torch.bfloat16)
        elif kind == "ones":
            W[n_] = torch.ones(shape, device="cuda")
        else:
            W[n_] = torch.randn(shape, device="cuda", generator=g) * 0.02
    model = rlt.Model(c1, W)
    d, H, hd = c.d, c.n_heads, c.head_dim
    stream = torch.cuda.current_stream()
    bw, _, src = load_peaks()
    case = args.profile_case
    if case in ("xattn", "swa"):
        T_mem = wl.T if case == "xattn" else c.window
        t = wl.T // 2 if case == "xattn" else c.window
        mk = torch.randn(B, H, T_mem, hd, device="cuda", generator=g).to(torch.bfloat16)
        mv = torch.randn(B, H, T_mem, hd, device="cuda", generator=g).to(torch.bfloat16)
        q = torch.randn(B, d, device="cuda", generator=g)
        out = torch.empty(B, d, device="cuda", dtype=torch.bfloat16)
        ws = model.workspace(B, T_mem)

        def launch():
            rlt.rlt_cross_attention(model.handle, q, mk, mv, B, T_mem, t, out, ws, ws.numel(), stream)
        nbytes = 2 * B * t * 2 * d + B * d * 4 + B * d * 2
        kernel = "dec_xattn_kernel"
        shape = f"B={B} H={H} hd={hd} T_mem={T_mem} t={t}"
    else:
        M, K = B, d
        N = 3 * d if case == "proj" else c.d_ffn
        A = (torch.randn(M, K, device="cuda", generator=g)).to(torch.bfloat16)
        Wm = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        W3 = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16) if case == "glu" else None
        Cm = torch.empty(M, N, device="cuda")
        ws = model.workspace(1, 1)

        def launch():
            rlt.rlt_linear(model.handle, A, K, M, K, Wm, W3, K, N, Cm, N, ws, ws.numel(), stream)
        nbytes = (2 if W3 is not None else 1) * N * K * 2 + M * K * 2 + M * N * 4
        kernel = "gemm_tc_kernel"
        shape = f"M={M} K={K} N={N}" + (" (W_1, W_3 pair)" if W3 is not None else "")
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    if rlt.rlt_status(ws, stream) != 0:
        raise RuntimeError("device status flag set")
    t_avg = float(np.mean(ts))
    print(json.dumps({"case": case, "workload": wl.name, "kernel": kernel, "shape": shape,
                      "bytes_per_launch": nbytes, "us_per_launch": round(1e6 * t_avg, 2),
                      "achieved_gbs": round(nbytes / t_avg / 1e9, 1), "peak_gbs": round(bw / 1e9, 1),
                      "frac": round(nbytes / t_avg / bw, 4), "peak_source": src, "l2": "flushed before each launch"}),
          flush=True)
    model.close()


def run_fused_case(args):
    """One rlt_decode_steps call over n = --bptt-steps (default 32) steps from
    the middle of the workload's sequences (the state is brought to position
    --case-pos, default T/2 - n/2, first and restored before each timed
    call), timed with CUDA events over --steps calls after --warmup; one JSON
    line with the call's algorithmic bytes and its fraction of HBM
    bandwidth.  Case "fused": the persistent cluster decoder (one launch, for
    ncu captures); case "decode": the path --decode-path names.  For small
    profiler captures of one kernel at the workload's widths, --case-layers
    L and --case-T T build an L-layer model (one memory group) over T
    positions instead of the workload's."""
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    from recurrent_looped_transformer_rlt_b300 import runner
    over = {}
    if args.case_layers:
        over.update(n_layers=args.case_layers, mem_groups=1)
    if args.case_T:
        over.update(T=args.case_T)
    wl = ri.preset(args.workload, **over)
    c, B, T = wl.cfg, wl.B, wl.T
    n = args.bptt_steps or 32
    p0 = args.case_pos if args.case_pos >= 0 else max(0, T // 2 - n // 2)
    if p0 + n > T:
        raise SystemExit("--case-pos + steps beyond T")
    path = "fused" if args.profile_case == "fused" else args.decode_path
    W = ri.make_weights(c, wl.seed)
    tok = ri.make_tokens(wl)
    model = rlt.Model(c, W)
    del W
    model.set_decode_path(path)
    plan = model.fused_plan(B) if path == "fused" else None
    if path == "fused" and plan is None:
        raise SystemExit(f"the fused decoder does not take the {wl.name} model")
    buf = runner.alloc_buffers(model, B, T)
    runner.encode(model, torch.from_numpy(tok).cuda(), buf)
    acts = torch.from_numpy(ri.teacher_actions(tok, 0, T)).cuda()
    st = runner.new_state(model, B)
    if p0 > 0 and args.case_synthetic_state:
        # timing only: a seeded random state at position p0 (s ~ N(0, 1),
        # window entries ~ N(0, 1) in storage precision) instead of p0 decoded
        # steps; no kernel's work depends on the values
        g = torch.Generator(device="cuda").manual_seed(p0)
        st.s.copy_(torch.randn(st.s.shape, device="cuda", generator=g))
        st.ring_k.copy_(torch.randn(st.ring_k.shape, device="cuda", generator=g).to(st.ring_k.dtype))
        st.ring_v.copy_(torch.randn(st.ring_v.shape, device="cuda", generator=g).to(st.ring_v.dtype))
        st.c.pos = p0
    elif p0 > 0:
        runner.decode(model, st, buf, p0, acts[:, :p0].contiguous())
    saved = (st.s.clone(), st.ring_k.clone(), st.ring_v.clone())
    a_n = acts[:, p0:p0 + n].contiguous()
    out = runner.StepOutputs(torch.empty(B, n, device="cuda"), torch.empty(B, n, device="cuda"),
                             torch.empty(B, n, dtype=torch.int32, device="cuda"), None)
    stream = torch.cuda.current_stream()
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    ts = []
    for it in range(args.warmup + args.steps):
        st.s.copy_(saved[0])
        st.ring_k.copy_(saved[1])
        st.ring_v.copy_(saved[2])
        st.c.pos = p0
        flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        runner.decode(model, st, buf, n, a_n, wl.temperature, wl.top_k, out=out)
        e1.record(stream)
        e1.synchronize()
        if it >= args.warmup:
            ts.append(e0.elapsed_time(e1) / 1e3)
    if runner.status(buf) != 0:
        raise RuntimeError("device status flag set")
    bw, _, src = load_peaks()
    t = float(np.mean(ts))
    nbytes = sum(step_bytes(c, B, p + 1) for p in range(p0, p0 + n))
    print(json.dumps({"case": args.profile_case, "workload": wl.name, "decode_path": path,
                      "kernel": "dec_fused_kernel" if path == "fused" else "decoder step graph", "B": B, "p0": p0,
                      "steps": n, "plan": (None if plan is None else
                                           {"cluster": plan[0], "seqs_per_cluster": plan[1], "clusters": plan[2],
                                            "smem_bytes": plan[3]}),
                      "us_per_call": round(1e6 * t, 2), "us_per_step": round(1e6 * t / n, 2),
                      "bytes_per_call": nbytes, "achieved_gbs": round(nbytes / t / 1e9, 1),
                      "peak_gbs": round(bw / 1e9, 1), "frac": round(nbytes / t / bw, 4), "peak_source": src,
                      "l2": "flushed before each call"}), flush=True)
    model.close()


def run_encode_case(args):
    """The token-parallel encoder alone (rlt_encode of B sequences of T
    positions) on a model of the workload's widths with --case-layers layers
    (default 1), timed with CUDA events over --steps calls after --warmup;
    --case-batch overrides B (smaller captures).  One JSON line with the
    algorithmic flops per layer (projections and causal attention) and the
    rate."""
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    from recurrent_looped_transformer_rlt_b300 import runner
    L = args.case_layers or 1
    wl = ri.preset(args.workload, n_layers=L, mem_groups=1, vocab=256)
    c = wl.cfg
    B = args.case_batch or wl.B
    T = wl.T
    W = ri.make_weights(c, wl.seed)
    tok = torch.from_numpy(ri.make_tokens(wl, B=B, T=T)).cuda()
    model = rlt.Model(c, W)
    buf = runner.alloc_buffers(model, B, T)
    stream = torch.cuda.current_stream()
    ts = []
    for it in range(args.warmup + args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        runner.encode(model, tok, buf)
        e1.record(stream)
        e1.synchronize()
        if it >= args.warmup:
            ts.append(e0.elapsed_time(e1) / 1e3)
    if runner.status(buf) != 0:
        raise RuntimeError("device status flag set")
    t = float(np.mean(ts))
    d, f, H, hd = c.d, c.d_ffn, c.n_heads, c.head_dim
    R = B * T
    gemm = 2 * R * (6 * d * d + 3 * d * f) * L + 2 * R * 2 * d * d  # layers + the memory projection
    attn = 4 * B * H * T * T * hd // 2 * L                          # causal: half of Q K^T and P V
    _, peak, src = load_peaks()
    print(json.dumps({"case": "encode", "workload": wl.name, "layers": L, "B": B, "T": T, "head_dim": hd,
                      "ms_per_call": round(1e3 * t, 3), "gemm_flops": gemm, "attn_flops": attn,
                      "tflops": round((gemm + attn) / t / 1e12, 1), "peak_tflops": round(peak / 1e12, 1),
                      "peak_source": src, "calls": len(ts)}), flush=True)
    model.close()


def run_bptt_case(args):
    """Backpropagation through time (rlt_bptt) over the first --bptt-steps
    positions of the workload's sequences (encoded on the GPU), full BPTT with
    the memory gradient, timed with CUDA events over --steps calls after
    --warmup; one JSON line with the call's algorithmic bytes and flops, its
    roofline time and the kernels it launched."""
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    from recurrent_looped_transformer_rlt_b300 import runner
    wl = ri.preset(args.workload)
    c, B = wl.cfg, wl.B
    n = args.bptt_steps or wl.T // 4
    T = max(n, 1)
    W = ri.make_weights(c, wl.seed)
    tok = ri.make_tokens(wl, B=B, T=T)
    model = rlt.Model(c, W)
    buf = runner.alloc_buffers(model, B, T)
    runner.encode(model, torch.from_numpy(tok).cuda(), buf)
    acts = torch.from_numpy(ri.teacher_actions(tok, 0, n)).cuda()
    nb = rlt.rlt_bptt_workspace_size(model.handle, B, n)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    rlt.rlt_workspace_init(ws, nb)
    stream = torch.cuda.current_stream()
    res = None
    ts, launches = [], 0
    for it in range(args.warmup + args.steps):
        torch.cuda.synchronize()
        l0 = rlt.rlt_launch_count()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        res = runner.bptt(model, buf, acts, ws=ws, stream=stream)
        e1.record(stream)
        e1.synchronize()
        if it >= args.warmup:
            ts.append(e0.elapsed_time(e1) / 1e3)
            launches = rlt.rlt_launch_count() - l0
    if rlt.rlt_status(ws, stream) != 0:
        raise RuntimeError("device status flag set")
    bw, peak, src = load_peaks()
    t = float(np.mean(ts))
    nbytes, nflops = bptt_bytes(c, B, n), bptt_flops(c, B, n)
    roof = max(nbytes / bw, nflops / peak)
    hbm = nbytes / bw >= nflops / peak
    roofline = {"bound": "hbm" if hbm else "tensor",
                "achieved": round((nbytes / t / 1e9) if hbm else (nflops / t / 1e12), 1),
                "peak": round(bw / 1e9, 1) if hbm else round(peak / 1e12, 1),
                "unit": "GB/s" if hbm else "TFLOP/s",
                "frac": round(roof / t, 4), "traffic": None, "kernel": "rlt_bptt (whole call)",
                "peak_source": src}
    print(json.dumps({"case": "bptt", "workload": wl.name, "B": B, "steps": n, "block": min(BPTT_BLOCK, n),
                      "tokens_per_s": round(B * n / t, 1), "ms_per_call": round(1e3 * t, 3),
                      "loss": float(res.loss.item()), "bytes_per_call": nbytes, "flops_per_call": nflops,
                      "roofline_ms": round(1e3 * roof, 3), "roofline": roofline,
                      "gpu_launches": int(launches), "calls": len(ts),
                      "timing": "CUDA events around rlt_bptt (recording pass, reverse pass, block flushes)"}),
          flush=True)
    model.close()


def run_generate_case(args):
    """Generation throughput of the workload's model: prefill of the first
    half of each sequence (token-parallel encoder keeping its keys and values,
    decoder over the prompt), then rlt_generate of the second half, timed with
    CUDA events over --steps calls after --warmup; one JSON line."""
    import torch
    import recurrent_looped_transformer_rlt_b300 as rlt
    from recurrent_looped_transformer_rlt_b300 import runner
    wl = ri.preset(args.workload)
    c, B, T = wl.cfg, wl.B, wl.T
    if c.dtype != "bf16":
        raise SystemExit("generation covers bf16 workloads")
    T0, n = T // 2, T - T // 2
    W = ri.make_weights(c, wl.seed)
    tok = ri.make_tokens(wl, B=B, T=T0)
    model = rlt.Model(c, W)
    model.set_decode_path(args.decode_path)  # the prompt's decode and the generation both take it
    dt = model.dtype
    e = torch.empty(B, T, c.d, dtype=dt, device="cuda")
    mem = torch.empty(c.mem_groups, 2, B, c.n_heads, T, c.head_dim, dtype=dt, device="cuda")
    kv = torch.empty(c.n_layers, 2, B, c.n_heads, T, c.head_dim, dtype=dt, device="cuda")
    ws = model.workspace(B, T)
    tok_d = torch.from_numpy(tok).cuda()
    acts = torch.from_numpy(ri.teacher_actions(tok, 0, T0)).cuda()
    lp0 = torch.empty(B, T0, device="cuda")
    toks = torch.empty(B, n, dtype=torch.int32, device="cuda")
    lp = torch.empty(B, n, device="cuda")
    stream = torch.cuda.current_stream()

    def prefill():
        rlt.rlt_encode_kv(model.handle, tok_d, B, T0, T, e, mem, kv, ws, ws.numel(), stream)
        st = runner.new_state(model, B, stream)
        rlt.rlt_decode_steps(model.handle, st.c, e, mem, T, T0, acts, 1.0, 0, lp0, None, None, (), None, ws,
                             ws.numel(), stream)
        return st
    ts = []
    for it in range(args.warmup + args.steps):
        st = prefill()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        rlt.rlt_generate(model.handle, st.c, e, mem, kv, T, n, 1234 + it, wl.temperature, wl.top_k, toks, lp, ws,
                         ws.numel(), stream)
        e1.record(stream)
        e1.synchronize()
        if it >= args.warmup:
            ts.append(e0.elapsed_time(e1) / 1e3)
    if rlt.rlt_status(ws, stream) != 0:
        raise RuntimeError("device status flag set")
    t = float(np.mean(ts))
    print(json.dumps({"case": "generate", "workload": wl.name, "decode_path": args.decode_path, "B": B,
                      "prompt": T0, "generated": n,
                      "tokens_per_s": round(B * n / t, 1), "us_per_token_step": round(1e6 * t / n, 2),
                      "calls": len(ts), "temperature": wl.temperature, "top_k": wl.top_k,
                      "timing": "CUDA events around rlt_generate (graph capture and all generated steps)"}),
          flush=True)
    model.close()


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="rlt", choices=["rlt", "reference"])
    ap.add_argument("--workload", default="refdep", choices=sorted(ri.PRESETS))
    ap.add_argument("--kernel-class", default="xattn", choices=["xattn", ""])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-path", default="graph", choices=["graph", "fused"],
                    help="decoder path of rlt_decode_steps: the per-step graph or the persistent cluster kernel")
    ap.add_argument("--profile-case", default="",
                    choices=["", "xattn", "swa", "proj", "glu", "generate", "bptt", "fused", "decode", "encode"],
                    help="time one kernel of the workload (profiler captures), generation, the decoder's "
                         "backpropagation through time, or one call of the persistent decoder, instead of the "
                         "bench step")
    ap.add_argument("--bptt-steps", type=int, default=0,
                    help="steps of the bptt case (default: T / 4) and of the fused / decode cases (default: 32)")
    ap.add_argument("--case-pos", type=int, default=-1,
                    help="first position of the fused / decode cases (default: T/2 - steps/2)")
    ap.add_argument("--case-layers", type=int, default=0,
                    help="layers of the encode case (default 1), or of the decode case (default: the workload's)")
    ap.add_argument("--case-T", type=int, default=0, help="positions of the decode case (default: the workload's)")
    ap.add_argument("--case-batch", type=int, default=0, help="sequences of the encode case (default: the workload's)")
    ap.add_argument("--case-synthetic-state", action="store_true",
                    help="fused / decode cases: start from a seeded random state at --case-pos instead of "
                         "decoding up to it (timing and profiler captures only)")
    args = ap.parse_args()
    if args.profile_case == "generate":
        run_generate_case(args)
        return
    if args.profile_case == "bptt":
        run_bptt_case(args)
        return
    if args.profile_case in ("fused", "decode"):
        run_fused_case(args)
        return
    if args.profile_case == "encode":
        run_encode_case(args)
        return
    if args.profile_case:
        run_profile_case(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    r = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        wl, B, T = r["wl"], r["B"], r["T"]
        bw, peak, src = load_peaks()
        n_tok = B * T * world
        t_pass = r["t_enc"] + r["t_dec"]
        value = job_throughput(B, T, world, t_pass)
        roof_s = decode_roofline_s(wl.cfg, B, T, bw, peak)
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * r["t_step"], 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.cfg.dtype, "data": "synthetic",
            "config": workload_config(wl, world, r["K"]),
            "decode_ms": round(1e3 * r["t_dec"], 3),
            "encode_ms": round(1e3 * r["t_enc"], 3),
            "decoder_tokens_per_s": round(n_tok / r["t_dec"], 1),
            "max_step_ms": round(1e3 * r["t_max_step"], 3),
            "decode_roofline_ms": round(1e3 * roof_s, 3),
            "decode_roofline_frac": round(roof_s / r["t_dec"], 4),
            "roofline": (fused_roofline(wl, r["t_dec"], bw, src, r["K"]) if args.decode_path == "fused"
                         else kernel_roofline(wl, r["kernel_ms"], args.kernel_class, bw, peak, src)),
            "decode_path": args.decode_path,
            "e2e": {"value": round(n_tok / r["t_e2e"], 1), "unit": UNIT, "h2d_bytes_per_step": int(r["h2d"]),
                    "d2h_bytes_per_step": int(r["d2h"])},
            "gpu_launches": int(r["launches"]),
            "clocks": r["clocks"],
        }
        proj = projection_roofline(wl, r.get("proj_ms"), bw, src)
        if proj is not None:
            line["rooflines"] = {"projections": proj}
        if not args.no_cpu_baseline:
            v, sample, _ = oracle_sample(wl)
            line["cpu_baseline"] = {"value": round(v, 3), "unit": UNIT, "cores": cores_used(), "kind": "oracle",
                                    "sample": sample}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
