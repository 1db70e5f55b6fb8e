// Persistent cluster decoder: all n steps of a decode call of bf16 models in
// one launch, one thread-block cluster per group of sequences (the plan and
// the shared-memory layout are in fused_plan.h).
//
// A step is the transition of "Understanding and Applying the Recurrent
// Looped Transformer Architecture" (architecture section): the gated merge
// u = z s_{t-1} + (1 - z) e_t, then per decoder layer sliding-window
// self-attention over the ring of the last W keys and values (the current one
// included), cross-attention to encoder memory positions 1..t, and a SwiGLU
// feed-forward, each with a pre-RMSNorm and a residual add; s_t is the last
// residual stream, and the head scores the next action under
// softmax(W_o RMSNorm_o(s_t) / temperature), optionally truncated to the
// top k.  The values stored in bf16 are the ones the other decoder path
// stores: the normalised projection inputs, the RoPE'd keys and the values,
// the two attention outputs and the SwiGLU product.
//
// Phases of a step (one cluster barrier after each but the head):
//   gate  rows of z, h = z s + (1 - z) e        -> h rows pushed to every CTA
//   per layer:
//   QKV   q, k, v of this CTA's heads, RoPE, ring write, window attention
//                                                -> attention output pushed
//   O     rows of h += O o                       -> h rows pushed
//   Qx    queries of this CTA's heads, cross-attention over memory 0..p
//                                                -> cross-attention output pushed
//   Ox    rows of h += Ox ox                     -> h rows pushed
//   W13   rows of m = silu(W_1 b) * (W_3 b)      -> m rows pushed
//   W2    rows of h += W_2 m                     -> h rows pushed
//   head  (CTAs that score) logits of every row, scores of the CTA's rows
// Projections run on the tensor cores as warp-level bf16 MMAs with the
// weights as the 16-row operand and the cluster's sequences as the 8-column
// operand; the weights of phase q + 1 are copied from L2 into one half of a
// double-buffered stage while phase q computes from the other half (the
// copy starts once phase q - 1 has read that half), and the memory rows of
// the next layer's cross-attention are prefetched into L2.
// The residual streams of step i live in h buffer i mod 2, so the step's
// first pushes never land on the buffer another CTA may still be reading for
// the previous step's head.  Each CTA keeps the window keys and values of its
// pairs in shared memory (loaded from the state's ring at the start, written
// through to it every step).  Exchanges move 16 bytes per store.
#pragma once
#include "common.cuh"
#include "fused_plan.h"
#include "fused_ptx.cuh"
#include "sampling.cuh"

namespace rlt {
namespace fused {

struct Args {
  const bf16 *W_g, *W_qkv, *W_O, *W_Qx, *W_Ox, *W_1, *W_3, *W_2, *W_o;
  const float *b_g, *attn_norm, *xattn_norm, *ffn_norm, *head_norm;
  const float2* rope;    // [T_mem][hd / 2] (cos, sin) of position p, rows p0 .. p0 + n - 1
  bf16* e;               // [B][T_mem][d] (written at p in generation)
  bf16* mem;             // [G][2][B][H][T_mem][hd] (written at p in generation)
  const int* actions;    // [B][n] or null
  const int* emit_map;   // [n]: index into logits_out or -1; or null
  float* logits_out;     // [n_emit][B][V] or null
  float* logp;           // [B][n] or null
  float* logp_full;      // [B][n] or null
  int* argmax;           // [B][n] or null
  float* s;              // [B][d] f32 state, read at the start and written at the end
  bf16* ring_k;          // [L][B][H][W][hd]
  bf16* ring_v;
  int* status;
  int B, T_mem, p0, n, top_k;
  float eps, theta, scale, inv_temp;
  // generation (gen != 0): step i draws x_p (p = p0 + i) from the state's
  // tempered top-k distribution with the uniform number of (seed, b, p),
  // writes it to tokens [B][n] and its log-probability to logp, encodes it
  // against the encoder cache enc_kv [L][2][B][H][T_mem][hd] (writing row p
  // of enc_kv, e and mem) and consumes it
  int gen;
  const bf16* tok_emb;   // [V][d]
  const float *enc_attn_norm, *enc_ffn_norm, *enc_norm;
  const bf16 *W_K, *W_V;  // [G][d][d]
  bf16* enc_kv;
  int* tokens;
  unsigned long long seed;
  Shape sh;
  Plan P;
};

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bround(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
__device__ __forceinline__ unsigned bf16x2(float lo, float hi) {
  return (unsigned)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((unsigned)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  return make_uint4(bf16x2(v[0], v[1]), bf16x2(v[2], v[3]), bf16x2(v[4], v[5]), bf16x2(v[6], v[7]));
}
__device__ __forceinline__ void unpack8(const uint4& u, float (&v)[8]) {
  const unsigned w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// The heads and sequences CTA r attends for.
struct Work {
  int hlo, hpc, blo, bhi, npairs;
};
__device__ __forceinline__ Work work_of(const Plan& P, int r, int nbv) {
  Work w;
  w.hpc = P.hpc;
  if (P.gph > 0) {
    w.hlo = r / P.gph;
    const int sg = r % P.gph;
    w.blo = sg * P.Bc / P.gph;
    w.bhi = (sg + 1) * P.Bc / P.gph;
  } else {
    w.hlo = r * P.hpc;
    w.blo = 0;
    w.bhi = P.Bc;
  }
  w.bhi = min(w.bhi, nbv);
  w.blo = min(w.blo, w.bhi);
  w.npairs = (w.bhi - w.blo) * w.hpc;
  return w;
}

struct Ph {
  int kind, l, nt, K, U;
  int lo;  // first tile of the row-split phases (gate, O, Ox, W_1/W_3, W_2)
};
struct Tile {
  const bf16* W;
  int row0, N;
};

// Phases of a generation step before the decoder's: the draw, per encoder
// layer QKV + attention, O, W_1/W_3, W_2 (with per-layer memory also the
// memory rows of group l after layer l), then the memory rows e_p feeds.
__device__ __forceinline__ int enc_phases(const Shape& s) { return 4 * s.L + (s.mem_source ? s.L : s.G); }

// Phase k of a step on CTA r (scorer: the CTA scores at least one sequence).
__device__ __forceinline__ Ph phase_at(const Args& a, int k, int r, const Work& wk, bool scorer) {
  const Shape& s = a.sh;
  const int CS = a.P.CS;
  Ph ph{};
  int kd = k;  // index among the decoder step's phases
  if (a.gen) {
    if (k == 0) {
      ph.kind = kTok;
      kd = -1;
    } else if (k - 1 < enc_phases(s)) {
      const int e = k - 1;
      if (s.mem_source) {
        ph.l = e / 5;
        ph.kind = e % 5 < 4 ? kEQKV + e % 5 : kMem;
      } else if (e < 4 * s.L) {
        ph.l = e / 4;
        ph.kind = kEQKV + e % 4;
      } else {
        ph.l = e - 4 * s.L;
        ph.kind = kMem;
      }
      kd = -1;
    } else {
      kd = k - 1 - enc_phases(s);
    }
  }
  if (kd >= 0) {
    // decoding with a gate: the head of the previous step runs right after
    // the gate (between the halves of its cluster barrier) on the CTAs that
    // score; otherwise it ends the step
    const bool hov = !a.gen && s.gate;
    if (s.gate && kd == 0) {
      ph.kind = kGate;
    } else if (hov && scorer && kd == 1) {
      ph.kind = kHead;
    } else {
      const int kk = kd - (s.gate ? 1 : 0) - (hov && scorer ? 1 : 0);
      if (kk < 6 * s.L) {
        ph.kind = kQKV + kk % 6;
        ph.l = kk / 6;
      } else {
        ph.kind = kHead;
      }
    }
  }
  int lo, hi;
  const int th = wk.npairs > 0 ? wk.hpc * (s.hd / 16) : 0;
  switch (ph.kind) {
    case kGate: part_range(s.d / 16, CS, r, &lo, &hi); ph.lo = lo; ph.nt = hi - lo; ph.K = 2 * s.d; break;
    case kQKV:
    case kEQKV: ph.nt = 3 * th; ph.K = s.d; break;
    case kQx: ph.nt = th; ph.K = s.d; break;
    case kMem: ph.nt = 2 * th; ph.K = s.d; break;
    case kO:
    case kOx:
    case kEO: part_range(s.d / 16, CS, r, &lo, &hi); ph.lo = lo; ph.nt = hi - lo; ph.K = s.d; break;
    case kW13:
    case kEW13: part_range(cdivi(s.f, 16), CS, r, &lo, &hi); ph.lo = lo; ph.nt = 2 * (hi - lo); ph.K = s.d; break;
    case kW2:
    case kEW2: part_range(s.d / 16, CS, r, &lo, &hi); ph.lo = lo; ph.nt = hi - lo; ph.K = s.f; break;
    case kTok: ph.nt = scorer ? cdivi(s.V, 16) : 0; ph.K = s.d; break;
    default: ph.nt = cdivi(s.V, 16); ph.K = s.d; break;
  }
  ph.U = round32(ph.K) / 32;
  return ph;
}

// Weight rows of tile t of phase ph (ph.lo: the CTA's first tile of the
// row-split phases).
__device__ __forceinline__ Tile tile_at(const Args& a, const Ph& ph, int t, int, const Work& wk) {
  const Shape& s = a.sh;
  const int d = s.d, hd = s.hd, nh = hd / 16;
  const size_t dd = (size_t)d * d, fd = (size_t)s.f * d;
  const int lo = ph.lo;
  Tile T;
  switch (ph.kind) {
    case kGate:
      T = Tile{a.W_g, (lo + t) * 16, d};
      break;
    case kQKV:
    case kEQKV: {
      const int hh = t / (3 * nh), rem = t - hh * 3 * nh, part = rem / nh, j = rem - part * nh;
      T = Tile{a.W_qkv + (size_t)ph.l * 3 * dd, part * d + (wk.hlo + hh) * hd + 16 * j, 3 * d};
      break;
    }
    case kQx: {
      const int hh = t / nh, j = t - hh * nh;
      T = Tile{a.W_Qx + (size_t)ph.l * dd, (wk.hlo + hh) * hd + 16 * j, d};
      break;
    }
    case kMem: {  // keys then values of the CTA's heads, group ph.l
      const int hh = t / (2 * nh), rem = t - hh * 2 * nh, kv = rem / nh, j = rem - kv * nh;
      T = Tile{(kv ? a.W_V : a.W_K) + (size_t)ph.l * dd, (wk.hlo + hh) * hd + 16 * j, d};
      break;
    }
    case kO:
    case kOx:
    case kEO:
      T = Tile{(ph.kind == kOx ? a.W_Ox : a.W_O) + (size_t)ph.l * dd, (lo + t) * 16, d};
      break;
    case kW13:
    case kEW13:
      T = Tile{((t & 1) ? a.W_3 : a.W_1) + (size_t)ph.l * fd, (lo + (t >> 1)) * 16, s.f};
      break;
    case kW2:
    case kEW2:
      T = Tile{a.W_2 + (size_t)ph.l * fd, (lo + t) * 16, d};
      break;
    default:
      T = Tile{a.W_o, 16 * t, s.V};
      break;
  }
  return T;
}

// Copies the weights of phase ph into a stage buffer: unit (t, u) holds rows
// row0 .. row0 + 15 and columns 32 u .. 32 u + 31 of tile t, as lane L's
// 16 bytes of row row0 + L/4 (first 512 bytes) and of row row0 + 8 + L/4
// (second 512), columns 32 u + 8 (L % 4) .. + 7 - the A operand of two MMAs
// with the 16 columns of one MMA taken as 8 (L % 4) + {0, 1, 2, 3} and the
// other's as + {4, 5, 6, 7} (B uses the same pairing).  Rows past N and
// columns past K are zero.
__device__ __forceinline__ void issue(const Args& a, const Ph& ph, int r, const Work& wk, unsigned char* stg, int t0,
                                      int t1) {
  // tiles t0 .. t1 - 1 of the phase, unit (t - t0, u) at ((t - t0) U + u);
  // thread t copies piece t % 64 of units t / 64, t / 64 + kThreads / 64, ...
  const int jj = threadIdx.x & 63, half = jj >> 5, ln = jj & 31;
  const int rofs = (ln >> 2) + 8 * half, kofs = 8 * (ln & 3);
  const int nunits = (t1 - t0) * ph.U;
  constexpr int kStep = kThreads / 64;
  int t = t0, u = threadIdx.x >> 6;
  while (u >= ph.U && t < t1) {
    u -= ph.U;
    ++t;
  }
  Tile T{};
  int tcur = -1;
  for (int unit = threadIdx.x >> 6; unit < nunits; unit += kStep) {
    if (t != tcur) {
      T = tile_at(a, ph, t, r, wk);
      tcur = t;
    }
    const int row = T.row0 + rofs, k = u * 32 + kofs;
    const bf16* src = T.W;
    int bytes = 0;
    if (row < T.N && k < ph.K) {
      src = T.W + (size_t)row * ph.K + k;
      bytes = min(16, (ph.K - k) * 2);
    }
    cp_async16(stg + (size_t)unit * kUnitBytes + half * 512 + ln * 16, src, bytes);
    u += kStep;
    while (u >= ph.U) {
      u -= ph.U;
      ++t;
    }
  }
}

// The outputs of a projection phase: y(t, row, col) of tile t, either in
// out [t][16][cols] or as the split-K partial sums of the warps in part
// (added in split order when read).
struct PY {
  const float* out;
  const float* part;
  int cols, ks;  // ks = 0: whole tiles in out
  __device__ __forceinline__ float operator()(int t, int row, int col) const {
    if (ks == 0) return out[(size_t)(t * 16 + row) * cols + col];
    const int lane = (row & 7) * 4 + ((col & 7) >> 1), q = (row >> 3) * 2 + (col & 1), j = col >> 3;
    float v = 0.f;
    for (int s2 = 0; s2 < ks; ++s2) v += part[(((t * ks + s2) * 2 + j) * 32 + lane) * 4 + q];
    return v;
  }
};

// W_tile X^T for the phase's tiles from the stage, with X [cols][ldX] bf16
// (zero past K).  With at least kWarps tiles each warp takes whole tiles and
// writes out; otherwise each tile's K is split over kWarps / nt warps whose
// partial sums stay in part (reduce: added into out here, in split order).
// Ends with a block barrier; the stage is no longer read after it.
__device__ __forceinline__ PY proj(const Ph& ph, int cols, const unsigned char* stg, const bf16* X, int ldX,
                                   float* out, float* part, bool reduce, int tout = 0) {
  const int nt = ph.nt, U = ph.U, NT = cols / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  if (nt == 0) return PY{out, part, cols, 0};
  auto run = [&](int t, int u0, int u1, float (&acc)[2][4]) {
    for (int u = u0; u < u1; ++u) {
      const uint4* up = reinterpret_cast<const uint4*>(stg + ((size_t)t * U + u) * kUnitBytes);
      const uint4 w0 = up[lane], w1 = up[32 + lane];
      const unsigned A1[4] = {w0.x, w1.x, w0.y, w1.y}, A2[4] = {w0.z, w1.z, w0.w, w1.w};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (j < NT) {
          const uint4 xv = *reinterpret_cast<const uint4*>(X + (size_t)(8 * j + g) * ldX + u * 32 + 8 * c);
          const unsigned B1[2] = {xv.x, xv.y}, B2[2] = {xv.z, xv.w};
          mma_bf16(acc[j], A1, B1);
          mma_bf16(acc[j], A2, B2);
        }
      }
    }
  };
  if (nt >= kWarps) {
    for (int t = warp; t < nt; t += kWarps) {
      float acc[2][4] = {};
      run(t, 0, U, acc);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (j < NT) {
          float* o0 = out + (size_t)((tout + t) * 16 + g) * cols + 8 * j + 2 * c;
          float* o1 = o0 + 8 * cols;
          o0[0] = acc[j][0];
          o0[1] = acc[j][1];
          o1[0] = acc[j][2];
          o1[1] = acc[j][3];
        }
      }
    }
    __syncthreads();
    return PY{out, part, cols, 0};
  }
  const int ks = kWarps / nt, t = warp / ks, sp = warp - t * ks;
  if (t < nt) {
    float acc[2][4] = {};
    run(t, sp * U / ks, (sp + 1) * U / ks, acc);
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) part[((warp * 2 + j) * 32 + lane) * 4 + q] = acc[j][q];
  }
  __syncthreads();
  const PY y{out, part, cols, ks};
  if (!reduce) return y;
  for (int e = threadIdx.x; e < nt * 16 * cols; e += kThreads) {
    const int tt = e / (16 * cols), rem = e - tt * 16 * cols, row = rem / cols, col = rem - row * cols;
    out[(size_t)tout * 16 * cols + e] = y(tt, row, col);
  }
  __syncthreads();
  return PY{out, part, cols, 0};
}

// The head of column b (global sequence bg) at step i (position p) from the
// logits in out: the tempered log-softmax, the top-k set (exact k-th largest
// key by radix select, ties to the lower id) and the argmax (lowest id on
// ties).  Scoring: the action's lp, lp_full, argmax and the optional logits
// copy.  Generation: the draw with the uniform number of (seed, bg, p)
// (sample_chunked), written to tokens with its lp and pushed to every CTA's
// tok[b].  sx: V floats of shared memory.
__device__ void head_col(const Args& a, const float* out, int cols, int b, int bg, int i, int p,
                         unsigned char* misc, float* sx, int* tok) {
  float* fred = reinterpret_cast<float*>(misc);                // [32]
  int* ired = reinterpret_cast<int*>(misc + 128);              // [32]
  unsigned* hist = reinterpret_cast<unsigned*>(misc + 256);    // [256]
  unsigned* sc = reinterpret_cast<unsigned*>(misc + 1280);     // prefix, remain, count
  int* s_res = reinterpret_cast<int*>(misc + 1296);            // [5]
  float* s_part = reinterpret_cast<float*>(misc + 1536);       // [kThreads]
  unsigned* s_tie = reinterpret_cast<unsigned*>(misc + 2560);  // [kThreads]
  const int V = a.sh.V, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float it = a.inv_temp;
  auto lg = [&](int v) { return out[(size_t)((v >> 4) * 16 + (v & 15)) * cols + b]; };
  float bmax = -INFINITY;
  int barg = 0x7fffffff;
  for (int v = tid; v < V; v += kThreads) {
    const float x = lg(v);
    sx[v] = x * it;
    if (x > bmax || (x == bmax && v < barg)) {
      bmax = x;
      barg = v;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, bmax, o);
    const int oa = __shfl_xor_sync(0xffffffffu, barg, o);
    if (om > bmax || (om == bmax && oa < barg)) {
      bmax = om;
      barg = oa;
    }
  }
  if (lane == 0) {
    fred[warp] = bmax;
    ired[warp] = barg;
  }
  __syncthreads();
  if (tid == 0) {
    float mm = fred[0];
    int aa = ired[0];
    for (int w = 1; w < kWarps; ++w)
      if (fred[w] > mm || (fred[w] == mm && ired[w] < aa)) {
        mm = fred[w];
        aa = ired[w];
      }
    fred[0] = mm;
    ired[0] = aa;
  }
  __syncthreads();
  const int amax = ired[0];
  const float mx = fred[0] * it;
  __syncthreads();
  float se = 0.f;
  for (int v = tid; v < V; v += kThreads) se += expf(sx[v] - mx);
  se = warp_sum(se);
  if (lane == 0) fred[warp] = se;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kWarps; ++w) t += fred[w];
    fred[0] = t;
  }
  __syncthreads();
  const float lse = mx + logf(fred[0]);
  __syncthreads();
  const bool topk = a.top_k > 0 && a.top_k < V;
  int act = a.gen ? -1 : (a.actions ? a.actions[(size_t)bg * a.n + i] : -1);
  if (act >= V) {
    if (tid == 0) set_error(a.status, kErrBounds);
    act = -1;
  }
  if (a.gen && !topk) act = sample_chunked(sx, V, mx, true, 0u, 0u, uniform24(a.seed, bg, p), s_part, s_tie, s_res);
  float lp_full = act >= 0 ? sx[act] - lse : NAN;
  float lp = lp_full;
  if (topk) {
    // k-th largest key by radix select, 8 bits at a time from the top
    if (tid == 0) {
      sc[0] = 0;
      sc[1] = (unsigned)a.top_k;
    }
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int j = tid; j < 256; j += kThreads) hist[j] = 0;
      __syncthreads();
      const unsigned pref = sc[0];
      const unsigned hmask = pass == 0 ? 0u : (0xffffffffu << (shift + 8));
      for (int v = tid; v < V; v += kThreads) {
        const unsigned kk = f2key(sx[v]);
        if ((kk & hmask) == pref) atomicAdd(&hist[(kk >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        unsigned rem = sc[1];
        int bin = 255;
        for (; bin > 0; --bin) {
          if (hist[bin] >= rem) break;
          rem -= hist[bin];
        }
        sc[0] = pref | ((unsigned)bin << shift);
        sc[1] = rem;
      }
      __syncthreads();
    }
    const unsigned kth = sc[0], need = sc[1];
    const float xk = __uint_as_float((kth & 0x80000000u) ? (kth & 0x7fffffffu) : ~kth);
    if (a.gen) {
      act = sample_chunked(sx, V, mx, false, kth, need, uniform24(a.seed, bg, p), s_part, s_tie, s_res);
      lp_full = sx[act] - lse;
    }
    float sg = 0.f;
    for (int v = tid; v < V; v += kThreads)
      if (f2key(sx[v]) > kth) sg += expf(sx[v] - mx);
    sg = warp_sum(sg);
    unsigned below = 0;  // ids below the action with the k-th key
    if (act >= 0 && f2key(sx[act]) == kth)
      for (int v = tid; v < act; v += kThreads) below += f2key(sx[v]) == kth ? 1u : 0u;
    __syncthreads();
    if (lane == 0) fred[warp] = sg;
    if (tid == 0) sc[2] = 0;
    __syncthreads();
    if (below) atomicAdd(&sc[2], below);
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      for (int w = 0; w < kWarps; ++w) t += fred[w];
      fred[0] = t;
    }
    __syncthreads();
    const float lse_k = mx + logf(fred[0] + (float)need * expf(xk - mx));
    if (act >= 0) {
      const unsigned ka = f2key(sx[act]);
      const bool in = ka > kth || (ka == kth && sc[2] < need);
      lp = in ? sx[act] - lse_k : -INFINITY;
    }
  }
  const size_t o = (size_t)bg * a.n + i;
  if (a.gen) {
    if (tid == 0) {
      a.tokens[o] = act;
      if (a.logp) a.logp[o] = lp;
    }
    if (tid < a.P.CS) *map_rank(tok + b, (unsigned)tid) = act;
  } else {
    const int em = a.emit_map ? a.emit_map[i] : -1;
    if (em >= 0 && a.logits_out)
      for (int v = tid; v < V; v += kThreads) a.logits_out[((size_t)em * a.B + bg) * V + v] = lg(v);
    if (tid == 0) {
      if (a.logp) a.logp[o] = lp;
      if (a.logp_full) a.logp_full[o] = lp_full;
      if (a.argmax) a.argmax[o] = amax;
    }
  }
  __syncthreads();
}

template <class T>
__device__ __forceinline__ void push(T* p, const T& v, int CS) {  // the same address in every CTA of the cluster
  for (int rk = 0; rk < CS; ++rk) *map_rank(p, (unsigned)rk) = v;
}

__global__ void __launch_bounds__(kThreads, 1) dec_fused_kernel(const __grid_constant__ Args a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const Shape& s = a.sh;
  const Plan& P = a.P;
  const int CS = P.CS, cols = P.cols;
  const int r = (int)cluster_rank();
  const int b0 = (int)(blockIdx.x / CS) * P.Bc;  // first sequence of the cluster
  const int nbv = min(P.Bc, a.B - b0);           // its sequences
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int d = s.d, hd = s.hd, H = s.H, W = s.W, nh = hd / 16, half = hd / 2, hd8 = hd / 8;
  float* hb = reinterpret_cast<float*>(smem + P.o_h);     // [2][cols][d] residual streams
  bf16* xb = reinterpret_cast<bf16*>(smem + P.o_x);       // [cols][ldx] local projection input
  bf16* ob = reinterpret_cast<bf16*>(smem + P.o_ob);      // [cols][ldo] gathered attention output
  bf16* mb = reinterpret_cast<bf16*>(smem + P.o_mb);      // [cols][ldm] gathered SwiGLU product
  float* out = reinterpret_cast<float*>(smem + P.o_out);  // [maxT][16][cols] projection outputs
  float* part = reinterpret_cast<float*>(smem + P.o_part);
  float* pr = reinterpret_cast<float*>(smem + P.o_pr);    // [npairs][hd] queries (log2 units)
  bf16* ringK = reinterpret_cast<bf16*>(smem + P.o_ring); // [L][npairs][W][hd]
  bf16* ringV = ringK + (size_t)s.L * P.npairs * W * hd;
  float* xp = reinterpret_cast<float*>(smem + P.o_xp);    // [units][hd + 2] cross-attention partials
  unsigned char* misc = smem + P.o_misc;
  bf16* eb = reinterpret_cast<bf16*>(smem + P.o_e);       // [2][cols][d] e_p of step i in half i mod 2
  float2* rb = reinterpret_cast<float2*>(eb + (size_t)2 * cols * d);  // [2][hd / 2] its (cos, sin) row
  float* he = reinterpret_cast<float*>(smem + P.o_he);    // [cols][d] generation: encoder streams
  int* tokb = reinterpret_cast<int*>(smem + P.o_tok);     // [cols] generation: this step's tokens
  float* sx = reinterpret_cast<float*>(smem + P.o_sx);    // [V] tempered logits of the scored row
  unsigned char* stage = smem + P.o_stage;
  const Work wk = work_of(P, r, nbv);
  const bool scorer = r < nbv;
  const float qscale = a.scale * kLog2e;
  const int CH = hd8, RPW = 32 / CH, rg = lane / CH, cc = lane - rg * CH;  // attention lanes: CH per key row
  auto pair_b = [&](int pi) { return wk.blo + pi / wk.hpc; };
  auto pair_h = [&](int pi) { return wk.hlo + pi % wk.hpc; };
  auto gring = [&](int l, int pi) {  // the pair's ring rows in the state, [W][hd]
    return (((size_t)l * a.B + b0 + pair_b(pi)) * H + pair_h(pi)) * W * hd;
  };

  // zero operands and streams (padding rows and columns stay zero); s -> h
  // buffer 1; the pairs' ring rows -> shared memory
  for (size_t i = tid; i < P.o_stage / 16; i += kThreads) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  for (int i = tid; i < nbv * d; i += kThreads) hb[(size_t)cols * d + i] = a.s[(size_t)b0 * d + i];
  for (int i = tid; i < s.L * wk.npairs * W * hd8; i += kThreads) {
    const int c8 = i % hd8, row = i / hd8, slot = row % W, lp = row / W, pi = lp % wk.npairs, l = lp / wk.npairs;
    const size_t go = gring(l, pi) + (size_t)slot * hd + 8 * c8;
    const size_t so = (((size_t)l * P.npairs + pi) * W + slot) * hd + 8 * c8;
    *reinterpret_cast<uint4*>(ringK + so) = ld_cg16(a.ring_k + go);
    *reinterpret_cast<uint4*>(ringV + so) = ld_cg16(a.ring_v + go);
  }
  cluster_sync();  // no CTA pushes into one that is still zeroing

  // L2 prefetch of the memory rows the cross-attention of (layer l, position p) reads
  auto prefetch_mem = [&](int l, int p) {
    const int g = s.G == 1 ? 0 : l;
    const unsigned bytes = (unsigned)(p + 1) * hd * 2;
    for (int j = tid; j < 2 * wk.npairs; j += kThreads) {
      const int pi = j >> 1, kv = j & 1;
      prefetch_l2(a.mem + ((((size_t)g * 2 + kv) * a.B + b0 + pair_b(pi)) * H + pair_h(pi)) * (size_t)a.T_mem * hd,
                  bytes);
    }
  };
  // xb = bf16(RMSNorm(h) g) (h in shared memory): lane j takes columns
  // 8j .. 8j + 7 of each 256-column group, 16-byte accesses; the row is read
  // twice (sum of squares, then the scaled values) so that nothing is held in
  // registers across the groups
  auto rmsnorm_x = [&](const float* h, const float* g) {
    for (int b = warp; b < nbv; b += kWarps) {
      const float* hr = h + (size_t)b * d;
      float ss = 0.f;
      for (int c = 8 * lane; c < d; c += 256) {
        const float4 u0 = *reinterpret_cast<const float4*>(hr + c);
        const float4 u1 = *reinterpret_cast<const float4*>(hr + c + 4);
        ss = fmaf(u0.x, u0.x, fmaf(u0.y, u0.y, fmaf(u0.z, u0.z, fmaf(u0.w, u0.w, ss))));
        ss = fmaf(u1.x, u1.x, fmaf(u1.y, u1.y, fmaf(u1.z, u1.z, fmaf(u1.w, u1.w, ss))));
      }
      ss = warp_sum(ss);
      const float rv = 1.0f / sqrtf(ss / (float)d + a.eps);
      for (int c = 8 * lane; c < d; c += 256) {
        const float4 u0 = *reinterpret_cast<const float4*>(hr + c);
        const float4 u1 = *reinterpret_cast<const float4*>(hr + c + 4);
        const float4 g0 = ld_nc_f4(g + c), g1 = ld_nc_f4(g + c + 4);
        const float v8[8] = {u0.x * rv * g0.x, u0.y * rv * g0.y, u0.z * rv * g0.z, u0.w * rv * g0.w,
                             u1.x * rv * g1.x, u1.y * rv * g1.y, u1.z * rv * g1.z, u1.w * rv * g1.w};
        *reinterpret_cast<uint4*>(xb + (size_t)b * P.ldx + c) = pack8(v8);
      }
    }
    __syncthreads();
  };
  // residual add of this CTA's d rows, four rows per push
  auto residual = [&](float* h, const PY& y) {
    int lo, hi;
    part_range(d / 16, CS, r, &lo, &hi);
    const int nq = (hi - lo) * 4;
    for (int i2 = tid; i2 < nbv * nq; i2 += kThreads) {
      const int b = i2 / nq, rr = 4 * (i2 - b * nq), row = lo * 16 + rr, t0 = rr >> 4, w = rr & 15;
      float* hp = h + (size_t)b * d + row;
      const float4 v = make_float4(hp[0] + y(t0, w, b), hp[1] + y(t0, w + 1, b), hp[2] + y(t0, w + 2, b),
                                   hp[3] + y(t0, w + 3, b));
      push(reinterpret_cast<float4*>(hp), v, CS);
    }
  };
  // online-softmax attention of one warp's query (8 elements a lane, CH lanes
  // per key row) over key rows [ka, kb) read by ldk / ldv; merged over the
  // warp's row groups, the result is in every lane of row group 0
  struct Acc {
    float m, l, o[8];
  };
  auto attend = [&](const float (&qv)[8], int ka, int kb, auto ldk, auto ldv) {
    Acc A;
    A.m = -INFINITY;
    A.l = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) A.o[e] = 0.f;
    constexpr int UN = 8;
    for (int j0 = ka; j0 < kb; j0 += UN * RPW) {
      uint4 kk[UN], vv[UN];
#pragma unroll
      for (int u = 0; u < UN; ++u) {
        const int j = j0 + u * RPW + rg;
        kk[u] = j < kb ? ldk(j) : make_uint4(0, 0, 0, 0);
        vv[u] = j < kb ? ldv(j) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < UN; ++u) {
        const int j = j0 + u * RPW + rg;
        float kf[8];
        unpack8(kk[u], kf);
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) dot = fmaf(qv[e], kf[e], dot);
        for (int o = 1; o < CH; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (j < kb) {
          const float mn = fmaxf(A.m, dot);
          const float corr = exp2f(A.m - mn), pj = exp2f(dot - mn);
          float vf[8];
          unpack8(vv[u], vf);
          A.l = A.l * corr + pj;
#pragma unroll
          for (int e = 0; e < 8; ++e) A.o[e] = fmaf(pj, vf[e], A.o[e] * corr);
          A.m = mn;
        }
      }
    }
    for (int o = CH; o < 32; o <<= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, A.m, o), l2 = __shfl_xor_sync(0xffffffffu, A.l, o);
      float a2[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) a2[e] = __shfl_xor_sync(0xffffffffu, A.o[e], o);
      const float mn = fmaxf(A.m, m2);
      const float c1 = A.m == -INFINITY ? 0.f : exp2f(A.m - mn), c2 = m2 == -INFINITY ? 0.f : exp2f(m2 - mn);
      A.l = A.l * c1 + l2 * c2;
#pragma unroll
      for (int e = 0; e < 8; ++e) A.o[e] = A.o[e] * c1 + a2[e] * c2;
      A.m = mn;
    }
    return A;
  };

  // e_p and the RoPE row of step `step` (p = p0 + step) into their halves of
  // eb and rb, in this thread's current cp.async group
  auto issue_e = [&](int step) {
    const int p = a.p0 + step, d8 = d / 8;
    for (int j = tid; j < (a.gen ? 0 : nbv * d8); j += kThreads) {  // generation computes e_p
      const int b = j / d8, c8 = j - b * d8;
      cp_async16(eb + ((size_t)(step & 1) * cols + b) * d + 8 * c8, a.e + ((size_t)(b0 + b) * a.T_mem + p) * d + 8 * c8,
                 16);
    }
    for (int j = tid; j < half / 2; j += kThreads)  // two (cos, sin) pairs per copy
      cp_async16(rb + (size_t)(step & 1) * half + 2 * j, a.rope + (size_t)p * half + 2 * j, 16);
  };
  // attention of each pair's query (pr, log2 units) over key rows 0..nk-1 at
  // Kb(pi), Vb(pi) ([nk][hd] bf16): each pair's keys split over ns warps,
  // partials combined in split order, the result pushed to ob.  coherent:
  // rows written during this launch, read through L2.
  // Segments: one per pair when the pairs fill the warps; otherwise the kWarps
  // warps split the pairs' keys, pair pi owning segments
  // [ceil(pi kWarps / np), ceil((pi + 1) kWarps / np)) (every warp busy).
  auto pair_attention = [&](auto Kb, auto Vb, int nk, bool coherent) {
    const int np = wk.npairs;
    const bool split = np > 0 && np < kWarps;
    const int nseg = split ? kWarps : np;
    auto seg_lo = [&](int pi) { return split ? (pi * kWarps + np - 1) / np : pi; };
    for (int w0 = warp; w0 < nseg; w0 += kWarps) {
      const int pi = split ? (w0 * np) / kWarps : w0;
      const int s0 = seg_lo(pi), ns = seg_lo(pi + 1) - s0, sp = w0 - s0;
      const bf16* Kp = Kb(pi) + 8 * cc;
      const bf16* Vp = Vb(pi) + 8 * cc;
      float qv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) qv[e] = pr[(size_t)pi * hd + 8 * cc + e];
      const Acc A = attend(
          qv, sp * nk / ns, (sp + 1) * nk / ns,
          [&](int j) { return coherent ? ld_cg16(Kp + (size_t)j * hd) : ld_nc16(Kp + (size_t)j * hd); },
          [&](int j) { return coherent ? ld_cg16(Vp + (size_t)j * hd) : ld_nc16(Vp + (size_t)j * hd); });
      float* xw = xp + (size_t)w0 * (hd + 2);
      if (rg == 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e) xw[8 * cc + e] = A.o[e];
      }
      if (lane == 0) {
        xw[hd] = A.m;
        xw[hd + 1] = A.l;
      }
    }
    __syncthreads();
    for (int i2 = tid; i2 < wk.npairs * hd8; i2 += kThreads) {
      const int pi = i2 / hd8, c8 = i2 - pi * hd8;
      const int s0 = seg_lo(pi), s1 = seg_lo(pi + 1);
      float M = -INFINITY;
      for (int sg = s0; sg < s1; ++sg) {
        const float* xw = xp + (size_t)sg * (hd + 2);
        if (xw[hd + 1] > 0.f) M = fmaxf(M, xw[hd]);
      }
      float num[8] = {}, den = 0.f;
      for (int sg = s0; sg < s1; ++sg) {
        const float* xw = xp + (size_t)sg * (hd + 2);
        if (xw[hd + 1] > 0.f) {
          const float cf = exp2f(xw[hd] - M);
#pragma unroll
          for (int e = 0; e < 8; ++e) num[e] = fmaf(xw[8 * c8 + e], cf, num[e]);
          den = fmaf(xw[hd + 1], cf, den);
        }
      }
      const float inv = 1.0f / den;
#pragma unroll
      for (int e = 0; e < 8; ++e) num[e] *= inv;
      push(reinterpret_cast<uint4*>(ob + (size_t)pair_b(pi) * P.ldo + pair_h(pi) * hd + 8 * c8), pack8(num), CS);
    }
  };
  // m = silu(W_1 b) * (W_3 b) of this CTA's f rows, eight rows per push
  auto swiglu_push = [&](const PY& y) {
    int lo, hi;
    part_range(cdivi(s.f, 16), CS, r, &lo, &hi);
    const int n8 = (hi - lo) * 2;
    for (int i2 = tid; i2 < nbv * n8; i2 += kThreads) {
      const int b = i2 / n8, rr = 8 * (i2 - b * n8), row = lo * 16 + rr;
      if (row >= s.f) continue;
      const int pi = rr >> 4, w = rr & 15;
      float m8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) m8[u] = silu_f(y(2 * pi, w + u, b)) * y(2 * pi + 1, w + u, b);
      push(reinterpret_cast<uint4*>(mb + (size_t)b * P.ldm + row), pack8(m8), CS);
    }
  };
  // RoPE (rotate-half pairs j, j + hd/2) of this CTA's q and k at position p
  // from the QKV tiles of y; q to pr (log2 units, rounded to bf16 first when
  // round_q), k and v rounded to bf16 and handed to put(pi, j, k1, k2, v1, v2)
  auto rope_qkv = [&](const PY& y, const float2* rope_row, bool round_q, auto put) {
    const int half_ = hd / 2;
    for (int i2 = tid; i2 < wk.npairs * half_; i2 += kThreads) {
      const int pi = i2 / half_, j = i2 - pi * half_;
      const int b = pair_b(pi), hh = pi % wk.hpc;
      auto val = [&](int part3, int e) { return y((hh * 3 + part3) * nh + (e >> 4), e & 15, b); };
      const float cf = rope_row[j].x, sf = rope_row[j].y;
      const float q1 = val(0, j), q2 = val(0, j + half_), k1 = val(1, j), k2 = val(1, j + half_);
      float qr1 = q1 * cf - q2 * sf, qr2 = q2 * cf + q1 * sf;
      if (round_q) {
        qr1 = bround(qr1);
        qr2 = bround(qr2);
      }
      pr[(size_t)pi * hd + j] = qr1 * qscale;
      pr[(size_t)pi * hd + j + half_] = qr2 * qscale;
      put(pi, j, __float2bfloat16_rn(k1 * cf - k2 * sf), __float2bfloat16_rn(k2 * cf + k1 * sf),
          __float2bfloat16_rn(val(2, j)), __float2bfloat16_rn(val(2, j + half_)));
    }
  };
  const int kdec0 = a.gen ? 1 + enc_phases(s) : 0;  // the decoder step's first phase
  const int PPS = kdec0 + (s.gate ? 1 : 0) + 6 * s.L + (a.gen ? 0 : (scorer ? 1 : 0));
  const bool hov = !a.gen && s.gate;      // the head of step i - 1 runs after step i's gate
  const bool tail = hov && scorer;        // ... and the last step's head after the loop
  // A phase whose tiles do not fit one stage half runs its projection in
  // parts (tile ranges of tpp tiles), each a pipeline step of its own; the
  // pipeline's steps are numbered over the launch (PSS per decoder step,
  // then the tail's)
  auto tpp_of = [&](const Ph& ph) { return max(1, P.stage_units / ph.U); };
  auto nparts_of = [&](const Ph& ph) { return ph.nt == 0 ? 1 : (ph.nt + tpp_of(ph) - 1) / tpp_of(ph); };
  int PSS = 0;
  for (int k = 0; k < PPS; ++k) PSS += nparts_of(phase_at(a, k, r, wk, scorer));
  const Ph ph_tail = phase_at(a, 1, r, wk, scorer);  // the head (phase 1 of a step when it is the tail)
  const int NQ = a.n * PSS + (tail ? nparts_of(ph_tail) : 0);
  // Pipeline steps are requested strictly in order (0, 1, 2, ...), so a
  // cursor over (phase of the step, part of the phase) names the next one:
  // one phase_at per phase instead of a search from the step's first phase.
  int ic_q = 0, ic_k = 0, ic_pt = 0;  // next pipeline step; its phase and part
  Ph ic_ph = phase_at(a, 0, r, wk, scorer);
  int ic_np = nparts_of(ic_ph);
  auto issue_next = [&](unsigned char* stg) {  // weights of pipeline step ic_q
    const bool in_tail = ic_q >= a.n * PSS;
    const Ph ph = in_tail ? ph_tail : ic_ph;
    const int pt = in_tail ? ic_q - a.n * PSS : ic_pt;
    const int tpp = tpp_of(ph), t0 = pt * tpp;
    issue(a, ph, r, wk, stg, min(t0, ph.nt), min(ph.nt, t0 + tpp));
    ++ic_q;
    if (!in_tail && ++ic_pt == ic_np) {  // the next phase (the next step's first after the last)
      ic_pt = 0;
      ic_k = ic_k + 1 == PPS ? 0 : ic_k + 1;
      ic_ph = phase_at(a, ic_k, r, wk, scorer);
      ic_np = nparts_of(ic_ph);
    }
  };
  auto stage_of = [&](int q) { return stage + (size_t)(q & 1) * P.stage_units * kUnitBytes; };
  // step q's weights go to stage q mod 2; they are requested right after
  // step q - 2's projection has read that half (one cp.async group per
  // step), so each copy has most of two steps to land
  int qc = 0;  // the pipeline step being computed
  issue_next(stage_of(0));
  issue_e(0);
  cp_async_commit();
  if (NQ > 1) issue_next(stage_of(1));
  cp_async_commit();
  prefetch_mem(0, a.p0);

  for (int i = 0; i < a.n; ++i) {
    const int p = a.p0 + i, t = p + 1;
    float* hcur = hb + (size_t)(i & 1) * cols * d;
    const float* hprev = hb + (size_t)((i + 1) & 1) * cols * d;
    const bf16* ecur = eb + (size_t)(i & 1) * cols * d;  // e_p, rows of the cluster's sequences
    const float2* rope_row = rb + (size_t)(i & 1) * half;  // (cos, sin) of position p
    for (int k = 0; k < PPS; ++k) {
      const Ph ph = phase_at(a, k, r, wk, scorer);
      cp_async_wait1();  // this step's group (the next step's may still be in flight)
      __syncthreads();
      // the projection of this phase (in parts when it has more tiles than a
      // stage half holds), each part followed by the request of pipeline
      // step qc + 2 into the half it has read
      auto project = [&](const bf16* X, int ldX, bool reduce = false) {
        const int np = nparts_of(ph), tpp = tpp_of(ph);
        PY y{out, part, cols, 0};
        for (int pt = 0; pt < np; ++pt) {
          if (pt > 0) {
            cp_async_wait1();
            __syncthreads();
          }
          unsigned char* stg = stage_of(qc);
          Ph sub = ph;
          const int t0 = min(pt * tpp, ph.nt);
          sub.nt = min(ph.nt, t0 + tpp) - t0;
          y = proj(sub, cols, stg, X, ldX, out, part, reduce || np > 1, t0);
          if (qc + 2 < NQ) issue_next(stg);  // pipeline step qc + 2 (= ic_q)
          if (k == 0 && pt == 0 && i + 1 < a.n) issue_e(i + 1);  // the next step's e, landed long before it is read
          cp_async_commit();
          ++qc;
        }
        return np > 1 ? PY{out, part, cols, 0} : y;
      };
      if (k == kdec0 && !s.gate) {  // the gate discards s: h = e_p
        for (int i2 = tid; i2 < nbv * d; i2 += kThreads) hcur[i2] = __bfloat162float(ecur[i2]);
        __syncthreads();
      }
      const int l = ph.l;
      switch (ph.kind) {
        case kGate: {
          for (int i2 = tid; i2 < nbv * 2 * d; i2 += kThreads) {
            const int b = i2 / (2 * d), k2 = i2 - b * 2 * d;
            xb[(size_t)b * P.ldx + k2] = k2 < d ? ecur[(size_t)b * d + k2]
                                                 : __float2bfloat16_rn(hprev[(size_t)b * d + k2 - d]);
          }
          __syncthreads();
          const PY y = project(xb, P.ldx);
          int lo, hi;
          part_range(d / 16, CS, r, &lo, &hi);
          const int nq = (hi - lo) * 4;
          for (int i2 = tid; i2 < nbv * nq; i2 += kThreads) {
            const int b = i2 / nq, rr = 4 * (i2 - b * nq), row = lo * 16 + rr;
            const bf16* ep = ecur + (size_t)b * d + row;
            const float* sp = hprev + (size_t)b * d + row;
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float z = sigmoid_f(y((rr + u) >> 4, (rr + u) & 15, b) + a.b_g[row + u]);
              v[u] = z * sp[u] + (1.f - z) * __bfloat162float(ep[u]);
            }
            push(reinterpret_cast<float4*>(hcur + (size_t)b * d + row), make_float4(v[0], v[1], v[2], v[3]), CS);
          }
          cluster_arrive();
          if (!(hov && scorer)) cluster_wait();  // the CTAs that score wait after the previous step's head
          break;
        }
        case kQKV: {
          rmsnorm_x(hcur, a.attn_norm + (size_t)l * d);
          if (l + 1 < s.L) prefetch_mem(l + 1, p);
          else if (i + 1 < a.n) prefetch_mem(0, p + 1);
          const PY y = project(xb, P.ldx);
          // q and k after RoPE; k and v rounded to bf16 into ring slot p mod
          // W, in shared memory and in the state
          const int slot = p % W;
          rope_qkv(y, rope_row, false, [&](int pi, int j, bf16 kr1, bf16 kr2, bf16 v1, bf16 v2) {
            const size_t so = (((size_t)l * P.npairs + pi) * W + slot) * hd;
            ringK[so + j] = kr1;
            ringK[so + j + half] = kr2;
            ringV[so + j] = v1;
            ringV[so + j + half] = v2;
            const size_t go = gring(l, pi) + (size_t)slot * hd;
            a.ring_k[go + j] = kr1;
            a.ring_k[go + j + half] = kr2;
            a.ring_v[go + j] = v1;
            a.ring_v[go + j + half] = v2;
          });
          __syncthreads();
          // window attention over slots 0..min(W, t) - 1 (softmax does not
          // depend on their order), one warp per pair
          const int nv = min(W, t);
          for (int pi = warp; pi < wk.npairs; pi += kWarps) {
            const bf16* Ks = ringK + ((size_t)l * P.npairs + pi) * W * hd;
            const bf16* Vs = ringV + ((size_t)l * P.npairs + pi) * W * hd;
            float qv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) qv[e] = pr[(size_t)pi * hd + 8 * cc + e];
            const Acc A = attend(
                qv, 0, nv, [&](int j) { return *reinterpret_cast<const uint4*>(Ks + (size_t)j * hd + 8 * cc); },
                [&](int j) { return *reinterpret_cast<const uint4*>(Vs + (size_t)j * hd + 8 * cc); });
            if (rg == 0) {
              float o[8];
              const float inv = 1.0f / A.l;
#pragma unroll
              for (int e = 0; e < 8; ++e) o[e] = A.o[e] * inv;
              push(reinterpret_cast<uint4*>(ob + (size_t)pair_b(pi) * P.ldo + pair_h(pi) * hd + 8 * cc), pack8(o), CS);
            }
          }
          cluster_sync();
          break;
        }
        case kO:
        case kOx:
          residual(hcur, project(ob, P.ldo));
          cluster_sync();
          break;
        case kQx: {
          rmsnorm_x(hcur, a.xattn_norm + (size_t)l * d);
          const PY y = project(xb, P.ldx);
          for (int i2 = tid; i2 < wk.npairs * hd; i2 += kThreads) {
            const int pi = i2 / hd, e = i2 - pi * hd;
            const int tt = (pi % wk.hpc) * nh + (e >> 4);
            pr[(size_t)pi * hd + e] = y(tt, e & 15, pair_b(pi)) * qscale;
          }
          __syncthreads();
          // cross-attention over memory positions 0..p (rows this launch
          // wrote, in generation, are read through L2)
          const int g = s.G == 1 ? 0 : l;
          const size_t plane = (size_t)a.T_mem * hd;
          pair_attention(
              [&](int pi) { return a.mem + (((size_t)g * 2 * a.B + b0 + pair_b(pi)) * H + pair_h(pi)) * plane; },
              [&](int pi) { return a.mem + ((((size_t)g * 2 + 1) * a.B + b0 + pair_b(pi)) * H + pair_h(pi)) * plane; },
              t, a.gen != 0);
          cluster_sync();
          break;
        }
        case kW13: {
          rmsnorm_x(hcur, a.ffn_norm + (size_t)l * d);
          const PY y = project(xb, P.ldx);
          swiglu_push(y);
          cluster_sync();
          break;
        }
        case kW2:
          residual(hcur, project(mb, P.ldm));
          cluster_sync();
          break;
        case kTok: {  // generation: x_p drawn from s_p by the CTAs that score, shared with every CTA
          if (scorer) rmsnorm_x(hprev, a.head_norm);
          project(xb, P.ldx, true);
          if (scorer)
            for (int b = r; b < nbv; b += CS) head_col(a, out, cols, b, b0 + b, i, p, misc, sx, tokb);
          cluster_sync();
          break;
        }
        case kEQKV: {  // encoder layer l at p: q, k, v, cache row p, causal attention over rows 0..p
          if (l + 1 < s.L && p > 0) {  // the next layer's cache rows 0..p-1 into L2
            for (int j = tid; j < 2 * wk.npairs; j += kThreads) {
              const int pi = j >> 1, kv = j & 1;
              prefetch_l2(a.enc_kv + ((((size_t)(l + 1) * 2 + kv) * a.B + b0 + pair_b(pi)) * H + pair_h(pi)) *
                                         (size_t)a.T_mem * hd,
                          (unsigned)p * hd * 2);
            }
          }
          if (l == 0) {
            for (int i2 = tid; i2 < nbv * d; i2 += kThreads) {
              const int b = i2 / d, j = i2 - b * d;
              he[i2] = __bfloat162float(a.tok_emb[(size_t)tokb[b] * d + j]);
            }
            __syncthreads();
          }
          rmsnorm_x(he, a.enc_attn_norm + (size_t)l * d);
          const PY y = project(xb, P.ldx);
          const size_t plane = (size_t)a.T_mem * hd;
          auto kv_rows = [&](int kv, int pi) {
            return a.enc_kv + ((((size_t)l * 2 + kv) * a.B + b0 + pair_b(pi)) * H + pair_h(pi)) * plane;
          };
          rope_qkv(y, rope_row, true, [&](int pi, int j, bf16 kr1, bf16 kr2, bf16 v1, bf16 v2) {
            bf16* kp = kv_rows(0, pi) + (size_t)p * hd;
            bf16* vp = kv_rows(1, pi) + (size_t)p * hd;
            kp[j] = kr1;
            kp[j + half] = kr2;
            vp[j] = v1;
            vp[j + half] = v2;
          });
          __syncthreads();
          pair_attention([&](int pi) { return kv_rows(0, pi); }, [&](int pi) { return kv_rows(1, pi); }, t, true);
          cluster_sync();
          break;
        }
        case kEO:
          residual(he, project(ob, P.ldo));
          cluster_sync();
          break;
        case kEW13: {
          rmsnorm_x(he, a.enc_ffn_norm + (size_t)l * d);
          swiglu_push(project(xb, P.ldx));
          cluster_sync();
          break;
        }
        case kEW2:
          residual(he, project(mb, P.ldm));
          cluster_sync();
          break;
        case kMem: {  // memory rows of group g at p, for this CTA's pairs
          const int g = l;
          const bool final_src = s.mem_source ? g == s.L - 1 : g == 0;
          if (s.mem_source || g == 0) rmsnorm_x(he, a.enc_norm);  // RMSNorm_e of the encoder stream
          if (final_src) {  // e_p: the decoder's input, and row p of e
            bf16* ew = eb + (size_t)(i & 1) * cols * d;
            for (int i2 = tid; i2 < nbv * d; i2 += kThreads) {
              const int b = i2 / d, j = i2 - b * d;
              const bf16 v = xb[(size_t)b * P.ldx + j];
              ew[i2] = v;
              if (r == 0) a.e[((size_t)(b0 + b) * a.T_mem + p) * d + j] = v;
            }
          }
          const PY y = project(xb, P.ldx);
          const size_t plane = (size_t)a.T_mem * hd;
          for (int i2 = tid; i2 < wk.npairs * 2 * hd; i2 += kThreads) {
            const int pi = i2 / (2 * hd), rem = i2 - pi * 2 * hd, kv = rem / hd, e = rem - kv * hd;
            const int hh = pi % wk.hpc;
            const float v = y((hh * 2 + kv) * nh + (e >> 4), e & 15, pair_b(pi));
            a.mem[((((size_t)g * 2 + kv) * a.B + b0 + pair_b(pi)) * H + pair_h(pi)) * plane + (size_t)p * hd + e] =
                __float2bfloat16_rn(v);
          }
          __syncthreads();
          break;
        }
        default: {  // head (logits materialised in out: the scoring reads them many times)
          if (!hov) {
            rmsnorm_x(hcur, a.head_norm);
            project(xb, P.ldx, true);
            for (int b = r; b < nbv; b += CS) head_col(a, out, cols, b, b0 + b, i, p, misc, sx, tokb);
          } else {  // the previous step's head, s_{p} = hprev; nothing to score before the first step
            if (i > 0) {
              rmsnorm_x(hprev, a.head_norm);
            } else {
              __syncthreads();  // the gate's epilogue has read the partial sums
            }
            project(xb, P.ldx, true);
            if (i > 0)
              for (int b = r; b < nbv; b += CS) head_col(a, out, cols, b, b0 + b, i - 1, p - 1, misc, sx, tokb);
            cluster_wait();
          }
          break;
        }
      }
    }
  }
  if (tail) {  // the last step's head
    rmsnorm_x(hb + (size_t)((a.n - 1) & 1) * cols * d, a.head_norm);
    const int np = nparts_of(ph_tail), tpp = tpp_of(ph_tail);
    for (int pt = 0; pt < np; ++pt) {
      cp_async_wait1();
      __syncthreads();
      Ph sub = ph_tail;
      const int t0 = min(pt * tpp, ph_tail.nt);
      sub.nt = min(ph_tail.nt, t0 + tpp) - t0;
      proj(sub, cols, stage_of(qc), xb, P.ldx, out, part, true, t0);
      if (qc + 2 < NQ) issue_next(stage_of(qc));  // pipeline step qc + 2 (= ic_q)
      cp_async_commit();
      ++qc;
    }
    for (int b = r; b < nbv; b += CS) head_col(a, out, cols, b, b0 + b, a.n - 1, a.p0 + a.n - 1, misc, sx, tokb);
  }
  cp_async_wait0();
  // s_n: the last step's streams
  if (r == 0) {
    const float* hl = hb + (size_t)((a.n - 1) & 1) * cols * d;
    for (int i = tid; i < nbv * d; i += kThreads) a.s[(size_t)b0 * d + i] = hl[i];
  }
  cluster_sync();  // no CTA leaves while another may still address its shared memory
}

}  // namespace fused
}  // namespace rlt
