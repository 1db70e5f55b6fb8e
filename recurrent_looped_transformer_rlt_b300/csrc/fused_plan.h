// Plan of the persistent cluster decoder (dec_fused.cuh): which CTA of a
// thread-block cluster computes which rows of every projection and which
// (sequence, head) pairs of the two attentions, and the layout of its
// shared memory.  Plain C++ (no CUDA types): the library's host code and the
// host emulation of the kernel share it.
//
// One cluster of CS CTAs advances Bc sequences through all n steps of a
// decode call.  Every CTA keeps the cluster's residual streams h [Bc][d]
// (fp32) in its own shared memory, and the window keys and values of the
// (sequence, head) pairs it attends for (the state's ring, written through
// to global memory every step); a projection is split by output rows
// (16-row tiles) across the CTAs, each CTA pushes the rows it produced into
// every CTA's copy (distributed shared memory), and a cluster barrier ends
// the phase.  The self- and cross-attention queries of a head are produced
// by the CTAs that attend with that head, so attention needs no exchange
// before it.  The weights of the next phase stream from L2 into a
// double-buffered stage while the current phase runs.
#pragma once
#include <stddef.h>

#ifdef __CUDACC__
#define RLT_HD __host__ __device__
#else
#define RLT_HD
#endif

namespace rlt {
namespace fused {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCols = 16;          // sequences per cluster: two 8-column MMA tiles
constexpr int kMaxD = 1024;           // model width the kernel's row norms keep in registers
constexpr int kUnitBytes = 1024;      // one staged weight unit: 16 rows x 32 columns, bf16
constexpr size_t kMaxSmem = 232448;   // dynamic shared memory per CTA (227 KB)

// phase kinds: the decoder step's (in step order) and, in generation, the
// draw and the incremental encoder step's
enum Kind { kGate = 0, kQKV, kO, kQx, kOx, kW13, kW2, kHead, kTok, kEQKV, kEO, kEW13, kEW2, kMem };

struct Shape {
  int d, H, hd, f, L, W, V, G;
  int gate;        // 1: learned merge gate; 0: the gate discards s (h = e)
  int mem_source;  // generation: 0 every memory group from e; 1 group l from encoder layer l
};

struct Plan {
  int CS;      // CTAs per cluster
  int Bc;      // sequences per cluster (the last cluster may hold fewer)
  int nclu;    // clusters
  int cols;    // MMA columns: Bc rounded up to 8
  int hpc;     // heads per CTA
  int gph;     // CTAs per head (their sequence groups split the cluster's sequences)
  int nseq;    // most sequences a CTA attends for
  int npairs;  // most (sequence, head) pairs of a CTA
  int ldx, ldo, ldm;  // row pitches (elements) of the bf16 operand buffers
  int maxT;           // most 16-row tiles of one phase on one CTA
  int stage_units;    // units of one stage half (a phase with more runs in parts)
  size_t o_h, o_x, o_ob, o_mb, o_out, o_part, o_pr, o_ring, o_xp, o_misc, o_e, o_he, o_tok, o_sx, o_stage, total;
};

RLT_HD inline int cdivi(int a, int b) { return (a + b - 1) / b; }
RLT_HD inline int round32(int k) { return (k + 31) / 32 * 32; }
inline size_t al128(size_t x) { return (x + 127) / 128 * 128; }

// Rows of a d- or f-row projection taken by CTA r: tiles [lo, hi) of nt
// (r <= 16 and nt < 2^26, so 32-bit products; a 64-bit division costs the
// device ~100 instructions, and the kernel asks for these ranges per tile).
RLT_HD inline void part_range(int nt, int CS, int r, int* lo, int* hi) {
  *lo = r * nt / CS;
  *hi = (r + 1) * nt / CS;
}
inline int part_max(int nt, int CS) { return cdivi(nt, CS); }

// Returns 0 and fills P when the kernel supports the shape with CS CTAs per
// cluster and Bc sequences per cluster, -1 otherwise.
inline int make_plan(const Shape& s, int B, int CS, int Bc, Plan* P) {
  if (CS < 1 || CS > 16 || Bc < 1 || Bc > kMaxCols || B < 1) return -1;
  if (s.d % 32 || s.d > kMaxD || s.hd % 16 || s.hd > 128 || s.f % 8 || s.H * s.hd != s.d || s.W < 1 || s.V < 1 ||
      s.L < 1)
    return -1;
  if (!(s.hd == 16 || s.hd == 32 || s.hd == 64 || s.hd == 128)) return -1;  // lanes per key row: hd / 8
  if (!(CS % s.H == 0 || s.H % CS == 0)) return -1;
  Plan p{};
  p.CS = CS;
  p.Bc = Bc;
  p.nclu = cdivi(B, Bc);
  p.cols = cdivi(Bc, 8) * 8;
  if (CS >= s.H) {
    p.hpc = 1;
    p.gph = CS / s.H;
    p.nseq = cdivi(Bc, p.gph);
  } else {
    p.hpc = s.H / CS;
    p.gph = 0;
    p.nseq = Bc;
  }
  p.npairs = p.nseq * p.hpc;
  const int Kx = round32(s.gate ? 2 * s.d : s.d);
  p.ldx = Kx + 8;
  p.ldo = round32(s.d) + 8;
  p.ldm = round32(s.f) + 8;
  const int td = part_max(s.d / 16, CS), tf = part_max(cdivi(s.f, 16), CS), th = p.hpc * (s.hd / 16);
  const int tv = cdivi(s.V, 16);
  const int Ud = round32(s.d) / 32, Uf = round32(s.f) / 32, U2 = round32(2 * s.d) / 32;
  int maxT = 3 * th, units = 3 * th * Ud;
  auto take = [&](int t, int u) {
    if (t > maxT) maxT = t;
    if (t * u > units) units = t * u;
  };
  if (s.gate) take(td, U2);
  take(td, Ud);       // O, Ox
  take(th, Ud);       // Qx
  take(2 * tf, Ud);   // W_1 / W_3 pairs
  take(td, Uf);       // W_2
  take(tv, Ud);       // head
  p.maxT = maxT;
  size_t off = 0;
  auto put = [&](size_t bytes) {
    size_t o = off;
    off = al128(off + bytes);
    return o;
  };
  p.o_h = put((size_t)2 * p.cols * s.d * 4);
  p.o_x = put((size_t)p.cols * p.ldx * 2);
  p.o_ob = put((size_t)p.cols * p.ldo * 2);
  p.o_mb = put((size_t)p.cols * p.ldm * 2);
  p.o_out = put((size_t)maxT * 16 * p.cols * 4);
  p.o_part = put((size_t)kWarps * 2 * 32 * 4 * 4);
  p.o_pr = put((size_t)p.npairs * s.hd * 4);                        // queries of the pairs
  p.o_ring = put((size_t)s.L * p.npairs * s.W * s.hd * 2 * 2);       // the pairs' window keys and values
  p.o_xp = put((size_t)(p.npairs > kWarps ? p.npairs : kWarps) * (s.hd + 2) * 4);  // cross-attention partials
  p.o_misc = put(4096);
  p.o_e = put((size_t)2 * p.cols * s.d * 2 + (size_t)2 * s.hd * 4);  // e_p rows and RoPE rows of this step and the next
  p.o_he = put((size_t)p.cols * s.d * 4);                            // generation: the encoder's residual streams
  p.o_tok = put((size_t)p.cols * 4);                                 // generation: the drawn tokens
  p.o_sx = put((size_t)s.V * 4);                                     // the scored row's tempered logits
  // the weight stage: two halves of the largest phase's units, or, when that
  // does not fit, of what does (phases with more tiles then run in parts;
  // one tile of the widest K must fit)
  const size_t rest = off;
  if (rest + (size_t)2 * units * kUnitBytes > kMaxSmem) {
    const int room = rest < kMaxSmem ? (int)((kMaxSmem - rest) / (2 * kUnitBytes)) : 0;
    int umax = Ud > Uf ? Ud : Uf;
    if (s.gate && U2 > umax) umax = U2;
    if (room < umax) return -1;
    units = room;
  }
  p.stage_units = units;
  p.o_stage = put((size_t)2 * units * kUnitBytes);
  p.total = off;
  if (p.total > kMaxSmem) return -1;
  *P = p;
  return 0;
}

// The plan for B sequences: over the cluster sizes 16, 8, 4, 2, 1 (only
// `force` when it is not 0), the most sequences per cluster (at most 16, at
// most what spreads B over the clusters the device holds at once) whose
// working set fits in shared memory; of these the plan with the fewest waves
// of clusters, then the largest cluster (fewer weight rows per CTA).
// max_clusters(CS, smem) is the number of clusters of CS CTAs with smem
// bytes each that the device holds at once (<= 0: none).  Returns 0 and fills
// P, or -1 when no cluster size takes the shape.
template <class MaxClusters>
inline int choose_plan(const Shape& s, int B, int force, MaxClusters max_clusters, Plan* P) {
  const int cands[5] = {16, 8, 4, 2, 1};
  int best_waves = 0;
  for (int CS : cands) {
    if (force > 0 && CS != force) continue;
    Plan p;
    int Bc = B < kMaxCols ? B : kMaxCols;
    while (Bc > 0 && make_plan(s, B, CS, Bc, &p)) --Bc;
    if (Bc == 0) continue;
    const int mac = max_clusters(CS, p.total);  // at the largest Bc: the most shared memory
    if (mac <= 0) continue;
    const int spread = (B + mac - 1) / mac;
    if (spread < Bc) Bc = spread;
    if (make_plan(s, B, CS, Bc, &p)) continue;
    const int waves = (p.nclu + mac - 1) / mac;
    if (best_waves == 0 || waves < best_waves) {
      *P = p;
      best_waves = waves;
    }
  }
  return best_waves > 0 ? 0 : -1;
}

}  // namespace fused
}  // namespace rlt
