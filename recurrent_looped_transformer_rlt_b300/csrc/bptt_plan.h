// Backpropagation through time of the RLT decoder recurrence (teacher
// forced, full or truncated at named detach points): the order of the
// operations, the workspace layout and the bookkeeping of the window's
// query-side records and of the step blocks, written once over a set of primitive
// operations (Ops, implemented by the device kernels of bptt.cuh).  Plain
// host C++: no CUDA types.
//
// What is differentiated (the decoder of "Understanding and Applying the
// Recurrent Looped Transformer Architecture", "How the Architecture Works",
// started at H_0 = (s_*, empty cache)):
//   L = - sum_t sum_b lp_t(a_{b,t}),  lp_t = tempered (top-k) log-softmax of
//   W_o RMSNorm_o(s_t) at the action,
// with respect to every decoder parameter, s_*, the encoder output e and the
// memory M.  Gradients pass through s, the window keys and values and the
// memory ("Princeton Researcher Proposes Recurrent Looped Transformer ...",
// training paragraph: the state Jacobian has cross terms through the decoder
// keys and values, so a truncation names each tensor it detaches;
// "Current-Policy Reinforcement Learning Replay": detaching the recurrent
// outputs, the decoder key-value entries or the memory is an approximation).
//
// Schedule.
//  * A forward pass records s_t for every step, the keys and values of every
//    position and layer, and every layer's cross-attention output and
//    log-sum-exp.
//  * The reverse pass visits t = n..1: it recomputes step t's activations
//    from s_{t-1}, the recorded keys/values and the recorded cross-attention
//    results (the same kernels, so bitwise the recorded values; the memory is
//    not read for this), runs the head and the layers backwards, and hands
//    d s_{t-1} to step t-1.
//  * The window keys and values of position j receive gradient from the
//    queries of positions j..j+W-1, whose steps the reverse pass visits
//    first.  Each step keeps, per layer, the query side of its window
//    attention - the query (after RoPE), the output gradient, the LSE and
//    D = g.o - in a ring of W slots (slot p mod W); position j's QKV backward
//    computes its key/value gradient in one pass over the records of
//    positions j..j+W-1.  Step p+1 overwrites the record of position p+W,
//    whose keys p+1..p+W are consumed by then.
//  * Steps are grouped in blocks of S consecutive steps.  Within a block each
//    step writes, into its own column slot, the transposed GEMM inputs X and
//    output gradients dY of every projection ([features][S * Bp]), and its
//    cross-attention query, output gradient and D = g.o.  At the end of a
//    block, one GEMM per projection adds dY^T X over the block's S * B rows
//    to the weight gradient, and one key-parallel pass adds the block's
//    contributions to the memory gradient (which feeds nothing in the
//    recurrence, so it can wait).
//  * A step is replayable: the operations read the step's position from a
//    device cell (Ops::step's last operation moves it) and get pointers that
//    depend only on the block slot, so the device Ops can capture the
//    recording step and each reverse slot once and replay them.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace bpplan {

struct Shape {
  int B, n, T_mem;                 // sequences, steps, positions of e / mem
  int d, H, hd, f, L, W, V, G;     // model
  bool gate_learned;               // false: z = 0 (u_t = e_t)
  float eps, theta, scale, inv_temp;
  int top_k;
  int Bp;                          // columns per step slot of the transposed operands (B rounded up; zero past B)
  int S;                           // steps per block (weight and memory gradients are added once per block)
  int chunk;                       // keys per warp of the split memory attention (scratch sizing)
};

struct Detach {
  int s_every;   // > 0: s_t enters step t+1 as a constant when t % s_every == 0
  bool cache;    // window keys/values of earlier positions enter as constants
  bool memory;   // the memory enters as a constant (no memory gradient)
};

// Decoder parameters: matrices in the storage type, gains, bias and s_* fp32.
template <typename T>
struct Params {
  const T *W_g, *W_qkv, *W_O, *W_Qx, *W_Ox, *W_1, *W_3, *W_2, *W_o;
  const float *b_g, *s_star, *attn_norm, *xattn_norm, *ffn_norm, *head_norm;
};

// Gradients (fp32, the parameters' shapes); zeroed and accumulated by run().
struct Grads {
  float *W_g, *b_g, *W_qkv, *W_O, *W_Qx, *W_Ox, *W_1, *W_3, *W_2, *W_o;
  float *attn_norm, *xattn_norm, *ffn_norm, *head_norm, *s_star;
};

// Byte offsets into the workspace.
struct Layout {
  size_t wt_g, wt_qkv, wt_O, wt_Qx, wt_Ox, wt_13, wt_2, wt_o;  // transposed weights
  size_t hist;          // [L][2][B][H][n][hd] keys (after RoPE) and values of every position
  size_t xo_all;        // [n][L][B][d] cross-attention outputs (storage type)
  size_t lse2_all;      // [n][L][B][H] f32 their log-sum-exp
  size_t s_all;         // [n+1][B][d] f32: s_0 = s_*, s_1..s_n
  size_t lp;            // [B][n] f32
  size_t qR, gR, lR, DR;  // [L][W][B][d], [L][W][B][d], [L][W][B][H], [L][W][B][H] f32 query-side records
  size_t zero_begin;    // [zero_begin, total) starts at zero
  // one step's activations
  size_t xg, zpre, z;
  size_t hA, hX, hF;    // [L][B][d] f32 residual stream into attention, cross-attention, FFN
  size_t rA, rX, rF, rO;
  size_t a, c, bb, oq;
  size_t g, u, m;
  size_t sn, qkv, logits;
  // block operands: [rows][S * Bp], step slot s at columns [s * Bp, (s + 1) * Bp)
  size_t xgT, aT, cT, bbT, oT, oxT, mT, snT;
  size_t dlT, dzT, dhfT, dhxT, dhaT, dqxT, dguT, dqkvT;
  size_t qxS, gxS, DxS;  // [S][L][B][d], [S][L][B][d] f32, [S][L][B][H] f32
  size_t part;          // f32 split-attention partials: [B][H][splits][hd + 2] or [3 hd + 1] (window backward)
  // gradient scratch
  size_t ds, dh, dx, dY, dY2;
  size_t pos, xo_step, g_step, s_cur;  // position cell (int); [L][B][d] T; [B][d] f32; [B][d] f32
  size_t total;
};

inline size_t bp_align(size_t x) { return (x + 255) / 256 * 256; }

// Workspace layout after a header of hdr bytes; es = bytes of the storage type.
inline Layout layout(const Shape& S, size_t es, size_t hdr) {
  const size_t B = S.B, n = S.n, d = S.d, H = S.H, hd = S.hd, f = S.f, L = S.L, W = S.W, V = S.V;
  const size_t Bd = B * d, ldT = (size_t)S.S * S.Bp, SB = S.S;
  Layout Lw{};
  size_t off = bp_align(hdr);
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = bp_align(off + bytes);
    return o;
  };
  Lw.wt_g = take(es * 2 * d * d);
  Lw.wt_qkv = take(es * L * 3 * d * d);
  Lw.wt_O = take(es * L * d * d);
  Lw.wt_Qx = take(es * L * d * d);
  Lw.wt_Ox = take(es * L * d * d);
  Lw.wt_13 = take(es * L * 2 * f * d);
  Lw.wt_2 = take(es * L * f * d);
  Lw.wt_o = take(es * V * d);
  Lw.hist = take(es * L * 2 * B * H * n * hd);
  Lw.xo_all = take(es * n * L * Bd);
  Lw.lse2_all = take(4 * n * L * B * H);
  Lw.s_all = take(4 * (n + 1) * Bd);
  Lw.lp = take(4 * B * n);
  Lw.qR = take(4 * L * W * Bd);
  Lw.gR = take(4 * L * W * Bd);
  Lw.lR = take(4 * L * W * B * H);
  Lw.DR = take(4 * L * W * B * H);
  Lw.zero_begin = off;
  Lw.xg = take(es * 2 * Bd);
  Lw.zpre = take(4 * Bd);
  Lw.z = take(4 * Bd);
  Lw.hA = take(4 * L * Bd);
  Lw.hX = take(4 * L * Bd);
  Lw.hF = take(4 * L * Bd);
  Lw.rA = take(4 * L * B);
  Lw.rX = take(4 * L * B);
  Lw.rF = take(4 * L * B);
  Lw.rO = take(4 * B);
  Lw.a = take(es * L * Bd);
  Lw.c = take(es * L * Bd);
  Lw.bb = take(es * L * Bd);
  Lw.oq = take(es * L * Bd);
  Lw.g = take(4 * L * B * f);
  Lw.u = take(4 * L * B * f);
  Lw.m = take(es * L * B * f);
  Lw.sn = take(es * Bd);
  Lw.qkv = take(4 * 3 * Bd);
  Lw.logits = take(4 * B * V);
  Lw.xgT = take(es * 2 * d * ldT);
  Lw.aT = take(es * L * d * ldT);
  Lw.cT = take(es * L * d * ldT);
  Lw.bbT = take(es * L * d * ldT);
  Lw.oT = take(es * L * d * ldT);
  Lw.oxT = take(es * L * d * ldT);
  Lw.mT = take(es * L * f * ldT);
  Lw.snT = take(es * d * ldT);
  Lw.dlT = take(es * V * ldT);
  Lw.dzT = take(es * d * ldT);
  Lw.dhfT = take(es * L * d * ldT);
  Lw.dhxT = take(es * L * d * ldT);
  Lw.dhaT = take(es * L * d * ldT);
  Lw.dqxT = take(es * L * d * ldT);
  Lw.dguT = take(es * L * 2 * f * ldT);
  Lw.dqkvT = take(es * L * 3 * d * ldT);
  Lw.qxS = take(4 * SB * L * Bd);
  Lw.gxS = take(4 * SB * L * Bd);
  Lw.DxS = take(4 * SB * L * B * H);
  const size_t nsplit = S.chunk > 0 ? (n + S.chunk - 1) / S.chunk : 1;
  const size_t wsplit = S.chunk > 0 ? (W + S.chunk - 1) / S.chunk : 1;
  const size_t per_pair = nsplit * (hd + 2) > wsplit * (3 * hd + 1) ? nsplit * (hd + 2) : wsplit * (3 * hd + 1);
  Lw.part = take(4 * B * H * per_pair);
  Lw.ds = take(4 * Bd);
  Lw.dh = take(4 * Bd);
  Lw.dx = take(4 * Bd);
  size_t ny = 3 * d;
  if (2 * f > ny) ny = 2 * f;
  if (V > ny) ny = V;
  Lw.dY = take(es * B * ny);
  Lw.dY2 = take(es * B * 2 * f);
  Lw.pos = take(sizeof(int));
  Lw.xo_step = take(es * L * Bd);
  Lw.g_step = take(4 * Bd);
  Lw.s_cur = take(4 * Bd);
  Lw.total = off;
  return Lw;
}

#define RLT_BP_TRY(x)          \
  do {                         \
    int rc_ = (x);             \
    if (rc_) return rc_;       \
  } while (0)

// Inputs/outputs of one call (device pointers for the device Ops).
template <typename T>
struct Io {
  const T* e;              // [B][T_mem][d]
  const T* mem;            // [G][2][B][H][T_mem][hd]
  const int32_t* actions;  // [B][n]
  float* loss;             // [1]
  float* lp_out;           // [B][n] or null
  float* d_e;              // [B][T_mem][d] or null
  float* d_mem;            // [G][2][B][H][T_mem][hd] or null
};

template <class Ops>
int run(Ops& k, const Shape& S, const Detach& D, const Params<typename Ops::T>& P, const Io<typename Ops::T>& io,
        const Grads& G, char* ws, const Layout& Lw) {
  using T = typename Ops::T;
  const int B = S.B, n = S.n, d = S.d, H = S.H, hd = S.hd, f = S.f, L = S.L, W = S.W, V = S.V, Bp = S.Bp;
  const int SB = S.S;
  const size_t Bd = (size_t)B * d, BH = (size_t)B * H, dd = (size_t)d * d, fd = (size_t)f * d;
  const int ldT = SB * Bp;
  const size_t dT = (size_t)d * ldT;  // one layer of a [L][d][S * Bp] block operand
  auto F = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  auto X = [&](size_t off) { return reinterpret_cast<T*>(ws + off); };
  T* wt_g = X(Lw.wt_g);
  T* wt_qkv = X(Lw.wt_qkv);
  T* wt_O = X(Lw.wt_O);
  T* wt_Qx = X(Lw.wt_Qx);
  T* wt_Ox = X(Lw.wt_Ox);
  T* wt_13 = X(Lw.wt_13);
  T* wt_2 = X(Lw.wt_2);
  T* wt_o = X(Lw.wt_o);
  T* hist = X(Lw.hist);
  T* xo_all = X(Lw.xo_all);
  float* lse2_all = F(Lw.lse2_all);
  float* s_all = F(Lw.s_all);
  float* lp = F(Lw.lp);
  const size_t plane_h = (size_t)B * H * n * hd;       // one key or value plane of the history
  const size_t plane_m = (size_t)B * H * S.T_mem * hd;  // of the memory
  const bool want_dmem = io.d_mem && !D.memory;

  // ---- set up: zeroed scratch and gradients, transposed weights, s_0
  RLT_BP_TRY(k.zero(ws + Lw.zero_begin, Lw.total - Lw.zero_begin));
  RLT_BP_TRY(k.zero(G.W_g, 4 * 2 * dd));
  RLT_BP_TRY(k.zero(G.b_g, 4 * (size_t)d));
  RLT_BP_TRY(k.zero(G.W_qkv, 4 * (size_t)L * 3 * dd));
  RLT_BP_TRY(k.zero(G.W_O, 4 * (size_t)L * dd));
  RLT_BP_TRY(k.zero(G.W_Qx, 4 * (size_t)L * dd));
  RLT_BP_TRY(k.zero(G.W_Ox, 4 * (size_t)L * dd));
  RLT_BP_TRY(k.zero(G.W_1, 4 * (size_t)L * fd));
  RLT_BP_TRY(k.zero(G.W_3, 4 * (size_t)L * fd));
  RLT_BP_TRY(k.zero(G.W_2, 4 * (size_t)L * fd));
  RLT_BP_TRY(k.zero(G.W_o, 4 * (size_t)V * d));
  RLT_BP_TRY(k.zero(G.attn_norm, 4 * (size_t)L * d));
  RLT_BP_TRY(k.zero(G.xattn_norm, 4 * (size_t)L * d));
  RLT_BP_TRY(k.zero(G.ffn_norm, 4 * (size_t)L * d));
  RLT_BP_TRY(k.zero(G.head_norm, 4 * (size_t)d));
  RLT_BP_TRY(k.zero(G.s_star, 4 * (size_t)d));
  if (io.d_e) RLT_BP_TRY(k.zero(io.d_e, 4 * Bd * S.T_mem));
  if (io.d_mem) RLT_BP_TRY(k.zero(io.d_mem, 4 * (size_t)S.G * 2 * plane_m));
  RLT_BP_TRY(k.transpose(P.W_g, d, 2 * d, 2 * d, wt_g, d));
  for (int l = 0; l < L; ++l) {
    RLT_BP_TRY(k.transpose(P.W_qkv + l * 3 * dd, 3 * d, d, d, wt_qkv + l * 3 * dd, 3 * d));
    RLT_BP_TRY(k.transpose(P.W_O + l * dd, d, d, d, wt_O + l * dd, d));
    RLT_BP_TRY(k.transpose(P.W_Qx + l * dd, d, d, d, wt_Qx + l * dd, d));
    RLT_BP_TRY(k.transpose(P.W_Ox + l * dd, d, d, d, wt_Ox + l * dd, d));
    RLT_BP_TRY(k.transpose(P.W_1 + l * fd, f, d, d, wt_13 + l * 2 * fd, 2 * f));
    RLT_BP_TRY(k.transpose(P.W_3 + l * fd, f, d, d, wt_13 + l * 2 * fd + f, 2 * f));
    RLT_BP_TRY(k.transpose(P.W_2 + l * fd, d, f, f, wt_2 + l * fd, d));
  }
  RLT_BP_TRY(k.transpose(P.W_o, V, d, d, wt_o, V));
  RLT_BP_TRY(k.bcast_rows(s_all, P.s_star, B, d));

  // ---- one step, written so that it can be captured once and replayed:
  // every quantity that depends on the step's position p is read on the
  // device from the position cell (*pos), and every pointer handed to an
  // operation depends only on the step's slot.  slot < 0: the recording pass
  // (cross-attention computed and recorded, s_t stored, no transposed
  // operands); slot >= 0: recomputation in the reverse pass (recorded
  // cross-attention, operands into the slot).
  int* pos = reinterpret_cast<int*>(ws + Lw.pos);
  T* xg = X(Lw.xg);
  float* zpre = F(Lw.zpre);
  float* z = F(Lw.z);
  float* qkv = F(Lw.qkv);
  T* xo_step = X(Lw.xo_step);
  // column slot of a block operand: rows_before rows into the buffer at off
  auto col = [&](size_t off, size_t rows_before, int slot) -> T* {
    return slot < 0 ? nullptr : X(off) + rows_before * ldT + (size_t)slot * Bp;
  };
  auto fwd = [&](int slot) -> int {
    if (S.gate_learned) {
      RLT_BP_TRY(k.merge_in(io.e, S.T_mem, pos, s_all, B, d, xg, col(Lw.xgT, 0, slot), ldT));
      RLT_BP_TRY(k.gemm(xg, 2 * d, B, 2 * d, P.W_g, 2 * d, d, zpre, d, false));
    }
    RLT_BP_TRY(k.merge_out(S.gate_learned ? zpre : nullptr, P.b_g, io.e, S.T_mem, pos, s_all, B, d, z, F(Lw.hA)));
    for (int l = 0; l < L; ++l) {
      float* hA = F(Lw.hA) + l * Bd;
      float* hX = F(Lw.hX) + l * Bd;
      float* hF = F(Lw.hF) + l * Bd;
      T* Kl = hist + (size_t)(2 * l) * plane_h;
      T* Vl = hist + (size_t)(2 * l + 1) * plane_h;
      // window self-attention (q and the LSE into this position's record slot)
      RLT_BP_TRY(k.rms_fwd(hA, nullptr, 0, P.attn_norm + (size_t)l * d, B, d, S.eps, F(Lw.rA) + l * B,
                           X(Lw.a) + l * Bd, col(Lw.aT, (size_t)l * d, slot), ldT));
      RLT_BP_TRY(k.gemm(X(Lw.a) + l * Bd, d, B, d, P.W_qkv + l * 3 * dd, d, 3 * d, qkv, 3 * d, false));
      RLT_BP_TRY(k.swa_fwd(qkv, pos, W, B, H, hd, S.theta, S.scale, F(Lw.qR) + (size_t)l * W * Bd,
                           F(Lw.lR) + (size_t)l * W * BH, Kl, Vl, n, X(Lw.oq) + l * Bd,
                           col(Lw.oT, (size_t)l * d, slot), ldT, F(Lw.part)));
      RLT_BP_TRY(k.gemm_res(X(Lw.oq) + l * Bd, d, B, d, P.W_O + l * dd, d, d, hA, hX, d));
      // cross-attention to memory positions 0..p (recorded in the first pass)
      RLT_BP_TRY(k.rms_fwd(hX, nullptr, 0, P.xattn_norm + (size_t)l * d, B, d, S.eps, F(Lw.rX) + l * B,
                           X(Lw.c) + l * Bd, col(Lw.cT, (size_t)l * d, slot), ldT));
      float* qx = slot < 0 ? qkv : F(Lw.qxS) + ((size_t)slot * L + l) * Bd;
      RLT_BP_TRY(k.gemm(X(Lw.c) + l * Bd, d, B, d, P.W_Qx + l * dd, d, d, qx, d, false));
      T* xo = xo_step + l * Bd;  // this step's output row (the record is [p][l])
      if (slot < 0) {
        const int g = S.G == 1 ? 0 : l;
        RLT_BP_TRY(k.attn_fwd(qx, io.mem + (size_t)(2 * g) * plane_m, io.mem + (size_t)(2 * g + 1) * plane_m,
                              S.T_mem, pos, n, B, H, hd, S.scale, lse2_all + l * BH, xo_all + l * Bd, L, xo,
                              F(Lw.part)));
      } else {
        RLT_BP_TRY(k.tcopy(xo_all + l * Bd, L, pos, B, d, xo, col(Lw.oxT, (size_t)l * d, slot), ldT));
      }
      RLT_BP_TRY(k.gemm_res(xo, d, B, d, P.W_Ox + l * dd, d, d, hX, hF, d));
      // SwiGLU feed-forward
      RLT_BP_TRY(k.rms_fwd(hF, nullptr, 0, P.ffn_norm + (size_t)l * d, B, d, S.eps, F(Lw.rF) + l * B,
                           X(Lw.bb) + l * Bd, col(Lw.bbT, (size_t)l * d, slot), ldT));
      float* gl = F(Lw.g) + (size_t)l * B * f;
      float* ul = F(Lw.u) + (size_t)l * B * f;
      RLT_BP_TRY(k.gemm(X(Lw.bb) + l * Bd, d, B, d, P.W_1 + l * fd, d, f, gl, f, false));
      RLT_BP_TRY(k.gemm(X(Lw.bb) + l * Bd, d, B, d, P.W_3 + l * fd, d, f, ul, f, false));
      RLT_BP_TRY(k.swiglu_fwd(gl, ul, B, f, X(Lw.m) + (size_t)l * B * f, col(Lw.mT, (size_t)l * f, slot), ldT));
      // the last layer's output is s_t, recorded by the first pass
      if (slot >= 0 && l + 1 == L) continue;
      float* next = (l + 1 < L) ? F(Lw.hA) + (l + 1) * Bd : F(Lw.s_cur);
      RLT_BP_TRY(k.gemm_res(X(Lw.m) + (size_t)l * B * f, f, B, f, P.W_2 + l * fd, f, d, hF, next, d));
    }
    if (slot < 0) RLT_BP_TRY(k.put_row(s_all, pos, 1, F(Lw.s_cur), B * d));  // s_{p+1}
    return 0;
  };

  // ---- end of a block of nb steps whose highest position is p_hi (step slot
  // s holds position p_hi - s): weight gradients over the block's rows, then
  // the block's memory-gradient contributions
  auto flush = [&](int nb, int p_hi) -> int {
    const int K = nb * Bp;
    RLT_BP_TRY(k.gemm(X(Lw.dlT), ldT, V, K, X(Lw.snT), ldT, d, G.W_o, d, true));
    if (S.gate_learned) RLT_BP_TRY(k.gemm(X(Lw.dzT), ldT, d, K, X(Lw.xgT), ldT, 2 * d, G.W_g, 2 * d, true));
    for (int l = 0; l < L; ++l) {
      const T* bbT = X(Lw.bbT) + l * dT;
      const T* dguT = X(Lw.dguT) + (size_t)l * 2 * f * ldT;
      RLT_BP_TRY(k.gemm(X(Lw.dhfT) + l * dT, ldT, d, K, X(Lw.mT) + (size_t)l * f * ldT, ldT, f, G.W_2 + l * fd, f,
                        true));
      RLT_BP_TRY(k.gemm(dguT, ldT, f, K, bbT, ldT, d, G.W_1 + l * fd, d, true));
      RLT_BP_TRY(k.gemm(dguT + (size_t)f * ldT, ldT, f, K, bbT, ldT, d, G.W_3 + l * fd, d, true));
      RLT_BP_TRY(k.gemm(X(Lw.dhxT) + l * dT, ldT, d, K, X(Lw.oxT) + l * dT, ldT, d, G.W_Ox + l * dd, d, true));
      RLT_BP_TRY(k.gemm(X(Lw.dqxT) + l * dT, ldT, d, K, X(Lw.cT) + l * dT, ldT, d, G.W_Qx + l * dd, d, true));
      RLT_BP_TRY(k.gemm(X(Lw.dhaT) + l * dT, ldT, d, K, X(Lw.oT) + l * dT, ldT, d, G.W_O + l * dd, d, true));
      RLT_BP_TRY(k.gemm(X(Lw.dqkvT) + (size_t)l * 3 * dT, ldT, 3 * d, K, X(Lw.aT) + l * dT, ldT, d,
                        G.W_qkv + l * 3 * dd, d, true));
    }
    if (want_dmem) {
      for (int g = 0; g < S.G; ++g) {
        const int l0 = S.G == 1 ? 0 : g, l1 = S.G == 1 ? L : g + 1;
        RLT_BP_TRY(k.mem_grad(io.mem + (size_t)(2 * g) * plane_m, io.mem + (size_t)(2 * g + 1) * plane_m, S.T_mem,
                              F(Lw.qxS), F(Lw.gxS), lse2_all, F(Lw.DxS), L, l0, l1, nb, p_hi, B, H, hd, S.scale,
                              io.d_mem + (size_t)(2 * g) * plane_m, io.d_mem + (size_t)(2 * g + 1) * plane_m));
      }
    }
    return 0;
  };

  // ---- the reverse step of slot `slot` at the position in the cell
  float* ds = F(Lw.ds);  // d L / d s_t from step t+1 (then from the head too)
  float* dh = F(Lw.dh);
  float* dx = F(Lw.dx);
  T* dY = X(Lw.dY);
  T* dY2 = X(Lw.dY2);
  float* g_step = F(Lw.g_step);
  auto rev = [&](int slot) -> int {
    RLT_BP_TRY(fwd(slot));
    // head: logits = W_o RMSNorm_o(s_t) (s_t = s_all row p + 1); d logits of -lp
    RLT_BP_TRY(k.rms_fwd(s_all, pos, 1, P.head_norm, B, d, S.eps, F(Lw.rO), X(Lw.sn), col(Lw.snT, 0, slot), ldT));
    RLT_BP_TRY(k.gemm(X(Lw.sn), d, B, d, P.W_o, d, V, F(Lw.logits), V, false));
    RLT_BP_TRY(k.head_bwd(F(Lw.logits), B, V, io.actions, n, pos, S.inv_temp, S.top_k, lp, dY,
                          col(Lw.dlT, 0, slot), ldT));
    RLT_BP_TRY(k.gemm(dY, V, B, V, wt_o, V, d, dx, d, false));
    // (each RMSNorm backward also writes the updated gradient as the next
    // section's dY operand and its transposed slot)
    RLT_BP_TRY(k.rms_bwd(s_all, pos, 1, F(Lw.rO), P.head_norm, dx, B, d, ds, G.head_norm, dY,
                         col(Lw.dhfT, (size_t)(L - 1) * d, slot), ldT));
    RLT_BP_TRY(k.copy(dh, ds, 4 * Bd));
    for (int l = L - 1; l >= 0; --l) {
      const float* hA = F(Lw.hA) + l * Bd;
      const float* hX = F(Lw.hX) + l * Bd;
      const float* hF = F(Lw.hF) + l * Bd;
      const T* Kl = hist + (size_t)(2 * l) * plane_h;
      const T* Vl = hist + (size_t)(2 * l + 1) * plane_h;
      // FFN: h_out = hF + m W_2^T, m = silu(bb W_1^T) * (bb W_3^T); dY holds dh
      RLT_BP_TRY(k.gemm_swiglu_bwd(dY, d, B, d, wt_2 + l * fd, d, f, F(Lw.g) + (size_t)l * B * f,
                                   F(Lw.u) + (size_t)l * B * f, dY2, col(Lw.dguT, (size_t)l * 2 * f, slot), ldT));
      RLT_BP_TRY(k.gemm(dY2, 2 * f, B, 2 * f, wt_13 + l * 2 * fd, 2 * f, d, dx, d, false));
      RLT_BP_TRY(k.rms_bwd(hF, nullptr, 0, F(Lw.rF) + l * B, P.ffn_norm + (size_t)l * d, dx, B, d, dh,
                           G.ffn_norm + (size_t)l * d, dY, col(Lw.dhxT, (size_t)l * d, slot), ldT));
      // cross-attention: hF = hX + ox W_Ox^T; the query gradient now, the
      // memory gradient at the end of the block
      float* gx = F(Lw.gxS) + ((size_t)slot * L + l) * Bd;
      RLT_BP_TRY(k.gemm(dY, d, B, d, wt_Ox + l * dd, d, d, gx, d, false));
      const int g = S.G == 1 ? 0 : l;
      RLT_BP_TRY(k.attn_bwd(F(Lw.qxS) + ((size_t)slot * L + l) * Bd, gx, xo_step + l * Bd, lse2_all + l * BH, L,
                            io.mem + (size_t)(2 * g) * plane_m, io.mem + (size_t)(2 * g + 1) * plane_m, S.T_mem, pos,
                            n, B, H, hd, S.scale, F(Lw.DxS) + ((size_t)slot * L + l) * BH, dY,
                            col(Lw.dqxT, (size_t)l * d, slot), ldT, F(Lw.part)));
      RLT_BP_TRY(k.gemm(dY, d, B, d, wt_Qx + l * dd, d, d, dx, d, false));
      RLT_BP_TRY(k.rms_bwd(hX, nullptr, 0, F(Lw.rX) + l * B, P.xattn_norm + (size_t)l * d, dx, B, d, dh,
                           G.xattn_norm + (size_t)l * d, dY, col(Lw.dhaT, (size_t)l * d, slot), ldT));
      // window self-attention: hX = hA + o W_O^T.  The output gradient goes to
      // this step's record with the query, LSE and D; the query gradient over
      // the window and position p's key/value gradient from the records of
      // positions p..p+W-1 (only its own with the cache detached), both back
      // through RoPE into d qkv
      RLT_BP_TRY(k.gemm(dY, d, B, d, wt_O + l * dd, d, d, g_step, d, false));
      RLT_BP_TRY(k.swa_bwd(Kl, Vl, n, pos, W, D.cache, X(Lw.oq) + l * Bd, g_step, F(Lw.qR) + (size_t)l * W * Bd,
                           F(Lw.gR) + (size_t)l * W * Bd, F(Lw.lR) + (size_t)l * W * BH,
                           F(Lw.DR) + (size_t)l * W * BH, B, H, hd, S.scale, S.theta, dY,
                           col(Lw.dqkvT, (size_t)l * 3 * d, slot), ldT, F(Lw.part)));
      RLT_BP_TRY(k.gemm(dY, 3 * d, B, 3 * d, wt_qkv + l * 3 * dd, 3 * d, d, dx, d, false));
      // (layer l-1's FFN section reads dh as its dY; the merge reads dh)
      RLT_BP_TRY(k.rms_bwd(hA, nullptr, 0, F(Lw.rA) + l * B, P.attn_norm + (size_t)l * d, dx, B, d, dh,
                           G.attn_norm + (size_t)l * d, l > 0 ? dY : nullptr,
                           l > 0 ? col(Lw.dhfT, (size_t)(l - 1) * d, slot) : nullptr, ldT));
    }
    // merge u = z s_{t-1} + (1 - z) e_t, z = sigmoid(W_g [e_t; s_{t-1}] + b_g)
    RLT_BP_TRY(k.merge_bwd(dh, z, io.e, S.T_mem, pos, s_all, B, d, S.gate_learned, dY, col(Lw.dzT, 0, slot), ldT,
                           G.b_g, io.d_e, ds));
    if (S.gate_learned) RLT_BP_TRY(k.gemm_merge_bwd(dY, d, B, d, wt_g, d, d, S.T_mem, pos, io.d_e, ds));
    // s_{t-1} = s_p detached after its step: no gradient from this merge
    if (D.s_every > 0) RLT_BP_TRY(k.zero_if_detached(ds, pos, D.s_every, B * d));
    return 0;
  };

  // ---- forward pass: s_t, every position's keys/values, cross-attention
  // results; one replayable step per position
  RLT_BP_TRY(k.set_pos(pos, 0));
  for (int t = 1; t <= n; ++t)
    RLT_BP_TRY(k.step(-1, [&]() -> int {
      RLT_BP_TRY(fwd(-1));
      return k.add_pos(pos, 1);
    }));

  // ---- reverse pass, one replayable step per slot of a block
  RLT_BP_TRY(k.set_pos(pos, n - 1));
  int slot = 0, p_hi = n - 1;
  for (int t = n; t >= 1; --t) {
    RLT_BP_TRY(k.step(slot, [&]() -> int {
      RLT_BP_TRY(rev(slot));
      return k.add_pos(pos, -1);
    }));
    if (++slot == SB || t == 1) {
      RLT_BP_TRY(flush(slot, p_hi));
      slot = 0;
      p_hi = t - 2;
    }
  }
  RLT_BP_TRY(k.colsum(ds, B, d, G.s_star));
  RLT_BP_TRY(k.loss_sum(lp, io.actions, B, n, V, io.loss));
  if (io.lp_out) RLT_BP_TRY(k.copy(io.lp_out, lp, 4 * (size_t)B * n));
  return 0;
}

}  // namespace bpplan
