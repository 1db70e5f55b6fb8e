// Runs the persistent cluster decoder (dec_fused_kernel) under the host
// emulation of emu.h: the library's plan (fused_plan.h), grid, block, cluster
// size and shared-memory layout, with the PTX operations of fused_ptx.cuh
// replaced by this directory's stand-ins.  The generated input
// dec_fused_emu.cuh comes from the test (dec_fused.cuh with its dynamic
// shared array taken from the emulator).  Test infrastructure only.
#include "emu.h"
#include "cuda_bf16.h"
#include <vector>
#include "dec_fused_emu.cuh"

using namespace rlt;

static std::vector<bf16> tob(const float* x, size_t n) {
  std::vector<bf16> v(n);
  for (size_t i = 0; i < n; ++i) v[i] = __float2bfloat16_rn(x[i]);
  return v;
}

// sh: B, T_mem, d, H, hd, f, L, W, V, G, gate, p0, n, top_k, CS, Bc (, mem_source, seed hi, seed lo)
// fp: eps, theta, temperature
// P:  W_g, W_qkv, W_O, W_Qx, W_Ox, W_1, W_3, W_2, W_o (f32 values, stored as bf16),
//     b_g, attn_norm, xattn_norm, ffn_norm, head_norm (f32),
//     e [B][T_mem][d], mem [G][2][B][H][T_mem][hd] (f32 values, stored as bf16),
//     s [B][d] f32 (in/out), ring_k, ring_v [L][B][H][W][hd] (f32 values in/out, stored as bf16),
//     actions [B][n] i32 or null, emit_map [n] i32 or null, logits_out f32 or null,
//     logp, logp_full f32 [B][n], argmax i32 [B][n], status i32 [1]
// Returns the plan's status (-1: shape not supported), else 0.
// sh[16]: mem_source (generation)
static int run(const int* sh, const float* fp, void** P, void** Q) {
  fused::Shape S{sh[2], sh[3], sh[4], sh[5], sh[6], sh[7], sh[8], sh[9], sh[10], sh[16]};
  const int B = sh[0], T_mem = sh[1], CS = sh[14], Bc = sh[15];
  fused::Plan plan;
  if (fused::make_plan(S, B, CS, Bc, &plan)) return -1;
  const size_t d = S.d, f = S.f, L = S.L, V = S.V, H = S.H, hd = S.hd, G = S.G, W = S.W;
  const size_t dd = d * d;
  auto wb = [&](int i, size_t n) { return tob((const float*)P[i], n); };
  std::vector<bf16> Wg = wb(0, 2 * dd), Wqkv = wb(1, L * 3 * dd), WO = wb(2, L * dd), WQx = wb(3, L * dd),
                    WOx = wb(4, L * dd), W1 = wb(5, L * f * d), W3 = wb(6, L * f * d), W2 = wb(7, L * f * d),
                    Wo = wb(8, V * d);
  std::vector<bf16> e = wb(14, (size_t)B * T_mem * d), mem = wb(15, G * 2 * B * H * T_mem * hd);
  // generation: Q = tok_emb, enc_attn_norm, enc_ffn_norm, enc_norm, W_K, W_V (f32 values),
  // enc_kv [L][2][B][H][T_mem][hd] (f32 values in/out), tokens i32 [B][n], e out, mem out (f32)
  std::vector<bf16> temb, WK, WV, ekv;
  if (Q) {
    temb = tob((const float*)Q[0], V * d);
    WK = tob((const float*)Q[4], G * dd);
    WV = tob((const float*)Q[5], G * dd);
    ekv = tob((const float*)Q[6], L * 2 * B * H * T_mem * hd);
  }
  const size_t ring_n = L * B * H * W * hd;
  std::vector<bf16> rk = wb(17, ring_n), rv = wb(18, ring_n);
  fused::Args a{};
  a.W_g = Wg.data(); a.W_qkv = Wqkv.data(); a.W_O = WO.data(); a.W_Qx = WQx.data(); a.W_Ox = WOx.data();
  a.W_1 = W1.data(); a.W_3 = W3.data(); a.W_2 = W2.data(); a.W_o = Wo.data();
  a.b_g = (const float*)P[9]; a.attn_norm = (const float*)P[10]; a.xattn_norm = (const float*)P[11];
  a.ffn_norm = (const float*)P[12]; a.head_norm = (const float*)P[13];
  // (cos, sin) of every position in float from double, as the library's table
  std::vector<float2> rope((size_t)T_mem * (hd / 2));
  for (int pp = 0; pp < T_mem; ++pp)
    for (size_t i = 0; i < hd / 2; ++i) {
      const double inv = std::pow((double)fp[1], -2.0 * (double)i / (double)hd);
      rope[pp * (hd / 2) + i] = make_float2((float)std::cos(pp * inv), (float)std::sin(pp * inv));
    }
  a.rope = rope.data();
  a.e = e.data(); a.mem = mem.data();
  a.s = (float*)P[16]; a.ring_k = rk.data(); a.ring_v = rv.data();
  a.actions = (const int*)P[19]; a.emit_map = (const int*)P[20]; a.logits_out = (float*)P[21];
  a.logp = (float*)P[22]; a.logp_full = (float*)P[23]; a.argmax = (int*)P[24]; a.status = (int*)P[25];
  a.B = B; a.T_mem = T_mem; a.p0 = sh[11]; a.n = sh[12]; a.top_k = sh[13];
  a.eps = fp[0]; a.theta = fp[1]; a.scale = 1.0f / std::sqrt((float)hd); a.inv_temp = 1.0f / fp[2];
  a.sh = S;
  a.P = plan;
  if (Q) {
    a.gen = 1;
    a.tok_emb = temb.data();
    a.enc_attn_norm = (const float*)Q[1];
    a.enc_ffn_norm = (const float*)Q[2];
    a.enc_norm = (const float*)Q[3];
    a.W_K = WK.data();
    a.W_V = WV.data();
    a.enc_kv = ekv.data();
    a.tokens = (int*)Q[7];
    a.seed = ((unsigned long long)(unsigned)sh[17] << 32) | (unsigned)sh[18];
  }
  emu_launch_cluster(dim3(plan.nclu * CS), dim3(fused::kThreads), plan.total, (unsigned)CS, fused::dec_fused_kernel,
                     a);
  float* rko = (float*)P[17];
  float* rvo = (float*)P[18];
  for (size_t i = 0; i < ring_n; ++i) {
    rko[i] = __bfloat162float(rk[i]);
    rvo[i] = __bfloat162float(rv[i]);
  }
  if (Q) {
    auto back = [](const std::vector<bf16>& v, void* dst) {
      float* o = (float*)dst;
      for (size_t i = 0; i < v.size(); ++i) o[i] = __bfloat162float(v[i]);
    };
    back(ekv, Q[6]);
    back(e, Q[8]);
    back(mem, Q[9]);
  }
  return 0;
}

extern "C" int fused_emu(const int* sh, const float* fp, void** P) { return run(sh, fp, P, nullptr); }

// generation: sh[16] mem_source, sh[17], sh[18] the seed's high and low words
extern "C" int fused_gen_emu(const int* sh, const float* fp, void** P, void** Q) { return run(sh, fp, P, Q); }
