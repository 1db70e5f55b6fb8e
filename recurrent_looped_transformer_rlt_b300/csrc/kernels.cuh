// Non-GEMM kernels of the RLT encoder and decoder step.
//
// Notation: B sequences, T positions, d = H * hd, L layers, W window, V vocab.
// T_ (template) is the storage type: float for fp32 models, bf16 for bf16
// models (fp32 arithmetic, bf16 storage rounded to nearest even).
#pragma once

#include "common.cuh"
#include "ptx.cuh"
#include "sampling.cuh"

namespace rlt {

// ---------------------------------------------------------------------------
// RoPE table: angle(p, i) = p * theta^(-2i/hd), evaluated in double and stored
// as (cos, sin) float pairs for positions [p0, p0 + n).
// Page "Princeton Researcher Proposes...": self-attention of encoder and
// decoder is positional; rotate-half RoPE is the reading taken.
__global__ void rope_table_kernel(float2* tab, int p0, int n, int half, double theta) {
  int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n * half) return;
  int pi = idx / half, i = idx - pi * half;
  int p = p0 + pi;
  double inv = pow(theta, -2.0 * (double)i / (double)(2 * half));
  double s, c;
  sincos((double)p * inv, &s, &c);
  tab[(size_t)p * half + i] = make_float2((float)c, (float)s);
}

// ---------------------------------------------------------------------------
// Token embedding: h[r, :] = tok_emb[tok[r], :] (fp32 residual stream).
template <typename T_>
__global__ void embed_kernel(const int* __restrict__ tok, const T_* __restrict__ emb, float* __restrict__ h,
                             int rows, int d, int V, int* status) {
  int r = blockIdx.x;
  if (r >= rows) return;
  int x = tok[r];
  if (x < 0 || x >= V) {
    if (threadIdx.x == 0) set_error(status, kErrBounds);
    for (int j = threadIdx.x; j < d; j += blockDim.x) h[(size_t)r * d + j] = 0.f;
    return;
  }
  for (int j = threadIdx.x; j < d; j += blockDim.x) h[(size_t)r * d + j] = to_f32(emb[(size_t)x * d + j]);
}

// Token embedding of bf16 models with the first RMSNorm: h[r] = tok_emb[tok[r]]
// (fp32) and x[r] = bf16(h[r] / sqrt(mean(h[r]^2) + eps) * g).  Block = one
// row, d/4 threads, 4 columns each (d a multiple of 128).
__global__ void embed_norm_kernel(const int* __restrict__ tok, const bf16* __restrict__ emb, float* __restrict__ h,
                                  bf16* __restrict__ xo, const float* __restrict__ g, int rows, int d, int V,
                                  float eps, int* status) {
  __shared__ float red[32];
  const int r = blockIdx.x, c = threadIdx.x * 4;
  if (r >= rows) return;
  int t = tok[r];
  const bool bad = (t < 0 || t >= V);
  if (bad && threadIdx.x == 0) set_error(status, kErrBounds);
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!bad) {
    const uint2 u = *reinterpret_cast<const uint2*>(emb + (size_t)t * d + c);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    v = make_float4(a.x, a.y, b.x, b.y);
  }
  *reinterpret_cast<float4*>(h + (size_t)r * d + c) = v;
  float q = warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = q;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
  const float rs = rsqrtf(tot / (float)d + eps);
  const float4 gg = *reinterpret_cast<const float4*>(g + c);
  __nv_bfloat162 x01 = __floats2bfloat162_rn(v.x * rs * gg.x, v.y * rs * gg.y);
  __nv_bfloat162 x23 = __floats2bfloat162_rn(v.z * rs * gg.z, v.w * rs * gg.w);
  uint2 xp;
  xp.x = *reinterpret_cast<unsigned*>(&x01);
  xp.y = *reinterpret_cast<unsigned*>(&x23);
  *reinterpret_cast<uint2*>(xo + (size_t)r * d + c) = xp;
}

// RMSNorm of bf16 models from the row sums of squares the producing GEMM
// left per 64-column block (ss[p][r], p < d/64):
//   x[r] = bf16(h[r] / sqrt(sum_p ss[p][r] / d + eps) * g).
// Block = one row, d/4 threads (4 columns each).
// The kernel lets its dependent start before waiting on its own predecessor:
// what follows a norm (a projection, a row copy) does nothing but request
// weights before its own wait, which ends only after this kernel - and so the
// projection before it - has completed.  A projection after a norm thereby
// streams its first weights while the projection before the norm drains and
// the norm runs (its CTAs take the SMs the earlier projection frees).
__global__ void norm_rows_kernel(const float* __restrict__ h, const float* __restrict__ ss, const float* __restrict__ g,
                                 bf16* __restrict__ xo, int rows, int d, float eps) {
  if (threadIdx.x == 0) pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, c = threadIdx.x * 4;
  if (r >= rows) return;
  // every thread sums the row's partials itself (L1 hits after the first;
  // one thread summing them for the block behind a barrier was measured
  // slower: 1.25 -> 2.0 ms per launch at 262144 rows)
  float tot = 0.f;
  for (int p = 0; p < d / 64; ++p) tot += ss[(size_t)p * rows + r];
  const float rs = rsqrtf(tot / (float)d + eps);
  const float4 v = *reinterpret_cast<const float4*>(h + (size_t)r * d + c);
  const float4 gg = *reinterpret_cast<const float4*>(g + c);
  __nv_bfloat162 x01 = __floats2bfloat162_rn(v.x * rs * gg.x, v.y * rs * gg.y);
  __nv_bfloat162 x23 = __floats2bfloat162_rn(v.z * rs * gg.z, v.w * rs * gg.w);
  uint2 xp;
  xp.x = *reinterpret_cast<unsigned*>(&x01);
  xp.y = *reinterpret_cast<unsigned*>(&x23);
  *reinterpret_cast<uint2*>(xo + (size_t)r * d + c) = xp;
}

// o = bf16(s), element-wise.
__global__ void to_bf16_kernel(const float* __restrict__ s, bf16* __restrict__ o, size_t n) {
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) o[i] = __float2bfloat16_rn(s[i]);
}

// ---------------------------------------------------------------------------
// RMSNorm, one warp per row: y = x / sqrt(mean(x^2) + eps) * g.
template <typename T_>
__global__ void rmsnorm_kernel(const float* __restrict__ x, const float* __restrict__ g, T_* __restrict__ y,
                               int rows, int d, int ldy, float eps) {
  int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const float* xr = x + (size_t)warp * d;
  float ss = 0.f;
  for (int j = lane; j < d; j += 32) ss = fmaf(xr[j], xr[j], ss);
  ss = warp_sum(ss);
  float inv = rsqrtf(ss / (float)d + eps);
  T_* yr = y + (size_t)warp * ldy;
  for (int j = lane; j < d; j += 32) yr[j] = from_f32<T_>(xr[j] * inv * g[j]);
}

// ---------------------------------------------------------------------------
// Encoder: split the fused QKV projection into per-head q, k, v [B][H][T][hd],
// applying RoPE at position t to q and k.  One thread per (row, head, pair i).
template <typename T_>
__global__ void rope_split_kernel(const float* __restrict__ qkv, T_* __restrict__ q, T_* __restrict__ k,
                                  T_* __restrict__ v, const float2* __restrict__ tab, int B, int T, int H, int hd) {
  const int half = hd / 2;
  size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  size_t total = (size_t)B * T * H * half;
  if (idx >= total) return;
  int i = idx % half;
  size_t r2 = idx / half;
  int h = r2 % H;
  size_t row = r2 / H;  // b*T + t
  int t = row % T, b = row / T;
  const int d = H * hd;
  const float* src = qkv + row * 3 * d + h * hd;
  float2 cs = tab[(size_t)t * half + i];
  size_t o = (((size_t)b * H + h) * T + t) * hd;
  float q1 = src[i], q2 = src[i + half];
  q[o + i] = from_f32<T_>(q1 * cs.x - q2 * cs.y);
  q[o + i + half] = from_f32<T_>(q2 * cs.x + q1 * cs.y);
  float k1 = src[d + i], k2 = src[d + i + half];
  k[o + i] = from_f32<T_>(k1 * cs.x - k2 * cs.y);
  k[o + i + half] = from_f32<T_>(k2 * cs.x + k1 * cs.y);
  v[o + i] = from_f32<T_>(src[2 * d + i]);
  v[o + i + half] = from_f32<T_>(src[2 * d + i + half]);
}

// ---------------------------------------------------------------------------
// Encoder causal attention (CUDA cores).  Block = 32 queries of one (b, h);
// 8 warps x 4 queries; keys staged 32 at a time in shared memory; online
// softmax.  For bf16 models the weights exp(s - m) are rounded to bf16 before
// the product with V (the tensor-core kernels feed P to the MMA in bf16), the
// row sum uses the unrounded weights.  Output o[b][t][h*hd + i].
template <typename T_>
__global__ void __launch_bounds__(256) enc_attn_simt_kernel(const T_* __restrict__ q, const T_* __restrict__ k,
                                                            const T_* __restrict__ v, T_* __restrict__ o, int T,
                                                            int H, int hd, float scale) {
  extern __shared__ float sm[];
  float* sQ = sm;                    // [32][hd]
  float* sK = sQ + 32 * hd;          // [32][hd+1]
  float* sV = sK + 32 * (hd + 1);    // [32][hd]
  const int b = blockIdx.z, h = blockIdx.y, q0 = blockIdx.x * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t base = (((size_t)b * H + h) * T) * hd;
  for (int i = tid; i < 32 * hd; i += 256) {
    int r = i / hd, c = i % hd;
    sQ[i] = (q0 + r < T) ? to_f32(q[base + (size_t)(q0 + r) * hd + c]) : 0.f;
  }
  float m_i[4], l_i[4], acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    m_i[a] = -INFINITY;
    l_i[a] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
  }
  const int q_last = min(q0 + 31, T - 1);
  for (int k0 = 0; k0 <= q_last; k0 += 32) {
    __syncthreads();
    for (int i = tid; i < 32 * hd; i += 256) {
      int r = i / hd, c = i % hd;
      bool ok = k0 + r < T;
      sK[r * (hd + 1) + c] = ok ? to_f32(k[base + (size_t)(k0 + r) * hd + c]) : 0.f;
      sV[r * hd + c] = ok ? to_f32(v[base + (size_t)(k0 + r) * hd + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int qi = warp * 4 + a, qpos = q0 + qi;
      if (qpos >= T) continue;
      const int kpos = k0 + lane;
      float s = 0.f;
      for (int c = 0; c < hd; ++c) s = fmaf(sQ[qi * hd + c], sK[lane * (hd + 1) + c], s);
      s = (kpos <= qpos) ? s * scale : -INFINITY;
      float mnew = fmaxf(m_i[a], warp_max(s));
      float p = (kpos <= qpos) ? expf(s - mnew) : 0.f;
      float corr = expf(m_i[a] - mnew);
      l_i[a] = l_i[a] * corr + warp_sum(p);
      m_i[a] = mnew;
      float pr = round_st<T_>(p);
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][c] *= corr;
      for (int j = 0; j < 32; ++j) {
        float pj = __shfl_sync(0xffffffffu, pr, j);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          int dim = lane + 32 * c;
          if (dim < hd) acc[a][c] = fmaf(pj, sV[j * hd + dim], acc[a][c]);
        }
      }
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int qpos = q0 + warp * 4 + a;
    if (qpos >= T) continue;
    const float inv = 1.f / l_i[a];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      int dim = lane + 32 * c;
      if (dim < hd) o[((size_t)b * T + qpos) * (H * hd) + h * hd + dim] = from_f32<T_>(acc[a][c] * inv);
    }
  }
}

// ---------------------------------------------------------------------------
// SwiGLU product m = silu(g1) * g3 from the fused [W_1; W_3] projection.
template <typename T_>
__global__ void swiglu_kernel(const float* __restrict__ g, T_* __restrict__ m, int rows, int f) {
  size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (size_t)rows * f) return;
  size_t r = idx / f;
  int j = idx % f;
  const float* gr = g + r * 2 * f;
  m[idx] = from_f32<T_>(silu_f(gr[j]) * gr[f + j]);
}

// ---------------------------------------------------------------------------
// Decoder merge.  Gate input x = [e_t; s_{t-1}] in storage precision, then
// (after the gate GEMM) h = z * s + (1 - z) * e with z = sigmoid(zpre + b_g).
template <typename T_>
__global__ void merge_prep_kernel(const T_* __restrict__ e, const float* __restrict__ s, T_* __restrict__ x,
                                  int B, int T_mem, int d, const StepCtx* ctx) {
  const int p = ctx->pos;
  int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= B * d) return;
  int b = idx / d, j = idx % d;
  x[(size_t)b * 2 * d + j] = e[((size_t)b * T_mem + p) * d + j];
  x[(size_t)b * 2 * d + d + j] = from_f32<T_>(s[idx]);
}
template <typename T_>
__global__ void merge_blend_kernel(const float* __restrict__ zpre, const float* __restrict__ bg,
                                   const T_* __restrict__ e, const float* __restrict__ s, float* __restrict__ h,
                                   int B, int T_mem, int d, int discard, const StepCtx* ctx) {
  const int p = ctx->pos;
  int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= B * d) return;
  int b = idx / d, j = idx % d;
  float ev = to_f32(e[((size_t)b * T_mem + p) * d + j]);
  if (discard) {
    h[idx] = ev;
    return;
  }
  float z = sigmoid_f(zpre[idx] + bg[j]);
  h[idx] = z * s[idx] + (1.f - z) * ev;
}

// ---------------------------------------------------------------------------
// Decoder sliding-window self-attention of one layer.  Block = one (b, h).
// RoPE on q and k at position p, k and v rounded to storage and written to
// ring slot p mod W, then attention over the min(W, p+1) entries of
// positions p-n+1..p (the window includes the current token).
// qkv: fp32 [B][3d]; ring: [B][H][W][hd] (this layer); out: [B][d].
template <typename T_>
__global__ void __launch_bounds__(128) dec_swa_kernel(const float* __restrict__ qkv, T_* __restrict__ ring_k,
                                                      T_* __restrict__ ring_v, T_* __restrict__ out,
                                                      const float2* __restrict__ tab, int H, int hd, int W,
                                                      float scale, const StepCtx* ctx) {
  extern __shared__ float sm[];
  float* sq = sm;             // [hd]
  float* sp = sq + hd;        // [W]
  __shared__ float red[32];
  const int b = blockIdx.y, h = blockIdx.x, tid = threadIdx.x;
  const int p = ctx->pos, half = hd / 2, d = H * hd;
  const float* src = qkv + (size_t)b * 3 * d + h * hd;
  const size_t rbase = (((size_t)b * H + h) * W) * hd;
  const int slot = p % W;
  for (int i = tid; i < half; i += blockDim.x) {
    float2 cs = tab[(size_t)p * half + i];
    float q1 = src[i], q2 = src[i + half];
    sq[i] = q1 * cs.x - q2 * cs.y;
    sq[i + half] = q2 * cs.x + q1 * cs.y;
    float k1 = src[d + i], k2 = src[d + i + half];
    ring_k[rbase + (size_t)slot * hd + i] = from_f32<T_>(k1 * cs.x - k2 * cs.y);
    ring_k[rbase + (size_t)slot * hd + i + half] = from_f32<T_>(k2 * cs.x + k1 * cs.y);
    ring_v[rbase + (size_t)slot * hd + i] = from_f32<T_>(src[2 * d + i]);
    ring_v[rbase + (size_t)slot * hd + i + half] = from_f32<T_>(src[2 * d + i + half]);
  }
  __syncthreads();
  const int n = min(W, p + 1);
  // scores of entries j = 0..n-1 <-> position p - n + 1 + j
  float lmax = -INFINITY;
  for (int j = tid; j < n; j += blockDim.x) {
    int sl = (p - n + 1 + j) % W;
    const T_* kr = ring_k + rbase + (size_t)sl * hd;
    float s = 0.f;
    for (int c = 0; c < hd; ++c) s = fmaf(sq[c], to_f32(kr[c]), s);
    s *= scale;
    sp[j] = s;
    lmax = fmaxf(lmax, s);
  }
  lmax = warp_max(lmax);
  if ((tid & 31) == 0) red[tid >> 5] = lmax;
  __syncthreads();
  float m = -INFINITY;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  float lsum = 0.f;
  for (int j = tid; j < n; j += blockDim.x) {
    float e = expf(sp[j] - m);
    sp[j] = e;
    lsum += e;
  }
  lsum = warp_sum(lsum);
  if ((tid & 31) == 0) red[tid >> 5] = lsum;
  __syncthreads();
  float l = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) l += red[w];
  const float inv = 1.f / l;
  for (int c = tid; c < hd; c += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < n; ++j) {
      int sl = (p - n + 1 + j) % W;
      acc = fmaf(sp[j], to_f32(ring_v[rbase + (size_t)sl * hd + c]), acc);
    }
    out[(size_t)b * d + h * hd + c] = from_f32<T_>(acc * inv);
  }
}

// ---------------------------------------------------------------------------
// End of the decoder layers: s_t = h; a = RMSNorm_o(h) for the head GEMM.
template <typename T_>
__global__ void head_prep_kernel(const float* __restrict__ h, float* __restrict__ s, const float* __restrict__ g,
                                 T_* __restrict__ a, int B, int d, float eps) {
  int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= B) return;
  const float* hr = h + (size_t)warp * d;
  float ss = 0.f;
  for (int j = lane; j < d; j += 32) {
    float x = hr[j];
    s[(size_t)warp * d + j] = x;
    ss = fmaf(x, x, ss);
  }
  ss = warp_sum(ss);
  float inv = rsqrtf(ss / (float)d + eps);
  for (int j = lane; j < d; j += 32) a[(size_t)warp * d + j] = from_f32<T_>(hr[j] * inv * g[j]);
}

// ---------------------------------------------------------------------------
// Head reduction of one row (block per sequence): tempered log-softmax of the
// action, its top-k renormalised value (exact k-th largest by radix select
// over order-preserving keys, ties to the lower id), argmax (lowest id on
// ties), the optional logits copy, and in generation the draw
// (sampling.cuh).
struct HeadArgs {
  const float* logits;     // [B][V] fp32 (this step)
  const int* actions;      // [B][n] or null
  float* logp;             // [B][n] or null
  float* logp_full;        // [B][n] or null
  int* argmax;             // [B][n] or null
  const int* emit_map;     // [n]: index into logits_out or -1
  float* logits_out;       // [n_emit][B][V] or null
  int B, V, n, top_k;
  float inv_temp;
  int* status;
  // sampling (generation): with next_tok set, the action is drawn from the
  // tempered (top-k) distribution instead of read from actions, with the
  // uniform draw of position ctx->pos + sample_off (the drawn token's
  // position); it goes to next_tok[b] and, when step + sample_off < n, to
  // sample_tok[b][step + sample_off] with its log-probabilities at the same
  // index
  int* next_tok;           // [B] or null
  int* sample_tok;         // [B][n] or null
  int sample_off;
  unsigned long long seed;
};


__global__ void __launch_bounds__(1024) head_reduce_kernel(HeadArgs a, const StepCtx* ctx) {
  pdl_wait();
  if (threadIdx.x == 0) pdl_trigger();
  extern __shared__ float sx[];  // [V] tempered logits
  __shared__ unsigned hist[256];
  __shared__ float fred[32];
  __shared__ int ired[32];
  __shared__ unsigned s_prefix, s_remain, s_cnt;
  __shared__ float s_part[1024];   // sampling: per-thread sums of its id chunk
  __shared__ unsigned s_tie[1024];  // sampling: per-thread count of ties at the k-th key
  __shared__ int s_res[5];
  const int b = blockIdx.x, tid = threadIdx.x, nthr = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
  const int i = ctx->step;
  const float* lg = a.logits + (size_t)b * a.V;
  const int em = (a.emit_map && a.logits_out) ? a.emit_map[i] : -1;
  float bmax = -INFINITY;
  int barg = 0x7fffffff;
  for (int v = tid; v < a.V; v += nthr) {
    float x = lg[v];
    if (em >= 0) a.logits_out[((size_t)em * a.B + b) * a.V + v] = x;
    if (x > bmax || (x == bmax && v < barg)) { bmax = x; barg = v; }
    sx[v] = x * a.inv_temp;
  }
  // argmax with lowest id on ties
  for (int o = 16; o > 0; o >>= 1) {
    float om = __shfl_xor_sync(0xffffffffu, bmax, o);
    int oa = __shfl_xor_sync(0xffffffffu, barg, o);
    if (om > bmax || (om == bmax && oa < barg)) { bmax = om; barg = oa; }
  }
  if (lane == 0) { fred[warp] = bmax; ired[warp] = barg; }
  __syncthreads();
  if (tid == 0) {
    float mm = fred[0];
    int aa = ired[0];
    for (int w = 1; w < nw; ++w)
      if (fred[w] > mm || (fred[w] == mm && ired[w] < aa)) { mm = fred[w]; aa = ired[w]; }
    fred[0] = mm;
    ired[0] = aa;
  }
  __syncthreads();
  const int amax = ired[0];
  const float mx = fred[0] * a.inv_temp;   // max of tempered logits (inv_temp > 0)
  __syncthreads();
  float se = 0.f;
  for (int v = tid; v < a.V; v += nthr) se += expf(sx[v] - mx);
  se = warp_sum(se);
  if (lane == 0) fred[warp] = se;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < nw; ++w) t += fred[w];
    fred[0] = t;
  }
  __syncthreads();
  const float lse = mx + logf(fred[0]);
  __syncthreads();
  const bool sampling = a.next_tok != nullptr;
  int act = (!sampling && a.actions) ? a.actions[(size_t)b * a.n + i] : -1;
  if (act >= a.V) {
    if (tid == 0) set_error(a.status, kErrBounds);
    act = -1;
  }
  const bool topk = a.top_k > 0 && a.top_k < a.V;
  if (sampling && !topk) {
    act = sample_chunked(sx, a.V, mx, true, 0u, 0u, uniform24(a.seed, b, ctx->pos + a.sample_off), s_part, s_tie,
                         s_res);
  }
  float lp_full = (act >= 0) ? sx[act] - lse : NAN;
  float lp = lp_full;
  if (topk) {
    // radix select of the k-th largest key, 8 bits at a time from the top
    if (tid == 0) { s_prefix = 0; s_remain = (unsigned)a.top_k; }
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int j = tid; j < 256; j += nthr) hist[j] = 0;
      __syncthreads();
      const unsigned pref = s_prefix;
      const unsigned hmask = (pass == 0) ? 0u : (0xffffffffu << (shift + 8));
      // the keys of a row are mostly alike in their high bytes, so the lanes
      // of a warp that fall into the same bin are counted with one add (the
      // same-address adds would otherwise serialise); every warp runs the
      // same number of iterations so that all its lanes take part
      for (int v0 = 0; v0 < a.V; v0 += nthr) {
        const int v = v0 + tid;
        int bin = -1;
        if (v < a.V) {
          const unsigned kk = f2key(sx[v]);
          if ((kk & hmask) == pref) bin = (int)((kk >> shift) & 255u);
        }
        const unsigned grp = __match_any_sync(0xffffffffu, bin);
        if (bin >= 0 && lane == __ffs(grp) - 1) atomicAdd(&hist[bin], (unsigned)__popc(grp));
      }
      __syncthreads();
      if (tid == 0) {
        unsigned rem = s_remain;
        int bin = 255;
        for (; bin > 0; --bin) {
          if (hist[bin] >= rem) break;
          rem -= hist[bin];
        }
        s_prefix = pref | ((unsigned)bin << shift);
        s_remain = rem;  // how many to take from keys equal to the final prefix
      }
      __syncthreads();
    }
    const unsigned kth = s_prefix;          // exact key of the k-th largest value
    const unsigned need = s_remain;         // ties at kth taken, lowest ids first
    const float xk = sx[0] * 0.f + __uint_as_float((kth & 0x80000000u) ? (kth & 0x7fffffffu) : ~kth);
    if (sampling) {
      act = sample_chunked(sx, a.V, mx, false, kth, need, uniform24(a.seed, b, ctx->pos + a.sample_off), s_part,
                           s_tie, s_res);
      lp_full = sx[act] - lse;
    }
    float sg = 0.f;
    for (int v = tid; v < a.V; v += nthr) {
      unsigned kk = f2key(sx[v]);
      if (kk > kth) sg += expf(sx[v] - mx);
    }
    sg = warp_sum(sg);
    __syncthreads();
    if (lane == 0) fred[warp] = sg;
    // rank of the action among ties (ids below it with the same key)
    unsigned below = 0;
    if (act >= 0 && f2key(sx[act]) == kth)
      for (int v = tid; v < act; v += nthr) below += (f2key(sx[v]) == kth) ? 1u : 0u;
    if (tid == 0) s_cnt = 0;
    __syncthreads();
    if (below) atomicAdd(&s_cnt, below);
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      for (int w = 0; w < nw; ++w) t += fred[w];
      fred[0] = t;
    }
    __syncthreads();
    const float lse_k = mx + logf(fred[0] + (float)need * expf(xk - mx));
    if (act >= 0) {
      unsigned ka = f2key(sx[act]);
      bool in = (ka > kth) || (ka == kth && s_cnt < need);
      lp = in ? sx[act] - lse_k : -INFINITY;
    }
  }
  if (tid == 0) {
    if (sampling) {
      a.next_tok[b] = act;
      const int j = i + a.sample_off;
      if (j < a.n) {
        const size_t o = (size_t)b * a.n + j;
        if (a.sample_tok) a.sample_tok[o] = act;
        if (a.logp) a.logp[o] = lp;
        if (a.logp_full) a.logp_full[o] = lp_full;
        if (a.argmax) a.argmax[o] = amax;
      }
    } else {
      const size_t o = (size_t)b * a.n + i;
      if (a.logp) a.logp[o] = lp;
      if (a.logp_full) a.logp_full[o] = lp_full;
      if (a.argmax) a.argmax[o] = amax;
    }
  }
}

// Per-row sums of squares of h [rows][d] in 64-column groups, ss[g][r], with
// the same lane mapping and half-warp reduction as the residual epilogue of
// the projections (so that an RMSNorm from them is bitwise the in-step one).
// One warp per (row, pair of groups); blockDim 128.
__global__ void row_ss_kernel(const float* __restrict__ h, float* __restrict__ ss, int rows, int d) {
  const int lane = threadIdx.x & 31;
  const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int pairs = d / 128;
  if (wid >= rows * pairs) return;  // warp-uniform
  const int r = wid / pairs, g2 = wid - r * pairs;
  const float4 v = *reinterpret_cast<const float4*>(h + (size_t)r * d + g2 * 128 + lane * 4);
  const float q2 = half_warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
  if ((lane & 15) == 0) ss[(size_t)(2 * g2 + (lane >> 4)) * rows + r] = q2;
}

// e[b][pos][:] = x[b][:] (bf16 rows, pos = ctx->pos), pos < T.
__global__ void put_row_kernel(const bf16* __restrict__ x, bf16* __restrict__ e, int B, int d, int T,
                               const StepCtx* ctx) {
  pdl_wait();
  if (threadIdx.x == 0) pdl_trigger();
  const int b = blockIdx.x;
  const int p = ctx->pos;
  if (b >= B || p >= T) return;
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8)
    *reinterpret_cast<uint4*>(e + ((size_t)b * T + p) * d + c) = *reinterpret_cast<const uint4*>(x + (size_t)b * d + c);
}

__global__ void advance_kernel(StepCtx* ctx) {
  pdl_wait();
  pdl_trigger();
  ctx->pos += 1;
  ctx->step += 1;
}
__global__ void set_ctx_kernel(StepCtx* ctx, int pos) {
  ctx->pos = pos;
  ctx->step = 0;
}

template <typename T_>
__global__ void fill_nan_kernel(T_* p, size_t n) {
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; i < n; i += stride) p[i] = nan_of<T_>();
}
__global__ void bcast_rows_kernel(float* dst, const float* src, int rows, int d) {
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < (size_t)rows * d) dst[i] = src[i % d];
}

}  // namespace rlt
