// Device kernels of the decoder's backpropagation through time (the
// operations that bptt_plan.h sequences).  Storage type T (fp32 or bf16) for
// GEMM operands and recorded keys/values; every gradient and reduction in
// fp32.  Row-major [B][N] operands come with a transposed copy, written to
// rows of length ldT (one step's column slot of a block operand: the
// row-contracted operand of the weight-gradient GEMMs).
//
// Attention backward (per sequence b, head h, over positions j0..j1): with
// s_j = scale q.K_j, P_j = exp(s_j - lse), o = sum_j P_j V_j and the output
// gradient g,
//   dP_j = g.V_j,  D = g.o,  dS_j = P_j (dP_j - D),
//   dq = scale sum_j dS_j K_j,  dK_j = scale dS_j q,  dV_j = P_j g.
// The query gradient is taken per step; the key/value gradients are summed
// per key over the queries that read it (swa_bwd_kernel for the window,
// mem_grad_kernel for the memory).
//
// Step kernels read the step's position p from a device cell (*pos) rather
// than from their arguments, so that a step can be captured once and
// replayed; split grids are sized for the largest range and chunks past the
// current one write neutral partials.
#pragma once

#include "common.cuh"
#include "fused_ptx.cuh"

namespace rlt {
namespace bptt {

constexpr int kThreads = 256;

__device__ __forceinline__ float sigmoid_acc(float x) { return 1.0f / (1.0f + expf(-x)); }

// RoPE angle of pair i at position p: p * theta^(-2i/hd), in double.
__device__ __forceinline__ void rope_cs(int p, int i, int hd, float theta, float& c, float& s) {
  const double ang = (double)p * pow((double)theta, -2.0 * (double)i / (double)hd);
  double sd, cd;
  sincos(ang, &sd, &cd);
  c = (float)cd;
  s = (float)sd;
}

// Head rows held by a warp: lane l holds elements l + 32 c (c < 4) of a
// head of hd <= 128.  The RoPE partner of element i is i ^ (hd / 2): for
// hd >= 64 it is in the same lane, register c ^ (hd / 64); for hd <= 32 it is
// lane l ^ (hd / 2) (a full-warp shuffle; lanes past hd hold zeros).
__device__ __forceinline__ float rope_partner(const float (&v)[4], int c, int hd) {
  const int half = hd >> 1;
  if (half >= 32) {
    const int pc = c ^ (half >> 5);
    float r = v[0];
#pragma unroll
    for (int k = 1; k < 4; ++k) r = (k == pc) ? v[k] : r;
    return r;
  }
  return __shfl_xor_sync(0xffffffffu, v[c], half);
}

// dst[c][r] = src[r][c] through a 32x33 shared tile; block (32, 8).
template <typename T>
__global__ void transpose_kernel(const T* __restrict__ src, int rows, int cols, int lds, T* __restrict__ dst,
                                 int ldd) {
  __shared__ T tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int j = threadIdx.y; j < 32; j += 8) {
    const int r = r0 + j, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[j][threadIdx.x] = src[(size_t)r * lds + c];
  }
  __syncthreads();
  for (int j = threadIdx.y; j < 32; j += 8) {
    const int c = c0 + j, r = r0 + threadIdx.x;
    if (r < rows && c < cols) dst[(size_t)c * ldd + r] = tile[threadIdx.x][j];
  }
}

// xg[b] = [e[b][p]; s_p[b]] in the storage type (and transposed).
template <typename T>
__global__ void merge_in_kernel(const T* __restrict__ e, int T_mem, const int* __restrict__ pos,
                                const float* __restrict__ s_all, int B, int d, T* __restrict__ xg,
                                T* __restrict__ xgT, int ldT) {
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (size_t)B * 2 * d) return;
  const int p = *pos;
  const float* s = s_all + (size_t)p * B * d;
  const int b = (int)(idx / (2 * d)), i = (int)(idx - (size_t)b * 2 * d);
  const T v = (i < d) ? e[((size_t)b * T_mem + p) * d + i] : from_f32<T>(s[(size_t)b * d + i - d]);
  xg[idx] = v;
  if (xgT) xgT[(size_t)i * ldT + b] = v;
}

// z = sigmoid(zpre + b_g) (0 without a gate), h = z s + (1 - z) e[b][p].
template <typename T>
__global__ void merge_out_kernel(const float* __restrict__ zpre, const float* __restrict__ bg,
                                 const T* __restrict__ e, int T_mem, const int* __restrict__ pos,
                                 const float* __restrict__ s_all, int B, int d, float* __restrict__ z,
                                 float* __restrict__ h) {
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (size_t)B * d) return;
  const int p = *pos;
  const float* s = s_all + (size_t)p * B * d;
  const int b = (int)(idx / d), i = (int)(idx - (size_t)b * d);
  const float zv = zpre ? sigmoid_acc(zpre[idx] + bg[i]) : 0.f;
  const float ev = to_f32(e[((size_t)b * T_mem + p) * d + i]);
  z[idx] = zv;
  h[idx] = zv * s[idx] + (1.f - zv) * ev;
}

// RMSNorm rows: r = 1 / sqrt(mean(x^2) + eps), y = x r g (storage type, and
// transposed when yT is given); x is [B][d], or with pos the rows of position
// *pos + off of [.][B][d].  One warp per row.
template <typename T>
__global__ void rms_fwd_kernel(const float* __restrict__ x, const int* __restrict__ pos, int off,
                               const float* __restrict__ g, int B, int d, float eps, float* __restrict__ r,
                               T* __restrict__ y, T* __restrict__ yT, int ldT) {
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (row >= B) return;
  if (pos) x += (size_t)(*pos + off) * B * d;
  const float* xr = x + (size_t)row * d;
  float ss = 0.f;
  for (int i = lane; i < d; i += 32) ss = fmaf(xr[i], xr[i], ss);
  ss = warp_sum(ss);
  const float rv = 1.0f / sqrtf(ss / (float)d + eps);
  if (lane == 0) r[row] = rv;
  for (int i = lane; i < d; i += 32) {
    const T v = from_f32<T>(xr[i] * rv * g[i]);
    y[(size_t)row * d + i] = v;
    if (yT) yT[(size_t)i * ldT + row] = v;
  }
}

// Memory attention of position p = *pos, one warp per (b, h): q [B][d] over
// positions 0..p of K, V [B][H][Tk][hd]; the output in the storage type to
// o_step [B][d] and to row p of the record o_rec (+ p * o_stride), the LSE to
// lse_rec + p * lse_stride.  Lane l holds elements l, l + 32, ... of the head.
template <typename T>
__global__ void attn_fwd_kernel(const float* __restrict__ q, const T* __restrict__ K, const T* __restrict__ V, int Tk,
                                const int* __restrict__ pos, int B, int H, int hd, float scale,
                                float* __restrict__ lse_rec, size_t lse_stride, T* __restrict__ o_step,
                                T* __restrict__ o_rec, size_t o_stride) {
  const int pair = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (pair >= B * H) return;
  const int p = *pos;
  const int b = pair / H, h = pair - b * H;
  const int d = H * hd;
  const int NC = (hd + 31) >> 5;  // <= 4
  float qr[4], acc[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    qr[c] = (c < NC && i < hd) ? q[(size_t)b * d + h * hd + i] : 0.f;
    acc[c] = 0.f;
  }
  const T* Kb = K + ((size_t)b * H + h) * Tk * hd;
  const T* Vb = V + ((size_t)b * H + h) * Tk * hd;
  float mx = -INFINITY, l = 0.f;
  for (int j = 0; j <= p; ++j) {
    float part = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      if (c < NC && i < hd) part = fmaf(qr[c], to_f32(Kb[(size_t)j * hd + i]), part);
    }
    const float sj = warp_sum(part) * scale;
    const float mn = fmaxf(mx, sj);
    const float corr = expf(mx - mn), w = expf(sj - mn);
    l = l * corr + w;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      if (c < NC && i < hd) acc[c] = acc[c] * corr + w * to_f32(Vb[(size_t)j * hd + i]);
    }
    mx = mn;
  }
  if (lane == 0) lse_rec[(size_t)p * lse_stride + pair] = mx + logf(l);
  const float inv = 1.0f / l;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    if (c < NC && i < hd) {
      const size_t col = (size_t)h * hd + i;
      const T vq = from_f32<T>(acc[c] * inv);
      o_step[(size_t)b * d + col] = vq;
      o_rec[(size_t)p * o_stride + (size_t)b * d + col] = vq;
    }
  }
}

// Window attention forward of position p = *pos, one warp per (b, h): q and
// k of qkv [B][3d] rotated by RoPE at p (q fp32 to its record slot p mod W of
// qR [W][B][d]; k and v rounded to the storage type and written to K, V
// [B][H][Tk][hd] at p), then the attention of q over positions
// max(0, p - W + 1)..p (position p from registers, the same rounded values):
// the LSE to its record slot of lR [W][B][H], the output to oq [B][d]
// (storage type) and its transposed slot oT.
template <typename T>
__global__ void swa_fwd_kernel(const float* __restrict__ qkv, const int* __restrict__ pos, int W, int B, int H,
                               int hd, float theta, float scale, float* __restrict__ qR, float* __restrict__ lR,
                               T* __restrict__ K, T* __restrict__ V, int Tk, T* __restrict__ oq, T* __restrict__ oT,
                               int ldT) {
  const int pair = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (pair >= B * H) return;
  const int p = *pos, j0 = p - W + 1 > 0 ? p - W + 1 : 0;
  float* qo = qR + (size_t)(p % W) * B * H * hd;
  float* lse = lR + (size_t)(p % W) * B * H;
  const int b = pair / H, h = pair - b * H;
  const int d = H * hd, half = hd >> 1;
  const int NC = (hd + 31) >> 5;
  const float* row = qkv + (size_t)b * 3 * d + h * hd;
  float qv[4], kv[4], vv[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    const bool ok = c < NC && i < hd;
    qv[c] = ok ? row[i] : 0.f;
    kv[c] = ok ? row[d + i] : 0.f;
    vv[c] = ok ? row[2 * d + i] : 0.f;
  }
  float qr[4], kr[4], acc[4];
  const size_t kp = (((size_t)b * H + h) * Tk + p) * hd;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    const float qp = rope_partner(qv, c, hd), kpv = rope_partner(kv, c, hd);
    float cs = 1.f, sn = 0.f;
    if (c < NC && i < hd) rope_cs(p, i % half, hd, theta, cs, sn);
    // (x1, x2) -> (x1 c - x2 s, x2 c + x1 s): element i < half is x1
    const float sg = (i % hd) < half ? -1.f : 1.f;
    qr[c] = qv[c] * cs + sg * qp * sn;
    kr[c] = round_st<T>(kv[c] * cs + sg * kpv * sn);
    vv[c] = round_st<T>(vv[c]);
    acc[c] = 0.f;
    if (c < NC && i < hd) {
      qo[(size_t)b * d + h * hd + i] = qr[c];
      K[kp + i] = from_f32<T>(kr[c]);
      V[kp + i] = from_f32<T>(vv[c]);
    }
  }
  const T* Kb = K + ((size_t)b * H + h) * Tk * hd;
  const T* Vb = V + ((size_t)b * H + h) * Tk * hd;
  float mx = -INFINITY, l = 0.f;
  for (int j = j0; j <= p; ++j) {
    float part = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      if (c < NC && i < hd) part = fmaf(qr[c], j == p ? kr[c] : to_f32(Kb[(size_t)j * hd + i]), part);
    }
    const float sj = warp_sum(part) * scale;
    const float mn = fmaxf(mx, sj);
    const float corr = expf(mx - mn), w = expf(sj - mn);
    l = l * corr + w;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      if (c < NC && i < hd) acc[c] = acc[c] * corr + w * (j == p ? vv[c] : to_f32(Vb[(size_t)j * hd + i]));
    }
    mx = mn;
  }
  if (lane == 0) lse[pair] = mx + logf(l);
  const float inv = 1.0f / l;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    if (c < NC && i < hd) {
      const size_t col = (size_t)h * hd + i;
      const T vq = from_f32<T>(acc[c] * inv);
      oq[(size_t)b * d + col] = vq;
      if (oT) oT[col * ldT + b] = vq;
    }
  }
}

// Memory attention split over the keys: warp w = pair * nsplit + s takes
// keys [j0 + s C, min(j1, j0 + (s + 1) C - 1)] (C = kAttnChunk), so that long
// memories fill the GPU instead of one warp per (b, h) walking every key.
// Partials part[(pair * nsplit + s) * (hd + 2) + ...]: the forward writes
// acc[hd], the chunk's max and sum of exponentials; the backward writes the
// unscaled query-gradient partial sum_j dS_j K_j and D.  The combines read the
// splits in order (deterministic).
#ifndef RLT_BPTT_ATTN_CHUNK
#define RLT_BPTT_ATTN_CHUNK 64  // a compile-time parameter (the CPU tests build with small chunks)
#endif
constexpr int kAttnChunk = RLT_BPTT_ATTN_CHUNK;
template <typename T>
__global__ void attn_part_fwd_kernel(const float* __restrict__ q, const T* __restrict__ K, const T* __restrict__ V,
                                     int Tk, const int* __restrict__ pos, int B, int H, int hd, float scale,
                                     int nsplit, float* __restrict__ part) {
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wid >= B * H * nsplit) return;
  const int p = *pos;
  const int pair = wid / nsplit, sp = wid - pair * nsplit;
  const int b = pair / H, h = pair - b * H;
  const int d = H * hd;
  const int NC = (hd + 31) >> 5;
  const int ja = sp * kAttnChunk, jb = min(p, ja + kAttnChunk - 1);  // memory positions 0..p
  float qr[4], acc[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    qr[c] = (c < NC && i < hd) ? q[(size_t)b * d + h * hd + i] : 0.f;
    acc[c] = 0.f;
  }
  const T* Kb = K + ((size_t)b * H + h) * Tk * hd;
  const T* Vb = V + ((size_t)b * H + h) * Tk * hd;
  float mx = -INFINITY, l = 0.f;  // an empty chunk leaves the neutral partial
  for (int j = ja; j <= jb; ++j) {
    float part_s = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      if (c < NC && i < hd) part_s = fmaf(qr[c], to_f32(Kb[(size_t)j * hd + i]), part_s);
    }
    const float sj = warp_sum(part_s) * scale;
    const float mn = fmaxf(mx, sj);
    const float corr = expf(mx - mn), w = expf(sj - mn);
    l = l * corr + w;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      if (c < NC && i < hd) acc[c] = acc[c] * corr + w * to_f32(Vb[(size_t)j * hd + i]);
    }
    mx = mn;
  }
  float* pp = part + (size_t)wid * (hd + 2);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    if (c < NC && i < hd) pp[i] = acc[c];
  }
  if (lane == 0) {
    pp[hd] = mx;
    pp[hd + 1] = l;
  }
}

// Combine of the forward partials, one warp per (b, h), splits in order
// (neutral partials of empty chunks weigh nothing): the LSE to lse_rec + row *
// lse_stride with row = p mod ring (ring > 0) or p; the output in the storage
// type to oq [B][d], to oT when given, and to row p of o_rec (+ p * o_stride)
// when given.
template <typename T>
__global__ void attn_combine_fwd_kernel(const float* __restrict__ part, int nsplit, int B, int H, int hd,
                                        const int* __restrict__ pos, float* __restrict__ lse_rec, size_t lse_stride,
                                        int ring, T* __restrict__ oq, T* __restrict__ oT, int ldT,
                                        T* __restrict__ o_rec, size_t o_stride) {
  const int pair = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (pair >= B * H) return;
  const int p = *pos;
  const int b = pair / H, h = pair - b * H;
  const int d = H * hd;
  const int NC = (hd + 31) >> 5;
  const float* pp = part + (size_t)pair * nsplit * (hd + 2);
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, pp[(size_t)s * (hd + 2) + hd]);
  float Lsum = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < nsplit; ++s) {
    const float* ps = pp + (size_t)s * (hd + 2);
    const float w = expf(ps[hd] - M);
    Lsum = fmaf(ps[hd + 1], w, Lsum);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      if (c < NC && i < hd) acc[c] = fmaf(ps[i], w, acc[c]);
    }
  }
  const size_t row = ring > 0 ? (size_t)(p % ring) : (size_t)p;
  if (lane == 0) lse_rec[row * lse_stride + pair] = M + logf(Lsum);
  const float inv = 1.0f / Lsum;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    if (c < NC && i < hd) {
      const size_t col = (size_t)h * hd + i;
      const T vq = from_f32<T>(acc[c] * inv);
      oq[(size_t)b * d + col] = vq;
      if (oT) oT[col * ldT + b] = vq;
      if (o_rec) o_rec[(size_t)p * o_stride + (size_t)b * d + col] = vq;
    }
  }
}

// Window attention forward of position p = *pos split over the keys: warp
// (pair, s) applies RoPE to q (and the split holding position p also to k,
// writing k and v at p) and attends over its chunk of positions
// max(0, p - W + 1)..p (empty chunks leave neutral partials); split 0 writes
// the rotated q to its record slot of qR.  Partials as
// attn_part_fwd_kernel (attn_combine_fwd_kernel finishes, with ring W).
template <typename T>
__global__ void swa_part_fwd_kernel(const float* __restrict__ qkv, const int* __restrict__ pos, int W, int B, int H,
                                    int hd, float theta, float scale, int nsplit, float* __restrict__ qR,
                                    T* __restrict__ K, T* __restrict__ V, int Tk, float* __restrict__ part) {
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wid >= B * H * nsplit) return;
  const int p = *pos, j0 = p - W + 1 > 0 ? p - W + 1 : 0;
  float* qo = qR + (size_t)(p % W) * B * H * hd;
  const int pair = wid / nsplit, sp = wid - pair * nsplit;
  const int b = pair / H, h = pair - b * H;
  const int d = H * hd, half = hd >> 1;
  const int NC = (hd + 31) >> 5;
  const int ja = j0 + sp * kAttnChunk, jb = min(p, ja + kAttnChunk - 1);
  const bool has_p = jb == p;
  const float* row = qkv + (size_t)b * 3 * d + h * hd;
  float qv[4], kv[4], vv[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    const bool ok = c < NC && i < hd;
    qv[c] = ok ? row[i] : 0.f;
    kv[c] = ok ? row[d + i] : 0.f;
    vv[c] = ok ? row[2 * d + i] : 0.f;
  }
  float qr[4], kr[4], acc[4];
  const size_t kp = (((size_t)b * H + h) * Tk + p) * hd;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    const float qp = rope_partner(qv, c, hd), kpv = rope_partner(kv, c, hd);
    float cs = 1.f, sn = 0.f;
    if (c < NC && i < hd) rope_cs(p, i % half, hd, theta, cs, sn);
    const float sg = (i % hd) < half ? -1.f : 1.f;
    qr[c] = qv[c] * cs + sg * qp * sn;
    kr[c] = round_st<T>(kv[c] * cs + sg * kpv * sn);
    vv[c] = round_st<T>(vv[c]);
    acc[c] = 0.f;
    if (c < NC && i < hd) {
      if (sp == 0) qo[(size_t)b * d + h * hd + i] = qr[c];
      if (has_p) {
        K[kp + i] = from_f32<T>(kr[c]);
        V[kp + i] = from_f32<T>(vv[c]);
      }
    }
  }
  const T* Kb = K + ((size_t)b * H + h) * Tk * hd;
  const T* Vb = V + ((size_t)b * H + h) * Tk * hd;
  float mx = -INFINITY, l = 0.f;
  for (int j = ja; j <= jb; ++j) {
    float part_s = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      if (c < NC && i < hd) part_s = fmaf(qr[c], j == p ? kr[c] : to_f32(Kb[(size_t)j * hd + i]), part_s);
    }
    const float sj = warp_sum(part_s) * scale;
    const float mn = fmaxf(mx, sj);
    const float corr = expf(mx - mn), w = expf(sj - mn);
    l = l * corr + w;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      if (c < NC && i < hd) acc[c] = acc[c] * corr + w * (j == p ? vv[c] : to_f32(Vb[(size_t)j * hd + i]));
    }
    mx = mn;
  }
  float* pp = part + (size_t)wid * (hd + 2);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    if (c < NC && i < hd) pp[i] = acc[c];
  }
  if (lane == 0) {
    pp[hd] = mx;
    pp[hd + 1] = l;
  }
}

// Row p = *pos of a record x_l [n][L][B][N] (layer offset folded into x_l)
// to the fixed rows y [B][N] and the column slot yT.
template <typename T>
__global__ void tcopy_kernel(const T* __restrict__ x_l, int L, const int* __restrict__ pos, int B, int N,
                             T* __restrict__ y, T* __restrict__ yT, int ldT) {
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (size_t)B * N) return;
  const T* x = x_l + (size_t)(*pos) * L * B * N;
  const int b = (int)(idx / N), j = (int)(idx - (size_t)b * N);
  const T v = x[idx];
  y[idx] = v;
  yT[(size_t)j * ldT + b] = v;
}

// dst[(*pos + off) * count + i] = src[i].
__global__ void put_row_kernel(float* __restrict__ dst, const int* __restrict__ pos, int off,
                               const float* __restrict__ src, int count) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < count) dst[(size_t)(*pos + off) * count + i] = src[i];
}

// The position cell: *pos = v, *pos += dv.
__global__ void set_pos_kernel(int* pos, int v) { *pos = v; }
__global__ void add_pos_kernel(int* pos, int dv) { *pos += dv; }

// ds = 0 when s_p was detached after its step (p >= 1, p % s_every == 0).
__global__ void zero_if_detached_kernel(float* __restrict__ ds, const int* __restrict__ pos, int s_every, int count) {
  const int p = *pos;
  if (p < 1 || p % s_every != 0) return;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < count) ds[i] = 0.f;
}

// m = silu(g) u in the storage type (and transposed).
template <typename T>
__global__ void swiglu_fwd_kernel(const float* __restrict__ g, const float* __restrict__ u, int B, int f,
                                  T* __restrict__ m, T* __restrict__ mT, int ldT) {
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (size_t)B * f) return;
  const int b = (int)(idx / f), j = (int)(idx - (size_t)b * f);
  const float gv = g[idx];
  const T v = from_f32<T>(gv * sigmoid_acc(gv) * u[idx]);
  m[idx] = v;
  if (mT) mT[(size_t)j * ldT + b] = v;
}

// Order-preserving unsigned key of a float.
__device__ __forceinline__ unsigned fkey(float x) {
  const unsigned u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Head of one step, one block of kThreadsHead per sequence b: x = logits /
// temperature; S = all ids, or the top-k set (the k largest x, ties to the
// lower id); lp = x_a - log sum_{v in S} exp(x_v) to lp[b][p] (p = *pos)
// (NaN for a < 0, -inf for a outside S); d(-lp)/d logits_v =
// inv_temp (p_v [v in S] - [v = a]) to dl [B][V] (and transposed), 0 for
// a < 0.  Shared memory: V floats.
constexpr int kThreadsHead = 1024;
__global__ void __launch_bounds__(kThreadsHead) head_bwd_kernel(const float* __restrict__ logits, int B, int V,
                                                                 const int32_t* __restrict__ actions, int n,
                                                                 const int* __restrict__ pos, float inv_temp,
                                                                 int top_k, float* __restrict__ lp,
                                                                 void* dl_, void* dlT_, int ldT, int bf16_out,
                                                                 int* status) {
  extern __shared__ float sx[];
  __shared__ unsigned hist[256];
  __shared__ float red[32];
  __shared__ unsigned ured[kThreadsHead];
  __shared__ unsigned s_prefix, s_remain;
  const int b = blockIdx.x, tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int nw = nthr >> 5;
  const int p = *pos;
  const float* lg = logits + (size_t)b * V;
  float mx = -INFINITY;
  for (int v = tid; v < V; v += nthr) {
    const float x = lg[v] * inv_temp;
    sx[v] = x;
    mx = fmaxf(mx, x);
  }
  mx = warp_max(mx);
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  if (tid == 0) {
    float t = red[0];
    for (int w = 1; w < nw; ++w) t = fmaxf(t, red[w]);
    red[0] = t;
  }
  __syncthreads();
  mx = red[0];
  __syncthreads();
  const bool topk = top_k > 0 && top_k < V;
  unsigned kth = 0, need = 0;
  if (topk) {
    // radix select of the k-th largest key, 8 bits per pass from the top
    if (tid == 0) {
      s_prefix = 0;
      s_remain = (unsigned)top_k;
    }
    __syncthreads();
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int j = tid; j < 256; j += nthr) hist[j] = 0;
      __syncthreads();
      const unsigned pref = s_prefix;
      const unsigned hmask = (pass == 0) ? 0u : (0xffffffffu << (shift + 8));
      for (int v = tid; v < V; v += nthr) {
        const unsigned kk = fkey(sx[v]);
        if ((kk & hmask) == pref) atomicAdd(&hist[(kk >> shift) & 255u], 1u);
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
        s_remain = rem;
      }
      __syncthreads();
    }
    kth = s_prefix;
    need = s_remain;
  }
  // members: thread tid owns the contiguous ids [tid C, (tid + 1) C); the
  // ties at kth are ranked in id order through an exclusive scan of counts
  const int C = (V + nthr - 1) / nthr;
  const int v0 = min(V, tid * C), v1 = min(V, v0 + C);
  unsigned ties = 0;
  if (topk)
    for (int v = v0; v < v1; ++v) ties += (fkey(sx[v]) == kth) ? 1u : 0u;
  ured[tid] = ties;
  __syncthreads();
  if (tid == 0) {
    unsigned acc = 0;
    for (int t = 0; t < nthr; ++t) {
      const unsigned cnt = ured[t];
      ured[t] = acc;
      acc += cnt;
    }
  }
  __syncthreads();
  const unsigned tie0 = ured[tid];
  // mark non-members with -inf in place (ids of this thread's chunk only)
  {
    unsigned tb = tie0;
    for (int v = v0; v < v1; ++v) {
      bool in = true;
      if (topk) {
        const unsigned kk = fkey(sx[v]);
        in = kk > kth || (kk == kth && tb < need);
        if (kk == kth) ++tb;
      }
      if (!in) sx[v] = -INFINITY;
    }
  }
  __syncthreads();
  float se = 0.f;
  for (int v = tid; v < V; v += nthr) se += expf(sx[v] - mx);
  se = warp_sum(se);
  if (lane == 0) red[warp] = se;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < nw; ++w) t += red[w];
    red[0] = t;
  }
  __syncthreads();
  const float lse = mx + logf(red[0]);
  int act = actions[(size_t)b * n + p];
  if (act >= V) {
    if (tid == 0) set_error(status, kErrBounds);
    act = -1;
  }
  if (tid == 0) lp[(size_t)b * n + p] = act < 0 ? NAN : sx[act] - lse;
  const bool a_in = act >= 0 && sx[act] > -INFINITY;
  for (int v = tid; v < V; v += nthr) {
    float gv = 0.f;
    if (act >= 0) gv = inv_temp * (expf(sx[v] - lse) - ((v == act && a_in) ? 1.f : 0.f));
    if (bf16_out) {
      const bf16 q = __float2bfloat16_rn(gv);
      static_cast<bf16*>(dl_)[(size_t)b * V + v] = q;
      static_cast<bf16*>(dlT_)[(size_t)v * ldT + b] = q;
    } else {
      static_cast<float*>(dl_)[(size_t)b * V + v] = gv;
      static_cast<float*>(dlT_)[(size_t)v * ldT + b] = gv;
    }
  }
}

// RMSNorm backward for y = x r g (r = 1/sqrt(mean(x^2) + eps)) given dy:
//   dx_i += r g_i dy_i - x_i r^3 (sum_j g_j dy_j x_j) / d     (rows: warp per row)
//   dg_i += sum_b dy_i x_i r                                 (columns: thread per column)
// With out given, the updated dx rows are also written in the storage type
// to out [B][d] and transposed to outT (the next projection's operands).
// x is [B][d], or with pos the rows of position *pos + off of [.][B][d].
// Blocks [0, row_blocks) do the rows, the rest the columns.
template <typename T>
__global__ void rms_bwd_kernel(const float* __restrict__ x, const int* __restrict__ pos, int off,
                               const float* __restrict__ r, const float* __restrict__ g,
                               const float* __restrict__ dy, int B, int d, float* __restrict__ dx,
                               float* __restrict__ dg, int row_blocks, T* __restrict__ out, T* __restrict__ outT,
                               int ldT) {
  if (pos) x += (size_t)(*pos + off) * B * d;
  if ((int)blockIdx.x < row_blocks) {
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (row >= B) return;
    const float* xr = x + (size_t)row * d;
    const float* dyr = dy + (size_t)row * d;
    float sd = 0.f;
    for (int i = lane; i < d; i += 32) sd = fmaf(g[i] * dyr[i], xr[i], sd);
    sd = warp_sum(sd);
    const float rv = r[row];
    const float coef = rv * rv * rv * sd / (float)d;
    for (int i = lane; i < d; i += 32) {
      const float v = dx[(size_t)row * d + i] + (rv * g[i] * dyr[i] - xr[i] * coef);
      dx[(size_t)row * d + i] = v;
      if (out) {
        const T q = from_f32<T>(v);
        out[(size_t)row * d + i] = q;
        outT[(size_t)i * ldT + row] = q;
      }
    }
  } else {
    const int i = (blockIdx.x - row_blocks) * blockDim.x + threadIdx.x;
    if (i >= d) return;
    float acc = 0.f;
    for (int b = 0; b < B; ++b) acc = fmaf(dy[(size_t)b * d + i] * x[(size_t)b * d + i], r[b], acc);
    dg[i] += acc;
  }
}

// Residual update into a new buffer: C[m][n] = R[m][n] + acc (the GEMMs'
// per-element epilogue path).
struct EpiResidualInto {
  const float* R;
  float* C;
  int ldc;
  __device__ __forceinline__ void operator()(int m, int n, float v) const {
    const size_t o = (size_t)m * ldc + n;
    C[o] = R[o] + v;
  }
};

// SwiGLU backward of dm = acc at (b, j): dg = dm u sigma(g) (1 + g (1 -
// sigma(g))), du = dm g sigma(g) to dY [B][2f] (columns j, f + j) and the
// transposed rows j, f + j of dYT.
template <typename T>
struct EpiSwigluBwd {
  const float* g;
  const float* u;
  int f;
  T* dY;
  T* dYT;
  int ldT;
  __device__ __forceinline__ void operator()(int m, int n, float v) const {
    const size_t o = (size_t)m * f + n;
    const float gv = g[o], uv = u[o];
    const float sg = sigmoid_acc(gv);
    const T dgq = from_f32<T>(v * uv * sg * (1.f + gv * (1.f - sg)));
    const T duq = from_f32<T>(v * gv * sg);
    dY[(size_t)m * 2 * f + n] = dgq;
    dY[(size_t)m * 2 * f + f + n] = duq;
    dYT[(size_t)n * ldT + m] = dgq;
    dYT[(size_t)(f + n) * ldT + m] = duq;
  }
};

// d[e; s] = acc at (b, n): n < d adds to the e gradient of position *pos,
// the rest to ds [B][d].
struct EpiMergeBwd {
  float* de;  // [B][T_mem][d] or null
  float* ds;
  int d, T_mem;
  const int* pos;
  __device__ __forceinline__ void operator()(int m, int n, float v) const {
    if (n < d) {
      if (de) de[((size_t)m * T_mem + *pos) * d + n] += v;
    } else {
      ds[(size_t)m * d + n - d] += v;
    }
  }
};

// Query gradient of the memory attention of position p = *pos (positions
// 0..p, see the header; LSE from lse_rec + p * lse_stride), with D = g.o from
// the stored output o (storage type), written as the next projection's
// operands: dqY [B][d] in the storage type and transposed to dqT; D to Dout
// [B][H] when given.  One warp per (b, h).
template <typename T>
__global__ void attn_bwd_kernel(const float* __restrict__ q, const float* __restrict__ gout, const T* __restrict__ o,
                                const float* __restrict__ lse_rec, size_t lse_stride, const T* __restrict__ K,
                                const T* __restrict__ V, int Tk, const int* __restrict__ pos, int B, int H, int hd,
                                float scale, float* __restrict__ Dout, T* __restrict__ dqY, T* __restrict__ dqT,
                                int ldT) {
  const int pair = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (pair >= B * H) return;
  const int j0 = 0, j1 = *pos;
  const float* lse = lse_rec + (size_t)j1 * lse_stride;
  const int b = pair / H, h = pair - b * H;
  const int d = H * hd;
  const int NC = (hd + 31) >> 5;
  float qr[4], gr[4], acc[4];
  float Dp = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    const bool ok = c < NC && i < hd;
    const size_t col = (size_t)b * d + h * hd + i;
    qr[c] = ok ? q[col] : 0.f;
    gr[c] = ok ? gout[col] : 0.f;
    acc[c] = 0.f;
    if (ok) Dp = fmaf(gr[c], to_f32(o[col]), Dp);
  }
  const float D = warp_sum(Dp);
  if (Dout && lane == 0) Dout[pair] = D;
  const float ls = lse[pair];
  const T* Kb = K + ((size_t)b * H + h) * Tk * hd;
  const T* Vb = V + ((size_t)b * H + h) * Tk * hd;
  for (int j = j0; j <= j1; ++j) {
    float kv[4], sp = 0.f, dpp = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      kv[c] = 0.f;
      if (c < NC && i < hd) {
        kv[c] = to_f32(Kb[(size_t)j * hd + i]);
        sp = fmaf(qr[c], kv[c], sp);
        dpp = fmaf(gr[c], to_f32(Vb[(size_t)j * hd + i]), dpp);
      }
    }
    const float P = expf(warp_sum(sp) * scale - ls);
    const float dS = P * (warp_sum(dpp) - D);
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c] = fmaf(dS, kv[c], acc[c]);
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    if (c < NC && i < hd) {
      const size_t col = (size_t)h * hd + i;
      const T v = from_f32<T>(scale * acc[c]);
      dqY[(size_t)b * d + col] = v;
      dqT[col * ldT + b] = v;
    }
  }
}

// Query-gradient partials over the key split of memory positions 0..*pos
// (see attn_part_fwd_kernel): warp (pair, s) writes sum_{j in its chunk}
// dS_j K_j (unscaled; zero for an empty chunk) and D = g.o.
template <typename T>
__global__ void attn_part_bwd_kernel(const float* __restrict__ q, const float* __restrict__ gout,
                                     const T* __restrict__ o, const float* __restrict__ lse_rec, size_t lse_stride,
                                     const T* __restrict__ K, const T* __restrict__ V, int Tk,
                                     const int* __restrict__ pos, int B, int H, int hd, float scale, int nsplit,
                                     float* __restrict__ part) {
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wid >= B * H * nsplit) return;
  const int j0 = 0, j1 = *pos;
  const float* lse = lse_rec + (size_t)j1 * lse_stride;
  const int pair = wid / nsplit, sp = wid - pair * nsplit;
  const int b = pair / H, h = pair - b * H;
  const int d = H * hd;
  const int NC = (hd + 31) >> 5;
  const int ja = j0 + sp * kAttnChunk, jb = min(j1, ja + kAttnChunk - 1);
  float qr[4], gr[4], acc[4];
  float Dp = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    const bool ok = c < NC && i < hd;
    const size_t col = (size_t)b * d + h * hd + i;
    qr[c] = ok ? q[col] : 0.f;
    gr[c] = ok ? gout[col] : 0.f;
    acc[c] = 0.f;
    if (ok) Dp = fmaf(gr[c], to_f32(o[col]), Dp);
  }
  const float D = warp_sum(Dp);
  const float ls = lse[pair];
  const T* Kb = K + ((size_t)b * H + h) * Tk * hd;
  const T* Vb = V + ((size_t)b * H + h) * Tk * hd;
  for (int j = ja; j <= jb; ++j) {
    float kv[4], spq = 0.f, dpp = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      kv[c] = 0.f;
      if (c < NC && i < hd) {
        kv[c] = to_f32(Kb[(size_t)j * hd + i]);
        spq = fmaf(qr[c], kv[c], spq);
        dpp = fmaf(gr[c], to_f32(Vb[(size_t)j * hd + i]), dpp);
      }
    }
    const float P = expf(warp_sum(spq) * scale - ls);
    const float dS = P * (warp_sum(dpp) - D);
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c] = fmaf(dS, kv[c], acc[c]);
  }
  float* pp = part + (size_t)wid * (hd + 2);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    if (c < NC && i < hd) pp[i] = acc[c];
  }
  if (lane == 0) pp[hd] = D;
}

// Combine of the query-gradient partials, one warp per (b, h): dq = scale *
// sum over splits in order, written as the next projection's operands (dqY
// [B][d] storage type, dqT transposed); D to Dout [B][H] when given.
template <typename T>
__global__ void attn_combine_bwd_kernel(const float* __restrict__ part, int nsplit, int B, int H, int hd, float scale,
                                        float* __restrict__ Dout, T* __restrict__ dqY, T* __restrict__ dqT, int ldT) {
  const int pair = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (pair >= B * H) return;
  const int b = pair / H, h = pair - b * H;
  const int d = H * hd;
  const int NC = (hd + 31) >> 5;
  const float* pp = part + (size_t)pair * nsplit * (hd + 2);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < nsplit; ++s) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      if (c < NC && i < hd) acc[c] += pp[(size_t)s * (hd + 2) + i];
    }
  }
  if (Dout && lane == 0) Dout[pair] = pp[hd];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    if (c < NC && i < hd) {
      const size_t col = (size_t)h * hd + i;
      const T v = from_f32<T>(scale * acc[c]);
      dqY[(size_t)b * d + col] = v;
      dqT[col * ldT + b] = v;
    }
  }
}

// Window attention backward of position p = *pos split over warps (pair,
// s): the query-gradient partial over key chunk s of positions
// max(0, p - W + 1)..p and the key/value-gradient partial of position p over
// record chunk s of positions p..p_last (p_last = p with the cache detached,
// else min(p + W - 1, Tk - 1); either chunk may be empty); this step's output
// gradient g (split 0 stores it in its record slot of gR), D = g.o with the
// stored output.  Partials part[(pair * nsplit + s) * (3 hd + 1)]: dq
// (unscaled), dK, dV, then D.  swa_combine_bwd_kernel finishes.
template <typename T>
__global__ void swa_part_bwd_kernel(const T* __restrict__ K, const T* __restrict__ V, int Tk,
                                    const int* __restrict__ pos, int W, int cache, const T* __restrict__ o,
                                    const float* __restrict__ g, const float* __restrict__ qR,
                                    float* __restrict__ gR, const float* __restrict__ lR,
                                    const float* __restrict__ DR, int B, int H, int hd, float scale, int nsplit,
                                    float* __restrict__ part) {
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wid >= B * H * nsplit) return;
  const int p = *pos, j0 = p - W + 1 > 0 ? p - W + 1 : 0;
  const int p_last = cache ? p : min(p + W - 1, Tk - 1);
  const int pair = wid / nsplit, sp = wid - pair * nsplit;
  const int b = pair / H, h = pair - b * H;
  const int d = H * hd;
  const int NC = (hd + 31) >> 5;
  const size_t r0 = (size_t)(p % W) * B + b;
  float qr[4], gr[4], kp[4], vp[4], dq[4], dk[4], dv[4];
  float Dp = 0.f;
  const size_t kpo = (((size_t)b * H + h) * Tk + p) * hd;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    const bool ok = c < NC && i < hd;
    qr[c] = ok ? qR[r0 * d + h * hd + i] : 0.f;
    gr[c] = ok ? g[(size_t)b * d + h * hd + i] : 0.f;
    kp[c] = ok ? to_f32(K[kpo + i]) : 0.f;
    vp[c] = ok ? to_f32(V[kpo + i]) : 0.f;
    dq[c] = dk[c] = dv[c] = 0.f;
    if (ok) Dp = fmaf(gr[c], to_f32(o[(size_t)b * d + h * hd + i]), Dp);
    if (ok && sp == 0) gR[r0 * d + h * hd + i] = gr[c];  // this step's record
  }
  const float D = warp_sum(Dp);
  const float ls = lR[r0 * H + h];
  const T* Kb = K + ((size_t)b * H + h) * Tk * hd;
  const T* Vb = V + ((size_t)b * H + h) * Tk * hd;
  const int ja = j0 + sp * kAttnChunk, jb = min(p, ja + kAttnChunk - 1);
  for (int j = ja; j <= jb; ++j) {
    float kv[4], s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      kv[c] = 0.f;
      if (c < NC && i < hd) {
        kv[c] = to_f32(Kb[(size_t)j * hd + i]);
        s1 = fmaf(qr[c], kv[c], s1);
        s2 = fmaf(gr[c], to_f32(Vb[(size_t)j * hd + i]), s2);
      }
    }
    const float P = expf(warp_sum(s1) * scale - ls);
    const float dS = P * (warp_sum(s2) - D);
#pragma unroll
    for (int c = 0; c < 4; ++c) dq[c] = fmaf(dS, kv[c], dq[c]);
  }
  const int ra = p + sp * kAttnChunk, rb = min(p_last, ra + kAttnChunk - 1);
  for (int pp = ra; pp <= rb; ++pp) {
    const size_t rr = (size_t)(pp % W) * B + b;
    float qv[4], gv[4], s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      const bool ok = c < NC && i < hd;
      qv[c] = pp == p ? qr[c] : (ok ? qR[rr * d + h * hd + i] : 0.f);
      gv[c] = pp == p ? gr[c] : (ok ? gR[rr * d + h * hd + i] : 0.f);
      s1 = fmaf(qv[c], kp[c], s1);
      s2 = fmaf(gv[c], vp[c], s2);
    }
    const float lsr = pp == p ? ls : lR[rr * H + h];
    const float Dr = pp == p ? D : DR[rr * H + h];
    const float P = expf(warp_sum(s1) * scale - lsr);
    const float dS = P * (warp_sum(s2) - Dr);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      dk[c] = fmaf(scale * dS, qv[c], dk[c]);
      dv[c] = fmaf(P, gv[c], dv[c]);
    }
  }
  float* pp_ = part + (size_t)wid * (3 * hd + 1);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    if (c < NC && i < hd) {
      pp_[i] = dq[c];
      pp_[hd + i] = dk[c];
      pp_[2 * hd + i] = dv[c];
    }
  }
  if (lane == 0) pp_[3 * hd] = D;
}

// Combine of the window-backward partials, one warp per (b, h): sums in split
// order, D to this step's record, then dq (scaled) and dK back through RoPE at
// p and dV as is into d qkv dY [B][3d] and its transposed slot dYT.
template <typename T>
__global__ void swa_combine_bwd_kernel(const float* __restrict__ part, int nsplit, const int* __restrict__ pos, int W,
                                       int B, int H, int hd, float scale, float theta, float* __restrict__ DR,
                                       T* __restrict__ dY, T* __restrict__ dYT, int ldT) {
  const int pair = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (pair >= B * H) return;
  const int p = *pos;
  const int b = pair / H, h = pair - b * H;
  const int d = H * hd, half = hd >> 1;
  const int NC = (hd + 31) >> 5;
  const float* pp = part + (size_t)pair * nsplit * (3 * hd + 1);
  float dq[4] = {0.f, 0.f, 0.f, 0.f}, dk[4] = {0.f, 0.f, 0.f, 0.f}, dv[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < nsplit; ++s) {
    const float* ps = pp + (size_t)s * (3 * hd + 1);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      if (c < NC && i < hd) {
        dq[c] += ps[i];
        dk[c] += ps[hd + i];
        dv[c] += ps[2 * hd + i];
      }
    }
  }
  if (lane == 0) DR[((size_t)(p % W) * B + b) * H + h] = pp[3 * hd];
#pragma unroll
  for (int c = 0; c < 4; ++c) dq[c] *= scale;
  float out_q[4], out_k[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    const float qp = rope_partner(dq, c, hd), kpp = rope_partner(dk, c, hd);
    float cs = 1.f, sn = 0.f;
    if (c < NC && i < hd) rope_cs(p, i % half, hd, theta, cs, sn);
    const float sg = (i % hd) < half ? 1.f : -1.f;
    out_q[c] = dq[c] * cs + sg * qp * sn;
    out_k[c] = dk[c] * cs + sg * kpp * sn;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    if (c < NC && i < hd) {
      const int cq = h * hd + i, ck = d + h * hd + i, cv = 2 * d + h * hd + i;
      const T vq = from_f32<T>(out_q[c]), vk = from_f32<T>(out_k[c]), vv = from_f32<T>(dv[c]);
      dY[(size_t)b * 3 * d + cq] = vq;
      dY[(size_t)b * 3 * d + ck] = vk;
      dY[(size_t)b * 3 * d + cv] = vv;
      dYT[(size_t)cq * ldT + b] = vq;
      dYT[(size_t)ck * ldT + b] = vk;
      dYT[(size_t)cv * ldT + b] = vv;
    }
  }
}

// Window attention backward of position p = *pos (one layer), one warp per
// (b, h): this step's output gradient g (stored to its record slot p mod W of
// gR), its record's query and LSE, and the stored output o give D = g.o
// (written to the record) and the query gradient over positions
// max(0, p - W + 1)..p; the key/value gradient of position p comes from the
// records of positions p..p_last (p_last = p with the cache detached, else
// min(p + W - 1, Tk - 1); this step's from registers):
//   dK = sum scale dS q,  dV = sum P g,  P = exp(scale q.K_p - lse),
//   dS = P (g.V_p - D);
// then dq and dK back through RoPE at p and dV as is, into d qkv
// dY [B][3d] (storage type) and its transposed slot dYT.
template <typename T>
__global__ void swa_bwd_kernel(const T* __restrict__ K, const T* __restrict__ V, int Tk, const int* __restrict__ pos,
                               int W, int cache, const T* __restrict__ o, const float* __restrict__ g,
                               const float* __restrict__ qR, float* __restrict__ gR, const float* __restrict__ lR,
                               float* __restrict__ DR, int B, int H, int hd, float scale, float theta,
                               T* __restrict__ dY, T* __restrict__ dYT, int ldT) {
  const int pair = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (pair >= B * H) return;
  const int p = *pos, j0 = p - W + 1 > 0 ? p - W + 1 : 0;
  const int p_last = cache ? p : min(p + W - 1, Tk - 1);
  const int b = pair / H, h = pair - b * H;
  const int d = H * hd, half = hd >> 1;
  const int NC = (hd + 31) >> 5;
  const size_t r0 = (size_t)(p % W) * B + b;  // this step's record row
  float qr[4], gr[4], kp[4], vp[4], dq[4], dk[4], dv[4];
  float Dp = 0.f;
  const size_t kpo = (((size_t)b * H + h) * Tk + p) * hd;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    const bool ok = c < NC && i < hd;
    qr[c] = ok ? qR[r0 * d + h * hd + i] : 0.f;
    gr[c] = ok ? g[(size_t)b * d + h * hd + i] : 0.f;
    kp[c] = ok ? to_f32(K[kpo + i]) : 0.f;
    vp[c] = ok ? to_f32(V[kpo + i]) : 0.f;
    dq[c] = dk[c] = dv[c] = 0.f;
    if (ok) Dp = fmaf(gr[c], to_f32(o[(size_t)b * d + h * hd + i]), Dp);
    if (ok) gR[r0 * d + h * hd + i] = gr[c];  // this step's record
  }
  const float D = warp_sum(Dp);
  const float ls = lR[r0 * H + h];
  if (lane == 0) DR[r0 * H + h] = D;
  const T* Kb = K + ((size_t)b * H + h) * Tk * hd;
  const T* Vb = V + ((size_t)b * H + h) * Tk * hd;
  // query gradient over the window
  for (int j = j0; j <= p; ++j) {
    float kv[4], sp = 0.f, dpp = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      kv[c] = 0.f;
      if (c < NC && i < hd) {
        kv[c] = to_f32(Kb[(size_t)j * hd + i]);
        sp = fmaf(qr[c], kv[c], sp);
        dpp = fmaf(gr[c], to_f32(Vb[(size_t)j * hd + i]), dpp);
      }
    }
    const float P = expf(warp_sum(sp) * scale - ls);
    const float dS = P * (warp_sum(dpp) - D);
#pragma unroll
    for (int c = 0; c < 4; ++c) dq[c] = fmaf(dS, kv[c], dq[c]);
  }
  // key/value gradient of position p from the records of p..p_last
  for (int pp = p; pp <= p_last; ++pp) {
    const size_t rr = (size_t)(pp % W) * B + b;
    float qv[4], gv[4], s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      const bool ok = c < NC && i < hd;
      qv[c] = pp == p ? qr[c] : (ok ? qR[rr * d + h * hd + i] : 0.f);
      gv[c] = pp == p ? gr[c] : (ok ? gR[rr * d + h * hd + i] : 0.f);
      s1 = fmaf(qv[c], kp[c], s1);
      s2 = fmaf(gv[c], vp[c], s2);
    }
    const float lsr = pp == p ? ls : lR[rr * H + h];
    const float Dr = pp == p ? D : DR[rr * H + h];
    const float P = expf(warp_sum(s1) * scale - lsr);
    const float dS = P * (warp_sum(s2) - Dr);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      dk[c] = fmaf(scale * dS, qv[c], dk[c]);
      dv[c] = fmaf(P, gv[c], dv[c]);
    }
  }
  // back through RoPE at p: (y1, y2) -> (y1 c + y2 s, -y1 s + y2 c)
#pragma unroll
  for (int c = 0; c < 4; ++c) dq[c] *= scale;
  float out_q[4], out_k[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    const float qp = rope_partner(dq, c, hd), kpp = rope_partner(dk, c, hd);
    float cs = 1.f, sn = 0.f;
    if (c < NC && i < hd) rope_cs(p, i % half, hd, theta, cs, sn);
    const float sg = (i % hd) < half ? 1.f : -1.f;
    out_q[c] = dq[c] * cs + sg * qp * sn;
    out_k[c] = dk[c] * cs + sg * kpp * sn;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = lane + 32 * c;
    if (c < NC && i < hd) {
      const int cq = h * hd + i, ck = d + h * hd + i, cv = 2 * d + h * hd + i;
      const T vq = from_f32<T>(out_q[c]), vk = from_f32<T>(out_k[c]), vv = from_f32<T>(dv[c]);
      dY[(size_t)b * 3 * d + cq] = vq;
      dY[(size_t)b * 3 * d + ck] = vk;
      dY[(size_t)b * 3 * d + cv] = vv;
      dYT[(size_t)cq * ldT + b] = vq;
      dYT[(size_t)ck * ldT + b] = vk;
      dYT[(size_t)cv * ldT + b] = vv;
    }
  }
}

// Memory gradient of one block of steps, key-parallel: for every position
// j <= p_hi of one (b, h),
//   dK_j += sum scale dS q,  dV_j += sum P g,
// over the block's steps s < nb whose position p_hi - s >= j and the layers
// l0 <= l < l1 reading this memory group, with the step's query q (qS),
// output gradient g (gS) [S][L][B][d], log-sum-exp (lse_all [n][L][B][H] at
// the step's position) and D (DS [S][L][B][H]); P = exp(scale q.K_j - lse),
// dS = P (g.V_j - D).  Grid (key blocks of kMemKeys, B * H); each warp owns
// kMemKeysPerWarp keys (accumulators in registers, one read-modify-write per
// key at the end); the block's queries pass through shared memory in chunks
// of kMemQueries.
constexpr int kMemWarps = 8, kMemKeysPerWarp = 4, kMemKeys = kMemWarps * kMemKeysPerWarp, kMemQueries = 32;
template <typename T>
__global__ void __launch_bounds__(kMemWarps * 32) mem_grad_kernel(
    const T* __restrict__ K, const T* __restrict__ V, int T_mem, const float* __restrict__ qS,
    const float* __restrict__ gS, const float* __restrict__ lse_all, const float* __restrict__ DS, int L, int l0,
    int l1, int nb, int p_hi, int B, int H, int hd, float scale, float* __restrict__ dK, float* __restrict__ dV) {
  __shared__ float sq[kMemQueries][128];
  __shared__ float sg[kMemQueries][128];
  __shared__ float sl[kMemQueries], sD[kMemQueries];
  __shared__ int sp[kMemQueries];
  const int bh = blockIdx.y, b = bh / H, h = bh - b * H;
  const int d = H * hd, nl = l1 - l0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int NC = (hd + 31) >> 5;
  const int jb = blockIdx.x * kMemKeys;            // lowest key of the block
  if (jb > p_hi) return;                           // uniform over the block
  const int s_end = min(nb, p_hi - jb + 1);        // steps that reach key jb
  const int nq = s_end * nl;
  float kr[kMemKeysPerWarp][4], vr[kMemKeysPerWarp][4], ak[kMemKeysPerWarp][4], av[kMemKeysPerWarp][4];
  int jj[kMemKeysPerWarp];
#pragma unroll
  for (int u = 0; u < kMemKeysPerWarp; ++u) {
    jj[u] = jb + warp * kMemKeysPerWarp + u;
    const bool kv_ok = jj[u] <= p_hi;
    const size_t base = ((size_t)bh * T_mem + (kv_ok ? jj[u] : 0)) * hd;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      const bool ok = kv_ok && c < NC && i < hd;
      kr[u][c] = ok ? to_f32(K[base + i]) : 0.f;
      vr[u][c] = ok ? to_f32(V[base + i]) : 0.f;
      ak[u][c] = 0.f;
      av[u][c] = 0.f;
    }
  }
  for (int q0 = 0; q0 < nq; q0 += kMemQueries) {
    const int cnt = min(kMemQueries, nq - q0);
    __syncthreads();  // the previous chunk is consumed
    for (int e = threadIdx.x; e < cnt * hd; e += blockDim.x) {
      const int qi = e / hd, i = e - qi * hd;
      const int s = (q0 + qi) / nl, l = l0 + (q0 + qi) - s * nl;
      const size_t row = ((size_t)s * L + l) * B + b;
      sq[qi][i] = qS[row * d + h * hd + i];
      sg[qi][i] = gS[row * d + h * hd + i];
    }
    for (int qi = threadIdx.x; qi < cnt; qi += blockDim.x) {
      const int s = (q0 + qi) / nl, l = l0 + (q0 + qi) - s * nl;
      const int p = p_hi - s;
      sp[qi] = p;
      sl[qi] = lse_all[(((size_t)p * L + l) * B + b) * H + h];
      sD[qi] = DS[(((size_t)s * L + l) * B + b) * H + h];
    }
    __syncthreads();
    for (int qi = 0; qi < cnt; ++qi) {
      float qv[4], gv[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = lane + 32 * c;
        const bool ok = c < NC && i < hd;
        qv[c] = ok ? sq[qi][i] : 0.f;
        gv[c] = ok ? sg[qi][i] : 0.f;
      }
      const int p = sp[qi];
      const float ls = sl[qi], Dq = sD[qi];
#pragma unroll
      for (int u = 0; u < kMemKeysPerWarp; ++u) {
        if (jj[u] > p) continue;  // uniform over the warp
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          s1 = fmaf(qv[c], kr[u][c], s1);
          s2 = fmaf(gv[c], vr[u][c], s2);
        }
        const float P = expf(warp_sum(s1) * scale - ls);
        const float dS = P * (warp_sum(s2) - Dq);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          ak[u][c] = fmaf(scale * dS, qv[c], ak[u][c]);
          av[u][c] = fmaf(P, gv[c], av[u][c]);
        }
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kMemKeysPerWarp; ++u) {
    if (jj[u] > p_hi) continue;
    const size_t base = ((size_t)bh * T_mem + jj[u]) * hd;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = lane + 32 * c;
      if (c < NC && i < hd) {
        dK[base + i] += ak[u][c];
        dV[base + i] += av[u][c];
      }
    }
  }
}

// Memory gradient on the tensor cores (bf16 models): the sums of
// mem_grad_kernel as a flash-attention backward without the query gradient.
// Per (b, h) and 16-key tile of a warp, over the block's queries in chunks of
// 16 (staged in shared memory as bf16, row-major and transposed):
//   S^T = K Q^T, dP^T = V G^T          (keys x queries, bf16 MMAs over hd)
//   P^T = exp(scale S^T - lse), zero for keys past the query's position,
//   dS^T = P^T (dP^T - D),
//   dK += (scale dS^T) Q,  dV += P^T G  (MMAs over the queries)
// with the accumulators in registers for the whole block of steps and one
// fp32 read-modify-write per key at the end.  The MMA operands q, g, P and
// dS are rounded to bf16 (the CUDA-core kernel keeps them in fp32).
constexpr int kMgWarps = 4, kMgKeys = 16 * kMgWarps, kMgQ = 16;
template <int HD>
__global__ void __launch_bounds__(kMgWarps * 32) mem_grad_tc_kernel(
    const bf16* __restrict__ K, const bf16* __restrict__ V, int T_mem, const float* __restrict__ qS,
    const float* __restrict__ gS, const float* __restrict__ lse_all, const float* __restrict__ DS, int L, int l0,
    int l1, int nb, int p_hi, int B, int H, float scale, float* __restrict__ dK, float* __restrict__ dV) {
  __shared__ __align__(16) bf16 sq[kMgQ][HD + 8];
  __shared__ __align__(16) bf16 sg[kMgQ][HD + 8];
  __shared__ __align__(16) bf16 sqT[HD][kMgQ + 8];
  __shared__ __align__(16) bf16 sgT[HD][kMgQ + 8];
  __shared__ float sl[kMgQ], sD[kMgQ];
  __shared__ int sp[kMgQ];
  constexpr int NK = HD / 16, NN = HD / 8;
  const int bh = blockIdx.y, b = bh / H, h = bh - b * H, d = H * HD, nl = l1 - l0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
  const int jb = blockIdx.x * kMgKeys;
  if (jb > p_hi) return;  // uniform over the block
  const int j0 = jb + warp * 16;  // this warp's keys j0 .. j0 + 15
  const int s_end = min(nb, p_hi - jb + 1);
  const int nq = s_end * nl;
  const size_t base = (size_t)bh * T_mem;
  auto ldpair = [&](const bf16* M, int row, int col) -> unsigned {  // elements (row, col), (row, col + 1)
    return row > p_hi ? 0u : *reinterpret_cast<const unsigned*>(M + (base + row) * HD + col);
  };
  auto spair = [](const bf16* p) { return *reinterpret_cast<const unsigned*>(p); };
  auto pack = [](float lo, float hi) {
    return (unsigned)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((unsigned)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
  };
  unsigned ka[NK][4], va[NK][4];  // the warp's K and V rows as A operands (16 keys x 16 of hd)
#pragma unroll
  for (int kk = 0; kk < NK; ++kk) {
    const int c0 = 16 * kk + 2 * c;
    ka[kk][0] = ldpair(K, j0 + g, c0);
    ka[kk][1] = ldpair(K, j0 + g + 8, c0);
    ka[kk][2] = ldpair(K, j0 + g, c0 + 8);
    ka[kk][3] = ldpair(K, j0 + g + 8, c0 + 8);
    va[kk][0] = ldpair(V, j0 + g, c0);
    va[kk][1] = ldpair(V, j0 + g + 8, c0);
    va[kk][2] = ldpair(V, j0 + g, c0 + 8);
    va[kk][3] = ldpair(V, j0 + g + 8, c0 + 8);
  }
  float dk[NN][4], dv[NN][4];
#pragma unroll
  for (int nn = 0; nn < NN; ++nn)
#pragma unroll
    for (int q = 0; q < 4; ++q) dk[nn][q] = dv[nn][q] = 0.f;
  for (int q0 = 0; q0 < nq; q0 += kMgQ) {
    const int cnt = min(kMgQ, nq - q0);
    __syncthreads();  // the previous chunk is consumed
    for (int e = threadIdx.x; e < kMgQ * HD; e += blockDim.x) {
      const int qi = e / HD, i = e - qi * HD;
      float qv = 0.f, gv = 0.f;
      if (qi < cnt) {
        const int s = (q0 + qi) / nl, l = l0 + (q0 + qi) - s * nl;
        const size_t row = ((size_t)s * L + l) * B + b;
        qv = qS[row * d + h * HD + i];
        gv = gS[row * d + h * HD + i];
      }
      const bf16 qb = __float2bfloat16_rn(qv), gb = __float2bfloat16_rn(gv);
      sq[qi][i] = qb;
      sqT[i][qi] = qb;
      sg[qi][i] = gb;
      sgT[i][qi] = gb;
    }
    for (int qi = threadIdx.x; qi < kMgQ; qi += blockDim.x) {
      if (qi < cnt) {
        const int s = (q0 + qi) / nl, l = l0 + (q0 + qi) - s * nl, p = p_hi - s;
        sp[qi] = p;
        sl[qi] = lse_all[(((size_t)p * L + l) * B + b) * H + h];
        sD[qi] = DS[(((size_t)s * L + l) * B + b) * H + h];
      } else {  // padding: every key masked
        sp[qi] = -1;
        sl[qi] = 0.f;
        sD[qi] = 0.f;
      }
    }
    __syncthreads();
    if (j0 > p_hi) continue;  // uniform over the warp
    float st[2][4] = {}, dpt[2][4] = {};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int kk = 0; kk < NK; ++kk) {
        const unsigned bq[2] = {spair(&sq[8 * nt + g][16 * kk + 2 * c]), spair(&sq[8 * nt + g][16 * kk + 2 * c + 8])};
        const unsigned bg[2] = {spair(&sg[8 * nt + g][16 * kk + 2 * c]), spair(&sg[8 * nt + g][16 * kk + 2 * c + 8])};
        fused::mma_bf16(st[nt], ka[kk], bq);
        fused::mma_bf16(dpt[nt], va[kk], bg);
      }
    float P[2][4], dS[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int key = j0 + g + 8 * (q >> 1), qi = 8 * nt + 2 * c + (q & 1);
        const float pv = key <= sp[qi] ? expf(st[nt][q] * scale - sl[qi]) : 0.f;
        P[nt][q] = pv;
        dS[nt][q] = scale * pv * (dpt[nt][q] - sD[qi]);
      }
    // the 16 x 16 accumulator tiles as A operands (queries on k)
    const unsigned pa[4] = {pack(P[0][0], P[0][1]), pack(P[0][2], P[0][3]), pack(P[1][0], P[1][1]),
                            pack(P[1][2], P[1][3])};
    const unsigned sa[4] = {pack(dS[0][0], dS[0][1]), pack(dS[0][2], dS[0][3]), pack(dS[1][0], dS[1][1]),
                            pack(dS[1][2], dS[1][3])};
#pragma unroll
    for (int nn = 0; nn < NN; ++nn) {
      const unsigned bq[2] = {spair(&sqT[8 * nn + g][2 * c]), spair(&sqT[8 * nn + g][2 * c + 8])};
      const unsigned bg[2] = {spair(&sgT[8 * nn + g][2 * c]), spair(&sgT[8 * nn + g][2 * c + 8])};
      fused::mma_bf16(dk[nn], sa, bq);
      fused::mma_bf16(dv[nn], pa, bg);
    }
  }
  if (j0 > p_hi) return;
#pragma unroll
  for (int nn = 0; nn < NN; ++nn)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int key = j0 + g + 8 * (q >> 1), col = 8 * nn + 2 * c + (q & 1);
      if (key <= p_hi) {
        dK[(base + key) * HD + col] += dk[nn][q];
        dV[(base + key) * HD + col] += dv[nn][q];
      }
    }
}

// Merge backward, one thread per column i (loop over sequences):
//   de[b][p][i] = dh (1 - z);  ds[b][i] = dh z;
//   gate: dzpre = dh (s - e) z (1 - z) to dY [B][d] (and transposed),
//         db_g[i] += sum_b dzpre.
template <typename T>
__global__ void merge_bwd_kernel(const float* __restrict__ dh, const float* __restrict__ z, const T* __restrict__ e,
                                 int T_mem, const int* __restrict__ pos, const float* __restrict__ s_all, int B,
                                 int d, int gate, T* __restrict__ dY, T* __restrict__ dYT, int ldT,
                                 float* __restrict__ dbg, float* __restrict__ de, float* __restrict__ ds) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d) return;
  const int p = *pos;
  const float* s = s_all + (size_t)p * B * d;
  float acc = 0.f;
  for (int b = 0; b < B; ++b) {
    const size_t o = (size_t)b * d + i;
    const size_t oe = ((size_t)b * T_mem + p) * d + i;
    const float g = dh[o], zv = z[o];
    if (de) de[oe] = g * (1.f - zv);
    ds[o] = g * zv;
    if (gate) {
      const float dz = g * (s[o] - to_f32(e[oe])) * zv * (1.f - zv);
      const T q = from_f32<T>(dz);
      dY[o] = q;
      dYT[(size_t)i * ldT + b] = q;
      acc += dz;
    }
  }
  if (gate) dbg[i] += acc;
}

// out[i] += sum_b x[b][i].
__global__ void colsum_kernel(const float* __restrict__ x, int B, int d, float* __restrict__ out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d) return;
  float acc = 0.f;
  for (int b = 0; b < B; ++b) acc += x[(size_t)b * d + i];
  out[i] += acc;
}

// loss = -sum over (b, t) with 0 <= a < V of lp[b][t]; one block of
// kThreads, fixed summation order.
__global__ void loss_sum_kernel(const float* __restrict__ lp, const int32_t* __restrict__ actions, int B, int n, int V,
                                float* __restrict__ loss) {
  __shared__ float red[kThreads];
  const int tid = threadIdx.x;
  float acc = 0.f;
  for (size_t i = tid; i < (size_t)B * n; i += blockDim.x)
    if (actions[i] >= 0 && actions[i] < V) acc -= lp[i];
  red[tid] = acc;
  __syncthreads();
  for (int s = blockDim.x >> 1; s > 0; s >>= 1) {
    if (tid < s) red[tid] += red[tid + s];
    __syncthreads();
  }
  if (tid == 0) *loss = red[0];
}

}  // namespace bptt
}  // namespace rlt
