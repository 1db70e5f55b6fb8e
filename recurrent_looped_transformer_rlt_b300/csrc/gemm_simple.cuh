// Epilogue functors of the projections (used by the tcgen05 kernel in
// gemm_tc.cuh and by the fp32 kernel below), and the fp32 CUDA-core GEMM of
// the fp32 models: C[M,N] = A[M,K] * B[N,K]^T with a per-element epilogue.
// Its B operand may come from two row blocks (rows n < n_split from B0, the
// rest from B1), which lets one launch cover W_1 and W_3 of a SwiGLU layer.
#pragma once

#include "common.cuh"

namespace rlt {

// ---------------------------------------------------------------------------
// epilogues: operator()(m, n, acc) is called once per in-range element.

// kStore4 / kAdd4: the tensor-core kernel writes (or adds into) C four
// columns at a time with 16-byte accesses (when ldc % 4 == 0).
struct EpiStoreF32 {
  static constexpr bool kStore4 = true;
  float* C;
  int ldc;
  __device__ __forceinline__ void operator()(int m, int n, float v) const { C[(size_t)m * ldc + n] = v; }
};
// Epilogues that declare kVec4 also take four consecutive columns n .. n + 3
// of one row at once (store4; n a multiple of 4, all four inside N), with the
// same values as four calls of operator().
template <typename T>
struct EpiStoreT {  // store rounded to the storage type
  static constexpr bool kVec4 = true;
  T* C;
  int ldc;
  __device__ __forceinline__ void operator()(int m, int n, float v) const { C[(size_t)m * ldc + n] = from_f32<T>(v); }
  __device__ __forceinline__ void store4(int m, int n, float4 v) const {
    T* p = C + (size_t)m * ldc + n;
    if ((reinterpret_cast<uintptr_t>(p) & (4 * sizeof(T) - 1)) == 0) {
      store4_st<T>(p, v);
    } else {
      p[0] = from_f32<T>(v.x);
      p[1] = from_f32<T>(v.y);
      p[2] = from_f32<T>(v.z);
      p[3] = from_f32<T>(v.w);
    }
  }
};
struct EpiAddF32 {  // residual stream update h += acc
  static constexpr bool kAdd4 = true;
  float* C;
  int ldc;
  __device__ __forceinline__ void operator()(int m, int n, float v) const { C[(size_t)m * ldc + n] += v; }
};
// Memory projection: row m = b*T + t, column n = h*hd + i, written to
// dst[b][h][t][i] (dst already offset to the group and key/value plane).
template <typename T>
struct EpiMemScatter {
  static constexpr bool kVec4 = true;
  T* dst;
  int T_len, H, hd;
  int T_stride = 0;  // positions per (b, h) plane row of dst; 0: T_len
  __device__ __forceinline__ void operator()(int m, int n, float v) const {
    int b = m / T_len, t = m - b * T_len;
    int h = n / hd, i = n - h * hd;
    const int ts = T_stride ? T_stride : T_len;
    dst[(((size_t)b * H + h) * ts + t) * hd + i] = from_f32<T>(v);
  }
  __device__ __forceinline__ void store4(int m, int n, float4 v) const {
    if (hd & 3) {  // four columns may cross a head: one at a time
      (*this)(m, n, v.x);
      (*this)(m, n + 1, v.y);
      (*this)(m, n + 2, v.z);
      (*this)(m, n + 3, v.w);
      return;
    }
    const int b = m / T_len, t = m - b * T_len;
    const int h = n / hd, i = n - h * hd;
    const int ts = T_stride ? T_stride : T_len;
    store4_st<T>(dst + (((size_t)b * H + h) * ts + t) * hd + i, v);
  }
};

// Memory keys or values of one position (incremental encoding): row m = b,
// column n = h*hd + i, written to dst[b][h][ctx->pos][i] of a plane with
// T_stride positions.
template <typename T>
struct EpiMemRow {
  T* dst;
  int T_stride, H, hd;
  const StepCtx* ctx;
  __device__ __forceinline__ void operator()(int m, int n, float v) const {
    const int h = n / hd, i = n - h * hd;
    dst[(((size_t)m * H + h) * T_stride + ctx->pos) * hd + i] = from_f32<T>(v);
  }
};

// Decoder QKV projection with RoPE, in pairs (i, i + hd/2) of one head:
// q (after RoPE, fp32) to q[b][d]; k (after RoPE) and v rounded to storage and
// written to ring slot pos mod W of this layer's ring [B][H][W][hd].
template <typename T>
struct EpiQKVRope {
  static constexpr bool kPair = true;
  float* q;
  T* ring_k;
  T* ring_v;
  const float2* tab;  // [position][hd/2] (cos, sin)
  const StepCtx* ctx;
  int d, H, hd, W;
  // what a pair of columns (n, n + hd/2) needs, the same for every row
  struct PairCtx {
    int which, head, i, slot;
    float2 cs;
  };
  __device__ __forceinline__ PairCtx pair_ctx(int n) const {
    PairCtx c;
    c.which = n / d;
    const int r = n - c.which * d;
    c.head = r / hd;
    c.i = r - c.head * hd;
    const int p = ctx->pos;
    c.slot = p % W;
    c.cs = (c.which == 2) ? make_float2(1.f, 0.f) : tab[(size_t)p * (hd >> 1) + c.i];
    return c;
  }
  __device__ __forceinline__ void pair(const PairCtx& c, int b, int, float x1, float x2) const {
    const int half = hd >> 1;
    if (c.which == 2) {
      const size_t o = (((size_t)b * H + c.head) * W + c.slot) * hd + c.i;
      ring_v[o] = from_f32<T>(x1);
      ring_v[o + half] = from_f32<T>(x2);
      return;
    }
    const float y1 = x1 * c.cs.x - x2 * c.cs.y, y2 = x2 * c.cs.x + x1 * c.cs.y;
    if (c.which == 0) {
      q[(size_t)b * d + c.head * hd + c.i] = y1;
      q[(size_t)b * d + c.head * hd + c.i + half] = y2;
    } else {
      const size_t o = (((size_t)b * H + c.head) * W + c.slot) * hd + c.i;
      ring_k[o] = from_f32<T>(y1);
      ring_k[o + half] = from_f32<T>(y2);
    }
  }
};

// Encoder QKV projection with RoPE, in pairs (i, i + hd/2) of one head: row
// m = b*T + t; q and k rotated at position t, v plain; all three rounded to
// storage and written head-major [B][H][T][hd].
template <typename T>
struct EpiEncQKVRope {
  static constexpr bool kPair = true;
  T* q;
  T* k;
  T* v;
  const float2* tab;  // [position][hd/2]
  int d, H, hd, T_len;
  struct PairCtx {
    int which, head, i;
  };
  __device__ __forceinline__ PairCtx pair_ctx(int n) const {
    PairCtx c;
    c.which = n / d;
    const int r = n - c.which * d;
    c.head = r / hd;
    c.i = r - c.head * hd;
    return c;
  }
  __device__ __forceinline__ void pair(const PairCtx& c, int m, int, float x1, float x2) const {
    const int half = hd >> 1;
    const int b = m / T_len, t = m - b * T_len;
    const size_t o = (((size_t)b * H + c.head) * T_len + t) * hd + c.i;
    if (c.which == 2) {
      v[o] = from_f32<T>(x1);
      v[o + half] = from_f32<T>(x2);
      return;
    }
    const float2 cs = tab[(size_t)t * half + c.i];
    T* dst = (c.which == 0) ? q : k;
    dst[o] = from_f32<T>(x1 * cs.x - x2 * cs.y);
    dst[o + half] = from_f32<T>(x2 * cs.x + x1 * cs.y);
  }
  // pairs i .. i + 3 of column n = which*d + head*hd + i (i a multiple of 4,
  // hd a multiple of 8): the same values as four calls of pair()
  static constexpr bool kPair4 = true;
  __device__ __forceinline__ void pair4(int m, int n, float4 x1, float4 x2) const {
    const int half = hd >> 1;
    const int which = n / d, r = n - which * d, head = r / hd, i = r - head * hd;
    const int b = m / T_len, t = m - b * T_len;
    const size_t o = (((size_t)b * H + head) * T_len + t) * hd + i;
    if (which == 2) {
      store4_st<T>(v + o, x1);
      store4_st<T>(v + o + half, x2);
      return;
    }
    const float4 c01 = *reinterpret_cast<const float4*>(tab + (size_t)t * half + i);  // (cos, sin) of i, i + 1
    const float4 c23 = *reinterpret_cast<const float4*>(tab + (size_t)t * half + i + 2);
    T* dst = (which == 0) ? q : k;
    store4_st<T>(dst + o, make_float4(x1.x * c01.x - x2.x * c01.y, x1.y * c01.z - x2.y * c01.w,
                                      x1.z * c23.x - x2.z * c23.y, x1.w * c23.z - x2.w * c23.w));
    store4_st<T>(dst + o + half, make_float4(x2.x * c01.x + x1.x * c01.y, x2.y * c01.z + x1.y * c01.w,
                                             x2.z * c23.x + x1.z * c23.y, x2.w * c23.z + x1.w * c23.w));
  }
};

// Epilogues that produce the residual stream h (fp32 [M][ldh]) declare kHOut,
// load(m, n) of what they combine with and combine(aux, acc4, n) -> the new
// h[m][n..n+3].  The kernel then writes h, optional copies s (fp32) and s16
// (bf16), and per row and 64-column block the sum of squares ss[n / 64][m]
// (the next RMSNorm reads these instead of reducing the row again).
struct HOut {
  float* h;
  int ldh;
  float* s;
  bf16* s16;
  float* ss;
  int M;
};
// h += acc (a residual update).
struct EpiResidual {
  static constexpr bool kHOut = true;
  HOut o;
  struct Aux {
    float4 old;
  };
  __device__ __forceinline__ Aux load(int m, int n) const {
    return Aux{*reinterpret_cast<const float4*>(o.h + (size_t)m * o.ldh + n)};
  }
  __device__ __forceinline__ float4 combine(const Aux& a, float4 v, int) const {
    return make_float4(a.old.x + v.x, a.old.y + v.y, a.old.z + v.z, a.old.w + v.w);
  }
};
// The gated merge h = z * s_{t-1} + (1 - z) * e_t with z = sigmoid(acc + b_g)
// (acc = W_g [e_t; s_{t-1}]); with discard, h = e_t.
struct EpiMerge {
  static constexpr bool kHOut = true;
  HOut o;
  const bf16* e;       // [B][T][d], row of sequence m at position ctx->pos
  size_t e_seq_stride;  // T * d
  const float* s_prev;  // [B][d]
  const float* bg;      // [d]
  const StepCtx* ctx;
  int discard;
  struct Aux {
    float4 e, s;
  };
  __device__ __forceinline__ Aux load(int m, int n) const {
    const bf16* ep = e + (size_t)m * e_seq_stride + (size_t)ctx->pos * o.ldh + n;
    const uint2 u = *reinterpret_cast<const uint2*>(ep);
    const float2 e01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 e23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return Aux{make_float4(e01.x, e01.y, e23.x, e23.y),
               *reinterpret_cast<const float4*>(s_prev + (size_t)m * o.ldh + n)};
  }
  __device__ __forceinline__ float4 combine(const Aux& a, float4 v, int n) const {
    if (discard) return a.e;
    const float4 b = *reinterpret_cast<const float4*>(bg + n);
    const float z0 = sigmoid_f(v.x + b.x), z1 = sigmoid_f(v.y + b.y), z2 = sigmoid_f(v.z + b.z),
                z3 = sigmoid_f(v.w + b.w);
    return make_float4(z0 * a.s.x + (1.f - z0) * a.e.x, z1 * a.s.y + (1.f - z1) * a.e.y,
                       z2 * a.s.z + (1.f - z2) * a.e.z, z3 * a.s.w + (1.f - z3) * a.e.w);
  }
};

struct GemmB {
  const void* B0;
  const void* B1;
  int n_split;  // rows n < n_split read B0[n], others B1[n - n_split]
  int ldb;
};

// ---------------------------------------------------------------------------
// fp32 CUDA-core kernel (fp32 models)

namespace simt_v0 {
constexpr int BM = 64, BN = 64, BK = 16, THREADS = 256;

template <class Epi>
__global__ void __launch_bounds__(THREADS) gemm_f32_kernel(const float* __restrict__ A, int lda, GemmB gb, int M,
                                                           int N, int K, Epi epi) {
  __shared__ float sA[BK][BM + 4];
  __shared__ float sB[BK][BN + 4];
  const int tid = threadIdx.x;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int tm = (tid / 16) * 4, tn = (tid % 16) * 4;
  const float* B0 = static_cast<const float*>(gb.B0);
  const float* B1 = static_cast<const float*>(gb.B1);
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int i = tid; i < BM * BK; i += THREADS) {
      int r = i / BK, c = i % BK;
      int gm = m0 + r, gk = k0 + c;
      sA[c][r] = (gm < M && gk < K) ? A[(size_t)gm * lda + gk] : 0.f;
      int gn = n0 + r;
      float bv = 0.f;
      if (gn < N && gk < K)
        bv = (gn < gb.n_split) ? B0[(size_t)gn * gb.ldb + gk] : B1[(size_t)(gn - gb.n_split) * gb.ldb + gk];
      sB[c][r] = bv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = sA[kk][tm + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = sB[kk][tn + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int m = m0 + tm + i, n = n0 + tn + j;
      if (m < M && n < N) epi(m, n, acc[i][j]);
    }
}
}  // namespace simt_v0

}  // namespace rlt
