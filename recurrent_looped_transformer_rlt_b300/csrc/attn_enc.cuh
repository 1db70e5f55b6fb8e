// Encoder causal self-attention, flash style, for bf16 models:
//   o[b][t][h*hd + i] = sum_{j<=t} softmax_j(q[b][h][t] . k[b][h][j] / sqrt(hd)) v[b][h][j][i]
// Pages: "Princeton Researcher Proposes Recurrent Looped Transformer ...",
// architecture paragraph (the encoder is a token-parallel causal stack);
// "Understanding and Applying the Recurrent Looped Transformer Architecture",
// "How the Architecture Works".
//
// One CTA = 64 queries of one (b, h), 4 warps x 16 query rows; keys and values
// stream through shared memory in 64-row blocks (double-buffered cp.async);
// S = Q K^T and O += P V on the tensor cores (m16n8k16 bf16, fp32
// accumulation).  Two passes over the keys: the first finds each row's max m
// of the scores, the second forms P = exp(s - m), rounds it to bf16 for P V
// (the rounding point of the numerics contract, on the same grid - the final
// row max - as a plain softmax), and sums the unrounded P for the
// denominator; the output is rounded to bf16.  The extra pass costs one more
// Q K^T (1.5x the FLOPs of a one-pass kernel) and buys rounding decisions
// that agree with the plain definition instead of a running-max grid.  Query
// blocks are scheduled latest first (the causal triangle makes them longest).
#pragma once

#include "common.cuh"

namespace rlt {
namespace fa {

constexpr int BQ = 64, BKV = 64, THREADS = 128;

__device__ __forceinline__ void cp16(void* smem, const void* gmem, bool valid) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void wait_group() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], const void* p) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(s));
}
__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], const void* p) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(s));
}
__device__ __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int HD>
constexpr size_t smem_bytes() {
  return (size_t)(BQ + 4 * BKV) * (HD + 8) * sizeof(bf16);
}

// q, k, v: [B][H][T][HD] bf16; o: [B][T][H*HD] bf16.  scale_log2 =
// log2(e) / sqrt(HD).
template <int HD>
__global__ void __launch_bounds__(THREADS) enc_flash_kernel(const bf16* __restrict__ q, const bf16* __restrict__ k,
                                                            const bf16* __restrict__ v, bf16* __restrict__ o, int T,
                                                            int H, float scale_log2) {
  constexpr int LDS = HD + 8;  // padded rows: conflict-free ldmatrix
  constexpr int KS = HD / 16, ND = HD / 8;
  extern __shared__ __align__(16) unsigned char fsm[];
  bf16* sQ = reinterpret_cast<bf16*>(fsm);  // [BQ][LDS]
  bf16* sK = sQ + BQ * LDS;                  // [2][BKV][LDS]
  bf16* sV = sK + 2 * BKV * LDS;             // [2][BKV][LDS]
  const int nqb = (T + BQ - 1) / BQ;
  const int qb = nqb - 1 - (int)blockIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t base = (((size_t)b * H + h) * T) * HD;
  const int q0 = qb * BQ;

  auto load_tile = [&](bf16* dst, const bf16* src, int row0) {
#pragma unroll 4
    for (int i = tid; i < 64 * (HD / 8); i += THREADS) {
      const int r = i / (HD / 8), c = (i % (HD / 8)) * 8;
      const bool ok = row0 + r < T;
      cp16(dst + r * LDS + c, ok ? src + base + (size_t)(row0 + r) * HD + c : src, ok);
    }
  };
  const int nkb = qb + 1;  // key blocks 0 .. qb (causal)
  const int row_a = q0 + warp * 16 + (lane >> 2);  // this thread's rows: row_a, row_a + 8
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  float oacc[ND][4];
#pragma unroll
  for (int n = 0; n < ND; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[n][e] = 0.f;
  uint32_t qf[KS][4];

  load_tile(sQ, q, q0);
  load_tile(sK, k, 0);
  commit();
  // pass 0: row maxima (K only); pass 1: P, row sums and P V (K and V)
  for (int pass = 0; pass < 2; ++pass) {
    if (pass == 1) {
      load_tile(sK, k, 0);
      load_tile(sV, v, 0);
      commit();
    }
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb & 1;
      if (kb + 1 < nkb) {
        load_tile(sK + (st ^ 1) * BKV * LDS, k, (kb + 1) * BKV);
        if (pass == 1) load_tile(sV + (st ^ 1) * BKV * LDS, v, (kb + 1) * BKV);
      }
      commit();
      wait_group<1>();  // everything but the newest group has landed
      __syncthreads();
      if (pass == 0 && kb == 0) {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) ldsm4(qf[ks], sQ + (warp * 16 + (lane & 15)) * LDS + ks * 16 + (lane >> 4) * 8);
      }
      // ---- S = Q K^T: 16 rows x 64 keys per warp
      float s[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
      const bf16* Ks = sK + st * BKV * LDS;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int nj = 0; nj < 4; ++nj) {
          uint32_t bb[4];
          ldsm4(bb, Ks + (nj * 16 + (lane & 7) + ((lane >> 4) << 3)) * LDS + ks * 16 + ((lane >> 3) & 1) * 8);
          mma(s[2 * nj], qf[ks], bb[0], bb[1]);
          mma(s[2 * nj + 1], qf[ks], bb[2], bb[3]);
        }
      // ---- causal mask, scale (log2 units)
      const int kbase = kb * BKV;
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kbase + n * 8 + 2 * (lane & 3) + (e & 1);
          const int row = row_a + (e >> 1) * 8;
          s[n][e] = (key <= row && key < T) ? s[n][e] * scale_log2 : -INFINITY;
        }
      if (pass == 0) {
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) m_r[e >> 1] = fmaxf(m_r[e >> 1], s[n][e]);
      } else {
        // ---- P = exp(s - m), row sums of the unrounded P, O += bf16(P) V
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float mrow = m_r[e >> 1];
            const float p = (mrow == -INFINITY) ? 0.f : exp2f(s[n][e] - mrow);
            s[n][e] = p;
            l_r[e >> 1] += p;
          }
        const bf16* Vs = sV + st * BKV * LDS;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t a[4];
          a[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
          a[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
          a[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
          a[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
          for (int nd = 0; nd < HD / 16; ++nd) {
            uint32_t bb[4];
            ldsm4t(bb, Vs + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LDS + nd * 16 + (lane >> 4) * 8);
            mma(oacc[2 * nd], a, bb[0], bb[1]);
            mma(oacc[2 * nd + 1], a, bb[2], bb[3]);
          }
        }
      }
      __syncthreads();  // stage st is read; the next iteration refills it
    }
    wait_group<0>();
    if (pass == 0) {
      // row max over the quad of lanes that share a row
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        m_r[r] = fmaxf(m_r[r], __shfl_xor_sync(0xffffffffu, m_r[r], 1));
        m_r[r] = fmaxf(m_r[r], __shfl_xor_sync(0xffffffffu, m_r[r], 2));
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
  }
  // ---- normalise and store o[b][t][h*HD + i] (bf16)
  const int d = H * HD;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = row_a + r * 8;
    if (row >= T) continue;
    const float inv = 1.f / l_r[r];
    bf16* orow = o + ((size_t)b * T + row) * d + h * HD;
#pragma unroll
    for (int n = 0; n < ND; ++n) {
      const int dim = n * 8 + 2 * (lane & 3);
      *reinterpret_cast<__nv_bfloat162*>(orow + dim) =
          __floats2bfloat162_rn(oacc[n][2 * r] * inv, oacc[n][2 * r + 1] * inv);
    }
  }
}

}  // namespace fa
}  // namespace rlt
