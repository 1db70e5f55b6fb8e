// Encoder causal self-attention of bf16 models on the 5th-generation tensor
// cores (tcgen05 MMAs, fp32 accumulators in tensor memory, operands staged by
// the TMA engine):
//   o[b][t][h*HD + i] = sum_{j<=t} softmax_j(q[b][h][t] . k[b][h][j] / sqrt(HD)) v[b][h][j][i]
// Pages: "Princeton Researcher Proposes Recurrent Looped Transformer ...",
// architecture paragraph (the encoder is a token-parallel causal stack);
// "Understanding and Applying the Recurrent Looped Transformer Architecture",
// "How the Architecture Works".
//
// One CTA = 128 queries of one (b, h); 192 threads:
//   warp 0     TMA producer: the Q tile once, then K blocks (both passes) and
//              V^T blocks (second pass) through 2-deep rings;
//   warp 1     allocates tensor memory; one lane issues the MMAs
//              S = Q K^T (128 x 128 keys, into one of two S buffers) and
//              O += P V (128 x HD, accumulated over the key blocks), the
//              S of block j + 1 ahead of the P V of block j, so that the
//              tensor core computes the next scores while the softmax
//              works on the current ones;
//   warps 2-5  softmax: thread = query row = tensor-memory lane.
// Two passes over the keys, as the numerics contract asks (P rounded to bf16
// on the grid of the final row maximum, the denominator summed from the
// unrounded P): the first pass only takes each row's maximum m of the scaled
// scores; the second forms P = exp2(s - m), adds it to the row sum, writes
// bf16(P) into shared memory in the operand layout of the second MMA (K-major,
// 128-byte swizzle; two P buffers) and lets the MMA warp add P V.  Every
// operand is K-major:
// V enters transposed ([b][h][HD][T], written by vt_transpose_kernel), so that
// its key blocks are [HD rows][keys] tiles like the K blocks.
// Every wait is bounded (RLT_ETIMEOUT in the status word on expiry); tensor
// memory is freed on every path.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace rlt {
namespace fat {

constexpr int BQ = 128;      // queries per CTA (MMA M)
constexpr int BKV = 128;     // keys per block (MMA N of S, K of P V)
constexpr int THREADS = 192;
constexpr int ST = 2;        // K and V ring depth
constexpr int TILE = 16384;  // one 128-row x 128-byte swizzled k-block

template <int HD>
struct Lay {
  static_assert(HD == 64 || HD == 128, "head width");
  static constexpr int QK_KB = HD / 64;                   // 64-element k-blocks of Q and K rows
  static constexpr int Q_BYTES = QK_KB * TILE;            // [128 q][HD]
  static constexpr int K_BYTES = QK_KB * TILE;            // [128 keys][HD]
  static constexpr int V_BYTES = 2 * HD * 128;            // two [HD rows][64 keys] k-blocks
  static constexpr int P_BYTES = 2 * TILE;                // two [128 q][64 keys] k-blocks per P buffer
  static constexpr int o_q = 0;
  static constexpr int o_k = o_q + Q_BYTES;
  static constexpr int o_v = o_k + ST * K_BYTES;
  static constexpr int o_p = o_v + ST * V_BYTES;
  static constexpr int o_bar = o_p + 2 * P_BYTES;
  static constexpr int N_BARS = 1 + 4 * ST + 2 * 2 + 2 * 2 + 1;  // q, k/v full/empty, s and p full/empty [2], o
  static constexpr size_t SMEM = 1024 + (size_t)o_bar + 8 * N_BARS + 16;
  static constexpr int TMEM_COLS = 512;                   // S0 [0,128), S1 [128,256), O [256, 256 + HD)
};

using tc::fence_async_smem;

// q, k: [B*H][T][HD] (maps tm_q, tm_k: dims {HD, T, B*H}, box {64, 128, 1});
// vt: [B*H][HD][T] (map tm_v: dims {T, HD, B*H}, box {64, HD, 1});
// o: [B][T][H*HD].  scale_log2 = log2(e) / sqrt(HD).
template <int HD>
__global__ void __launch_bounds__(THREADS, 1)
    enc_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, bf16* __restrict__ o, int T, int H, float scale_log2,
                       int* status) {
  using Lo = Lay<HD>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lo::o_bar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + ST;
  uint64_t* v_full = k_empty + ST;
  uint64_t* v_empty = v_full + ST;
  uint64_t* s_full = v_empty + ST;   // [2]
  uint64_t* s_empty = s_full + 2;    // [2], 128 arrivals
  uint64_t* p_full = s_empty + 2;    // [2], 128 arrivals
  uint64_t* p_empty = p_full + 2;    // [2]
  uint64_t* o_full = p_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_full + 1);
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (T + BQ - 1) / BQ;
  const int qb = nqb - 1 - (int)blockIdx.x;  // longest (latest) query blocks first
  const int h = blockIdx.y, b = blockIdx.z, bh = b * H + h;
  const int q0 = qb * BQ;
  const int nkb = (min(T, q0 + BQ) + BKV - 1) / BKV;  // key blocks 0 .. the diagonal one
  const int n_it = 2 * nkb;                          // pass 0 then pass 1

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], 128);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&p_full[s], 128);
      mbar_init(&p_empty[s], 1);
    }
    mbar_init(o_full, 1);
    s_fail = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tm_q);
    tc::tma_prefetch_desc(&tm_k);
    tc::tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, Lo::TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto failed = [&]() { return *reinterpret_cast<volatile int*>(&s_fail) != 0; };
  auto fail = [&]() { atomicExch(&s_fail, 1); };
  int k_issued = 0, v_issued = 0;  // producer: loads requested

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, Lo::Q_BYTES);
      for (int kk = 0; kk < Lo::QK_KB; ++kk) tc::tma_load_3d(sm + Lo::o_q + kk * TILE, &tm_q, 64 * kk, q0, bh, q_full);
      for (int it = 0; it < n_it && !failed(); ++it) {
        const int kb = it % nkb, s = it % ST;
        if (it >= ST && !mbar_wait(&k_empty[s], ((it / ST) - 1) & 1, kWaitBudget)) {
          fail();
          break;
        }
        unsigned char* kd = sm + Lo::o_k + s * Lo::K_BYTES;
        mbar_arrive_expect_tx(&k_full[s], Lo::K_BYTES);
        for (int kk = 0; kk < Lo::QK_KB; ++kk) tc::tma_load_3d(kd + kk * TILE, &tm_k, 64 * kk, kb * BKV, bh, &k_full[s]);
        k_issued = it + 1;
        if (it >= nkb) {  // second pass: the V^T block of the same keys
          const int j = kb, sv = j % ST;
          if (j >= ST && !mbar_wait(&v_empty[sv], ((j / ST) - 1) & 1, kWaitBudget)) {
            fail();
            break;
          }
          unsigned char* vd = sm + Lo::o_v + sv * Lo::V_BYTES;
          mbar_arrive_expect_tx(&v_full[sv], Lo::V_BYTES);
          for (int kk = 0; kk < 2; ++kk) tc::tma_load_3d(vd + kk * (HD * 128), &tm_v, kb * BKV + 64 * kk, 0, bh, &v_full[sv]);
          v_issued = j + 1;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_s = tc::idesc_bf16_f32(BQ, BKV);
      constexpr uint32_t id_o = tc::idesc_bf16_f32(BQ, HD);
      bool ok = mbar_wait(q_full, 0, kWaitBudget);
      if (!ok) fail();
      // O += P V of second-pass block j (P buffer j mod 2, V stage j mod ST)
      auto pv = [&](int j) -> bool {
        const int pb = j & 1, sv = j % ST;
        if (!mbar_wait(&p_full[pb], (j >> 1) & 1, kWaitBudget) || !mbar_wait(&v_full[sv], (j / ST) & 1, kWaitBudget))
          return false;
        tc::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint64_t da = tc::sdesc_k_sw128(sm + Lo::o_p + pb * Lo::P_BYTES + kk * TILE);
          const uint64_t db = tc::sdesc_k_sw128(sm + Lo::o_v + sv * Lo::V_BYTES + kk * (HD * 128));
#pragma unroll
          for (int k = 0; k < 4; ++k) tc::mma_bf16(tmem + 2 * BKV, da + 2 * k, db + 2 * k, id_o, (j | kk | k) ? 1 : 0);
        }
        tc::mma_commit(&p_empty[pb]);
        tc::mma_commit(&v_empty[sv]);
        return true;
      };
      for (int it = 0; ok && it < n_it && !failed(); ++it) {
        const int s = it % ST, sb = it & 1;
        if (!mbar_wait(&k_full[s], (it / ST) & 1, kWaitBudget) ||
            (it >= 2 && !mbar_wait(&s_empty[sb], ((it / 2) - 1) & 1, kWaitBudget))) {
          fail();
          ok = false;
          break;
        }
        tc::tc_fence_after();
        // S = Q K^T over HD in 16-element MMAs
        const uint32_t ts = tmem + sb * BKV;
#pragma unroll
        for (int kk = 0; kk < Lo::QK_KB; ++kk) {
          const uint64_t da = tc::sdesc_k_sw128(sm + Lo::o_q + kk * TILE);
          const uint64_t db = tc::sdesc_k_sw128(sm + Lo::o_k + s * Lo::K_BYTES + kk * TILE);
#pragma unroll
          for (int k = 0; k < 4; ++k) tc::mma_bf16(ts, da + 2 * k, db + 2 * k, id_s, (kk | k) ? 1 : 0);
        }
        tc::mma_commit(&s_full[sb]);
        tc::mma_commit(&k_empty[s]);
        // the previous iteration's block, once its P is written
        if (it - 1 >= nkb && !pv(it - 1 - nkb)) {
          fail();
          ok = false;
          break;
        }
      }
      if (ok && !failed() && !pv(nkb - 1)) fail();  // the last block
      tc::mma_commit(o_full);  // arrives once every issued MMA has completed
    }
    __syncwarp();
  } else {
    // softmax warps: query row r = tensor-memory lane
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int row = q0 + r;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    float m = -INFINITY, l = 0.f;
    const int sw = r & 7;
    // (every decision to leave is warp-uniform: tcgen05.ld is a warp-wide instruction)
    for (int it = 0; it < n_it; ++it) {
      if (!__all_sync(0xffffffffu, !failed())) break;
      const int kb = it % nkb, sb = it & 1;
      const bool second = it >= nkb;
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[sb], (it / 2) & 1, kWaitBudget))) {
        fail();
        break;
      }
      tc::tc_fence_after();
      const int pb = kb & 1;  // P buffer of this block
      if (second && kb >= 2 && !__all_sync(0xffffffffu, mbar_wait(&p_empty[pb], ((kb >> 1) - 1) & 1, kWaitBudget))) {
        fail();  // (the wait: the P V two blocks back has read this P buffer)
        break;
      }
      const int key0 = kb * BKV;
      // keys past this row (the diagonal block) or past T score -inf
      const int kmax = min(row, T - 1) - key0;  // keys key0 .. key0 + kmax are valid
      unsigned char* prow = sm + Lo::o_p + pb * Lo::P_BYTES + r * 128;
#pragma unroll 1
      for (int c1 = 0; c1 < BKV; c1 += 64) {
        uint32_t v[4][16];  // 64 columns in flight, one wait
#pragma unroll
        for (int u = 0; u < 4; ++u) tc::tmem_ld16_async(tl + sb * BKV + c1 + 16 * u, v[u]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c0 = c1 + 16 * u;
          float x[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) x[e] = (c0 + e <= kmax) ? __uint_as_float(v[u][e]) * scale_log2 : -INFINITY;
          if (!second) {
#pragma unroll
            for (int e = 0; e < 16; ++e) m = fmaxf(m, x[e]);
          } else {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float p0 = exp2f(x[2 * e] - m), p1 = exp2f(x[2 * e + 1] - m);  // exp2(-inf) = 0
              l += p0 + p1;
              __nv_bfloat162 t2 = __floats2bfloat162_rn(p0, p1);
              pk[e] = *reinterpret_cast<uint32_t*>(&t2);
            }
            // keys c0 .. c0 + 15: 16-byte chunks (c0 % 64) / 8 and + 1 of k-block c0 / 64
            const int kk = c0 >> 6, ch = (c0 & 63) >> 3;
            unsigned char* base = prow + kk * TILE;
            *reinterpret_cast<uint4*>(base + ((ch ^ sw) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(base + (((ch + 1) ^ sw) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
      tc::tc_fence_before();
      mbar_arrive(&s_empty[sb]);  // this S buffer may be overwritten
      if (second) {
        fence_async_smem();  // P (generic-proxy stores) visible to the MMA (async proxy)
        mbar_arrive(&p_full[pb]);
      }
    }
    // O / l, rounded to bf16, to o[b][row][h*HD ..]
    const bool ok = __all_sync(0xffffffffu, !failed() && mbar_wait(o_full, 0, kWaitBudget));
    if (!ok) fail();
    tc::tc_fence_after();
    if (ok) {
      const float inv = 1.f / l;
      bf16* orow = o + ((size_t)b * T + row) * (size_t)(H * HD) + (size_t)h * HD;
#pragma unroll 1
      for (int c1 = 0; c1 < HD; c1 += 64) {
        uint32_t v[4][16];  // 64 columns in flight, one wait
#pragma unroll
        for (int u = 0; u < 4; ++u) tc::tmem_ld16_async(tl + 2 * BKV + c1 + 16 * u, v[u]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c0 = c1 + 16 * u;
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            __nv_bfloat162 t2 =
                __floats2bfloat162_rn(__uint_as_float(v[u][2 * e]) * inv, __uint_as_float(v[u][2 * e + 1]) * inv);
            pk[e] = *reinterpret_cast<uint32_t*>(&t2);
          }
          if (row < T) {
            *reinterpret_cast<uint4*>(orow + c0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(orow + c0 + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (s_fail && threadIdx.x == 0) {
    set_error(status, kErrTimeout);
    // give the copies still in flight a bounded time to land before leaving
    for (int i = max(0, k_issued - ST); i < k_issued; ++i) mbar_wait(&k_full[i % ST], (i / ST) & 1, kWaitBudget);
    for (int j = max(0, v_issued - ST); j < v_issued; ++j) mbar_wait(&v_full[j % ST], (j / ST) & 1, kWaitBudget);
    mbar_wait(q_full, 0, kWaitBudget);
  }
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, Lo::TMEM_COLS);
}

// v [BH][T][HD] -> vt [BH][HD][T] through 32 x 32 shared-memory tiles
// (block 32 x 8, grid (ceil(T / 32), HD / 32, BH)).
__global__ void vt_transpose_kernel(const bf16* __restrict__ v, bf16* __restrict__ vt, int T, int HD) {
  __shared__ bf16 tile[32][34];
  const int bh = blockIdx.z, t0 = blockIdx.x * 32, i0 = blockIdx.y * 32;
  const bf16* src = v + (size_t)bh * T * HD;
  bf16* dst = vt + (size_t)bh * HD * T;
  for (int y = threadIdx.y; y < 32; y += 8) {
    const int t = t0 + y;
    tile[y][threadIdx.x] = t < T ? src[(size_t)t * HD + i0 + threadIdx.x] : __float2bfloat16(0.f);
  }
  __syncthreads();
  for (int y = threadIdx.y; y < 32; y += 8) {
    const int t = t0 + threadIdx.x;
    if (t < T) dst[(size_t)(i0 + y) * T + t] = tile[threadIdx.x][y];
  }
}

}  // namespace fat
}  // namespace rlt
