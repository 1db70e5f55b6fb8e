// Decoder cross-attention to encoder memory positions 1..t (the step that
// streams the memory): for every sequence b and head h,
//   o[b][h] = sum_{j<t} softmax_j(q[b][h] . K[b][h][j] / sqrt(hd)) V[b][h][j].
// The same kernel runs the sliding-window self-attention over the ring cache:
// the window's entries occupy ring slots 0 .. min(W, t) - 1 (every slot once
// the ring is full), and softmax attention does not depend on the order of its
// entries, so attending to that slot range is attending to the window.
// Pages: "Understanding and Applying the Recurrent Looped Transformer
// Architecture", "Three forms of context" (cross-attention reads encoder
// memory only through the current position); "Princeton Researcher Proposes
// Recurrent Looped Transformer ...", architecture paragraph.
//
// Design (HBM streaming, ~1 flop per byte, no tensor-core shape):
//  - work item = (pair = b*H + h, chunk of CH positions); CH*hd*es = 16 KB, so
//    one chunk of K and one of V are each a single contiguous 16 KB span of
//    the [B][H][T][hd] memory plane, fetched by one bulk asynchronous copy
//    (TMA engine) into shared memory;
//  - persistent CTAs walk the items of the current t round-robin with a
//    two-stage copy pipeline (the next-but-one item is in flight while the
//    current one is reduced);
//  - inside a chunk: scores with hd/8 lanes per key row (16-byte shared loads,
//    conflict-free), exact chunk max and sum, then P.V with the same layout;
//  - chunks of a pair are merged by the CTA that finishes the pair's last
//    chunk (device-scope fence + arrival counter), so no second launch is
//    needed; a pair with a single chunk is written out directly.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace rlt {

constexpr int kXThreads = 128;
constexpr int kXChunkBytes = 16384;  // bytes of K (and of V) per chunk
constexpr int kXStages = 2;

template <typename T_, int HD>
struct XShape {
  static constexpr int ES = (int)sizeof(T_);
  static constexpr int EPL = 16 / ES;           // elements per lane (one 16-byte load)
  static constexpr int LPR = HD / EPL;          // lanes per key row
  static constexpr int RPW = 32 / LPR;          // rows per warp and pass
  static constexpr int NW = kXThreads / 32;
  static constexpr int RPB = RPW * NW;          // rows per block and pass
  static constexpr int CH = kXChunkBytes / (HD * ES);  // positions per chunk
  static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "unsupported head_dim");
  static_assert(CH % RPB == 0, "chunk must be a whole number of passes");
  static constexpr size_t smem_bytes() {
    return (size_t)2 * kXStages * kXChunkBytes + sizeof(float) * (CH + NW * HD) + sizeof(uint64_t) * 2 * kXStages;
  }
};

struct XattnArgs {
  const float* q;     // [B][d]  projected query (fp32, no RoPE)
  const void* mk;     // [B][H][T_mem][hd]  memory keys of one group
  const void* mv;     // [B][H][T_mem][hd]  memory values
  float* part;        // [B*H][max_chunks][hd + 2]  (max, sum, unnormalised o)
  int* cnt;           // [B*H] arrival counters, zero between launches
  void* out;          // [B][d]  storage dtype
  int B, H, T_mem, max_chunks;
  int t_cap;          // attend to positions 0 .. min(t_cap, ctx->pos + 1) - 1
  float scale;
  const StepCtx* ctx;
  int* status;
};

template <typename T_, int EPL>
__device__ __forceinline__ void load_seg(const T_* p, float (&v)[EPL]);
template <>
__device__ __forceinline__ void load_seg<bf16, 8>(const bf16* p, float (&v)[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 f = __bfloat1622float2(h2[k]);
    v[2 * k] = f.x;
    v[2 * k + 1] = f.y;
  }
}
template <>
__device__ __forceinline__ void load_seg<float, 4>(const float* p, float (&v)[4]) {
  float4 f = *reinterpret_cast<const float4*>(p);
  v[0] = f.x;
  v[1] = f.y;
  v[2] = f.z;
  v[3] = f.w;
}

template <typename T_, int HD>
__global__ void __launch_bounds__(kXThreads) dec_xattn_kernel(XattnArgs a) {
  using S = XShape<T_, HD>;
  constexpr int CH = S::CH, EPL = S::EPL, LPR = S::LPR, RPW = S::RPW, RPB = S::RPB, NW = S::NW;
  extern __shared__ __align__(128) unsigned char xsm[];
  T_* sK = reinterpret_cast<T_*>(xsm);
  T_* sV = reinterpret_cast<T_*>(xsm + kXStages * kXChunkBytes);
  float* sp = reinterpret_cast<float*>(xsm + 2 * kXStages * kXChunkBytes);  // [CH]
  float* red = sp + CH;                                                       // [NW][HD]
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + NW * HD);                 // K stages, then V stages
  __shared__ float s_max[NW], s_sum[NW];
  __shared__ int s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane % LPR, rg = lane / LPR;
  const int t = min(a.t_cap, a.ctx->pos + 1);
  const int nch = (t + CH - 1) / CH;
  const int n_items = a.B * a.H * nch;
  const int d = a.H * HD;
  const T_* mk = static_cast<const T_*>(a.mk);
  const T_* mv = static_cast<const T_*>(a.mv);
  T_* out = static_cast<T_*>(a.out);

  if (tid == 0) {
    for (int i = 0; i < 2 * kXStages; ++i) mbar_init(&bar[i], 1);
    fence_mbar_init();
  }
  __syncwarp();
  __syncthreads();

  auto issue = [&](int item, int stage) {  // one thread
    const int pair = item / nch, c = item - pair * nch;
    const int j0 = c * CH, nj = min(CH, t - j0);
    const unsigned bytes = (unsigned)(nj * HD * S::ES);
    const size_t off = ((size_t)pair * a.T_mem + j0) * HD;
    mbar_arrive_expect_tx(&bar[stage], bytes);
    bulk_g2s(sK + stage * (CH * HD), mk + off, bytes, &bar[stage]);
    mbar_arrive_expect_tx(&bar[kXStages + stage], bytes);
    bulk_g2s(sV + stage * (CH * HD), mv + off, bytes, &bar[kXStages + stage]);
  };

  int item = blockIdx.x;
  if (tid == 0) {
    if (item < n_items) issue(item, 0);
    if (item + (int)gridDim.x < n_items) issue(item + gridDim.x, 1);
  }
  __syncwarp();  // warps reach every block-wide barrier converged
  unsigned phase = 0;  // bit s: parity of the next completion of stage s
  for (int it = 0; item < n_items; item += gridDim.x, ++it) {
    const int s = it & 1;
    const unsigned par = (phase >> s) & 1u;
    const int pair = item / nch, c = item - pair * nch;
    const int b = pair / a.H, h = pair - b * a.H;
    const int j0 = c * CH, nj = min(CH, t - j0);
    float qr[EPL];
    {
      const float* qp = a.q + (size_t)b * d + h * HD + sub * EPL;
#pragma unroll
      for (int e = 0; e < EPL; ++e) qr[e] = qp[e];
    }
    // ---- scores over the chunk's keys
    bool ok = mbar_wait(&bar[s], par, kWaitBudget);
    if (__syncthreads_or(!ok)) goto fail;
    {
      const T_* Ks = sK + s * (CH * HD);
      float lmax = -INFINITY;
      for (int r0 = warp * RPW; r0 < nj; r0 += RPB) {  // warp-uniform bound
        const int r = r0 + rg;
        float dot = 0.f;
        if (r < nj) {
          float kv[EPL];
          load_seg<T_, EPL>(Ks + r * HD + sub * EPL, kv);
#pragma unroll
          for (int e = 0; e < EPL; ++e) dot = fmaf(qr[e], kv[e], dot);
        }
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (r < nj) {
          dot *= a.scale;
          if (sub == 0) sp[r] = dot;
          lmax = fmaxf(lmax, dot);
        }
      }
      lmax = warp_max(lmax);
      if (lane == 0) s_max[warp] = lmax;
    }
    __syncthreads();
    {
      float m = s_max[0];
#pragma unroll
      for (int w = 1; w < NW; ++w) m = fmaxf(m, s_max[w]);
      float lsum = 0.f;
      for (int j = tid; j < nj; j += kXThreads) {
        const float p = expf(sp[j] - m);
        sp[j] = p;
        lsum += p;
      }
      lsum = warp_sum(lsum);
      if (lane == 0) s_sum[warp] = lsum;
      ok = mbar_wait(&bar[kXStages + s], par, kWaitBudget);
      if (__syncthreads_or(!ok)) goto fail;
      float l = s_sum[0];
#pragma unroll
      for (int w = 1; w < NW; ++w) l += s_sum[w];
      // ---- P . V
      const T_* Vs = sV + s * (CH * HD);
      float acc[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
      for (int r0 = warp * RPW; r0 < nj; r0 += RPB) {
        const int r = r0 + rg;
        if (r < nj) {
          const float p = sp[r];
          float vv[EPL];
          load_seg<T_, EPL>(Vs + r * HD + sub * EPL, vv);
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[e] = fmaf(p, vv[e], acc[e]);
        }
      }
#pragma unroll
      for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
      if (rg == 0)
#pragma unroll
        for (int e = 0; e < EPL; ++e) red[warp * HD + sub * EPL + e] = acc[e];
      __syncthreads();  // stage s fully consumed, red complete
      if (tid == 0 && item + 2 * (int)gridDim.x < n_items) issue(item + 2 * gridDim.x, s);
      __syncwarp();
      phase ^= (1u << s);
      if (nch == 1) {
        for (int i = tid; i < HD; i += kXThreads) {
          float o = 0.f;
#pragma unroll
          for (int w = 0; w < NW; ++w) o += red[w * HD + i];
          out[(size_t)b * d + h * HD + i] = from_f32<T_>(o / l);
        }
        continue;
      }
      float* pr = a.part + ((size_t)pair * a.max_chunks + c) * (HD + 2);
      for (int i = tid; i < HD; i += kXThreads) {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) o += red[w * HD + i];
        pr[2 + i] = o;
      }
      if (tid == 0) {
        pr[0] = m;
        pr[1] = l;
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) s_last = (atomicAdd(&a.cnt[pair], 1) == nch - 1);
      __syncwarp();
      __syncthreads();
      if (s_last) {
        __threadfence();
        const float* pp = a.part + (size_t)pair * a.max_chunks * (HD + 2);
        float M = -INFINITY;
        for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, __ldcg(pp + (size_t)cc * (HD + 2)));
        float L = 0.f;
        for (int cc = 0; cc < nch; ++cc)
          L += __ldcg(pp + (size_t)cc * (HD + 2) + 1) * expf(__ldcg(pp + (size_t)cc * (HD + 2)) - M);
        for (int i = tid; i < HD; i += kXThreads) {
          float o = 0.f;
          for (int cc = 0; cc < nch; ++cc)
            o += __ldcg(pp + (size_t)cc * (HD + 2) + 2 + i) * expf(__ldcg(pp + (size_t)cc * (HD + 2)) - M);
          out[(size_t)b * d + h * HD + i] = from_f32<T_>(o / L);
        }
        if (tid == 0) a.cnt[pair] = 0;  // ready for the next launch
      }
    }
  }
  return;
fail:
  // a copy never completed: record it, give in-flight copies a bounded time
  // to land (they write this CTA's shared memory), then leave
  if (tid == 0) {
    set_error(a.status, kErrTimeout);
    for (int s2 = 0; s2 < kXStages; ++s2) {
      const unsigned p2 = (phase >> s2) & 1u;
      mbar_wait(&bar[s2], p2, kWaitBudget);
      mbar_wait(&bar[kXStages + s2], p2, kWaitBudget);
    }
  }
  __syncthreads();
}

// Host-side launch: grid = resident CTAs on every SM (persistent).
template <typename T_, int HD>
inline cudaError_t launch_xattn_hd(const XattnArgs& a, int n_sm, cudaStream_t st) {
  using S = XShape<T_, HD>;
  static int occ = 0;
  if (occ == 0) {
    cudaFuncSetAttribute(dec_xattn_kernel<T_, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)S::smem_bytes());
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, dec_xattn_kernel<T_, HD>, kXThreads, S::smem_bytes()) !=
            cudaSuccess ||
        o < 1)
      o = 1;
    occ = o;
  }
  dec_xattn_kernel<T_, HD><<<n_sm * occ, kXThreads, S::smem_bytes(), st>>>(a);
  return cudaGetLastError();
}

template <typename T_>
inline int xattn_chunk(int hd) {
  return kXChunkBytes / (hd * (int)sizeof(T_));
}

template <typename T_>
inline cudaError_t launch_xattn(const XattnArgs& a, int hd, int n_sm, cudaStream_t st) {
  switch (hd) {
    case 8: return launch_xattn_hd<T_, 8>(a, n_sm, st);
    case 16: return launch_xattn_hd<T_, 16>(a, n_sm, st);
    case 32: return launch_xattn_hd<T_, 32>(a, n_sm, st);
    case 64: return launch_xattn_hd<T_, 64>(a, n_sm, st);
    case 128: return launch_xattn_hd<T_, 128>(a, n_sm, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rlt
