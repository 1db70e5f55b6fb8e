// Decoder cross-attention to encoder memory positions 1..t (the step that
// streams the memory): for every sequence b and head h,
//   o[b][h] = sum_{j<t} softmax_j(q[b][h] . K[b][h][j] / sqrt(hd)) V[b][h][j].
// The same kernel runs the sliding-window self-attention over the ring cache:
// the window's entries occupy ring slots 0 .. min(W, t) - 1 (every slot once
// the ring is full), and softmax attention does not depend on the order of its
// entries, so attending to that slot range is attending to the window.
// Pages: "Understanding and Applying the Recurrent Looped Transformer
// Architecture", "Three forms of context" (cross-attention reads encoder
// memory only through the current position; the window includes the current
// token); "Princeton Researcher Proposes Recurrent Looped Transformer ...",
// architecture paragraph.
//
// Design (HBM streaming, ~1 flop per byte: no tensor-core shape):
//  - the keys of one (b, h) pair are contiguous in the [B][H][T][hd] plane; a
//    chunk is CH consecutive positions = 4 KB of K and 4 KB of V, each fetched
//    by one bulk asynchronous copy (TMA engine) into shared memory;
//  - work is split per warp, not per block: a task is (pair, split) = a run of
//    chunks of one pair; every warp owns a ring of ST chunk buffers (2 or 3) and
//    their mbarriers, walks its tasks chunk by chunk with the next chunk always
//    in flight (across task boundaries too), and keeps an online softmax
//    (running max, sum, output) in registers: no block-wide barrier;
//  - within a chunk hd*es/16 lanes share a key row (16-byte shared loads), so a
//    chunk is 8 passes of the warp over its rows; the 8 partial dot products
//    of a lane are summed over the row's lanes by a transposed butterfly (each
//    halving step exchanges half of the remaining values), which leaves every
//    lane the full scores of its own passes: one exp2 per score, and each
//    probability fetched by the lanes that need it for the value pass;
//  - the work is balanced exactly: the (pair, chunk) units are cut into one
//    contiguous run per warp (on the device, from t), a run's piece inside one
//    pair is a segment, the segments of a pair are merged by the warp that
//    arrives last on the pair's counter (acquire-release atomic), and a pair
//    covered by a single segment is written out directly;
//  - copies that do not depend on the previous kernel start before waiting for
//    it: all of the encoder memory, and every ring chunk except the one that
//    holds this step's slot.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace rlt {

constexpr int kXWarps = 4;           // warps per CTA (each independent)
constexpr int kXThreads = 32 * kXWarps;
constexpr int kXChunkBytes = 4096;   // bytes of K (and of V) per chunk
constexpr int kXMaxSplits = 32;      // splits per pair at most (partials buffer)
// resident CTAs per SM the kernel is built for, by ring depth (shared
// memory: 4 warps x ST stages x 8 KB)
__host__ __device__ constexpr int xattn_blocks_per_sm(int st) { return st <= 2 ? 3 : 2; }
constexpr float kLog2e = 1.4426950408889634f;

template <typename T_, int HD, int ST = 2>
struct XShape {
  static constexpr int ES = (int)sizeof(T_);
  static constexpr int EPL = 16 / ES;           // elements per lane (one 16-byte load)
  static constexpr int LPR = HD / EPL;          // lanes per key row
  static constexpr int RPW = 32 / LPR;          // rows per warp pass
  static constexpr int CH = kXChunkBytes / (HD * ES);  // positions per chunk
  static constexpr int PASSES = CH / RPW;       // = 8
  static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "unsupported head_dim");
  static_assert(CH % RPW == 0, "chunk must be a whole number of passes");
  // per warp: ST stages x (K, V) chunk buffers; then 2 ST mbarriers per warp
  static constexpr size_t smem_bytes() { return (size_t)kXWarps * 2 * ST * kXChunkBytes + 16 * ST * kXWarps; }
};

struct XattnArgs {
  const float* q;     // [B][d]  query (fp32; RoPE already applied for the window)
  const void* mk;     // [B][H][T_mem][hd]  keys (memory plane of one group, or a layer's ring)
  const void* mv;     // [B][H][T_mem][hd]  values
  float* part;        // [B*H][kXMaxSplits][hd + 2]  (max, sum, unnormalised o)
  int* cnt;           // [B*H] arrival counters, zero between launches
  void* out;          // [B][d]  storage dtype
  int B, H, T_mem;
  int t_cap;          // attend to positions 0 .. min(t_cap, ctx->pos + 1) - 1
  int early;          // which first copies may start before waiting for the previous kernel:
                      // 0 none; 1 all (keys/values written two or more kernels earlier,
                      // the encoder memory); 2 all but the chunk holding ring slot
                      // pos mod t_cap (the window: that entry is this step's)
  float scale;
  const StepCtx* ctx;
  int* status;
  long long budget;   // clock cycles a wait may take before it gives up (0: kWaitBudget)
  int withhold;       // failure injection: global warp 0 never requests its first value chunk,
                      // so its wait on it runs out (tests of the timeout path)
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

constexpr int kXMergeCost = 3;  // chunk times of emitting a partial and merging

// Arrival on a counter with release (this warp's partial) and acquire (the
// other warps' partials) semantics at device scope; returns the old value.
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;\n" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

template <typename T_, int HD, int ST>
__global__ void __launch_bounds__(kXThreads, xattn_blocks_per_sm(ST)) dec_xattn_kernel(XattnArgs a) {
  using S = XShape<T_, HD, ST>;
  constexpr int CH = S::CH, EPL = S::EPL, LPR = S::LPR, RPW = S::RPW, PASSES = S::PASSES;
  constexpr int CHE = CH * HD;  // elements per chunk buffer
  extern __shared__ __align__(128) unsigned char xsm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T_* sbuf = reinterpret_cast<T_*>(xsm + (size_t)warp * 2 * ST * kXChunkBytes);  // [stage][K|V][CHE]
  // K of stage s at bar[s], V at bar[ST + s]
  uint64_t* bar = reinterpret_cast<uint64_t*>(xsm + (size_t)kXWarps * 2 * ST * kXChunkBytes) + warp * 2 * ST;

  const int sub = lane % LPR, rg = lane / LPR;
  // transposed reduction of the PASSES partial dots over the LPR lanes of a
  // row group: LV halving steps (offsets LPR/2, LPR/4, ...) leave NV values per
  // lane, shared by REP lanes when LPR > PASSES
  constexpr int RL = LPR < PASSES ? LPR : PASSES;
  constexpr int NV = PASSES / RL, REP = LPR / RL;
  constexpr int LV = RL >= 8 ? 3 : RL >= 4 ? 2 : RL >= 2 ? 1 : 0;
  int idx = 0;  // this lane's block of passes: idx * NV .. idx * NV + NV - 1
#pragma unroll
  for (int lv = 0; lv < LV; ++lv) idx = (idx << 1) | ((lane & (LPR >> (lv + 1))) ? 1 : 0);
  const bool rep0 = (lane & (REP - 1)) == 0;
  const long long budget = a.budget > 0 ? a.budget : kWaitBudget;
  const int t = min(a.t_cap, a.ctx->pos + 1);
  const int nch = (t + CH - 1) / CH;
  const int pairs = a.B * a.H;
  const int warps = gridDim.x * kXWarps;
  const int gw = blockIdx.x * kXWarps + warp;
  // balanced partition: the U = pairs x nch (pair, chunk) units are cut into
  // wp contiguous runs, one per active warp (wp <= U so that no run is empty,
  // wp <= 31 pairs so that a pair spans at most 32 runs); the piece of a run
  // inside one pair is a segment, and the segments of a pair are merged
  // When every pair fits on its own warp and a whole pair takes no longer than
  // a balanced run plus the cost of a merge (~3 chunk times: partial store,
  // arrival, combine), each warp takes one whole pair instead (no merges).
  const int U = pairs * nch;
  const int wp_bal = min(warps, min(U, 31 * pairs));
  const int wp = (pairs <= warps && nch <= (U + wp_bal - 1) / wp_bal + kXMergeCost) ? pairs : wp_bal;
  const long long u_beg = gw < wp ? (long long)gw * U / wp : 0;
  const long long u_end = gw < wp ? (long long)(gw + 1) * U / wp : 0;
  auto owner = [&](long long u) { return (int)(((u + 1) * wp - 1) / U); };  // warp whose run holds unit u
  const int d = a.H * HD;
  const T_* mk = static_cast<const T_*>(a.mk);
  const T_* mv = static_cast<const T_*>(a.mv);
  T_* out = static_cast<T_*>(a.out);

  if (lane == 0) {
    for (int i = 0; i < 2 * ST; ++i) mbar_init(&bar[i], 1);
    fence_mbar_init();
  }
  __syncwarp();

  long long iu = u_beg;  // next unit to copy
  auto issue_next = [&](int stage) {  // lane 0
    if (iu >= u_end) return;
    const int pair = (int)(iu / nch), c0 = (int)(iu - (long long)pair * nch) * CH;
    const int nj = min(CH, t - c0);
    const unsigned bytes = (unsigned)(nj * HD * S::ES);
    const size_t off = ((size_t)pair * a.T_mem + c0) * HD;
    mbar_arrive_expect_tx(&bar[stage], bytes);
    bulk_g2s(sbuf + (stage * 2) * CHE, mk + off, bytes, &bar[stage]);
    mbar_arrive_expect_tx(&bar[ST + stage], bytes);
    if (!(a.withhold && gw == 0 && iu == u_beg))  // (injection: the bytes are expected, never sent)
      bulk_g2s(sbuf + (stage * 2 + 1) * CHE, mv + off, bytes, &bar[ST + stage]);
    ++iu;
  };
  // copies that may start before the previous kernel has finished: all of the
  // encoder memory (early = 1); the ring except the chunk that holds this
  // step's slot pos mod W, written by the projection just before (early = 2)
  int pre = 0;
  if (lane == 0 && a.early) {
    const int c_now = (a.early == 2) ? (a.ctx->pos % a.t_cap) / CH : -1;
    while (pre < ST && iu < u_end && (int)(iu % nch) != c_now) issue_next(pre++);
  }
  pre = __shfl_sync(0xffffffffu, pre, 0);
  pdl_wait();  // q, this step's ring entry and the outputs depend on the previous kernels
  if (threadIdx.x == 0) pdl_trigger();
  if (lane == 0)
    for (int s0 = pre; s0 < ST; ++s0) issue_next(s0);
  __syncwarp();

  unsigned phase = 0;  // bit s: parity of the next completion of stage s
  int used = 0;        // chunks consumed (stage = used % ST)
  float acc[EPL], qr[EPL];
  for (long long u = u_beg; u < u_end;) {
    const int pair = (int)(u / nch), cbeg = (int)(u - (long long)pair * nch);
    const long long seg_end = min(u_end, (long long)(pair + 1) * nch);
    const int nct = (int)(seg_end - u);
    u = seg_end;
    const int b = pair / a.H, h = pair - b * a.H;
    {
      const float* qp = a.q + (size_t)b * d + h * HD + sub * EPL;
#pragma unroll
      for (int e = 0; e < EPL; ++e) qr[e] = qp[e] * (a.scale * kLog2e);  // scores in log2 units
    }
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    for (int c = 0; c < nct; ++c, ++used) {
      const int c0 = (cbeg + c) * CH;
      const int nj = min(CH, t - c0);
      const int st = used % ST;
      const unsigned par = (phase >> st) & 1u;
      if (!mbar_wait(&bar[st], par, budget)) goto fail;
      // ---- scores: pass p covers rows p*RPW + rg; partial dots of the lane's
      //      EPL dimensions, then a transposed reduction over the row group
      //      (LV halving steps leave NV full dots per lane: passes idx*NV + j)
      const T_* Ks = sbuf + (st * 2) * CHE;
      float v[PASSES];
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        float kv[EPL];
        load_seg<T_, EPL>(Ks + (p * RPW + rg) * HD + sub * EPL, kv);  // rows past nj: stale, masked below
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) dot = fmaf(qr[e], kv[e], dot);
        v[p] = dot;
      }
#pragma unroll
      for (int lv = 0; lv < LV; ++lv) {
        const int o = LPR >> (lv + 1), hn = PASSES >> (lv + 1);
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < hn; ++i) {
          const float send = up ? v[i] : v[i + hn];
          const float keep = up ? v[i + hn] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
#pragma unroll
      for (int o = REP >> 1; o > 0; o >>= 1)  // lanes that share a value (LPR > PASSES)
#pragma unroll
        for (int j = 0; j < NV; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], o);
      float cmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        if ((idx * NV + j) * RPW + rg >= nj) v[j] = -INFINITY;
        cmax = fmaxf(cmax, v[j]);
      }
#pragma unroll
      for (int lv = 0; lv < LV; ++lv) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, LPR >> (lv + 1)));
#pragma unroll
      for (int o = LPR; o < 32; o <<= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
      const float mn = fmaxf(m, cmax);
      const float corr = exp2f(m - mn);  // 0 on the first chunk (m = -inf)
      m = mn;
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        v[j] = exp2f(v[j] - mn);  // masked rows: exp2(-inf) = 0
        ls += v[j];
      }
      l = l * corr + (rep0 ? ls : 0.f);  // each row counted by one lane
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] *= corr;
      if (!mbar_wait(&bar[ST + st], par, budget)) goto fail;
      const T_* Vs = sbuf + (st * 2 + 1) * CHE;
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        // P of pass p from the lane that holds it (same row group)
        int g = 0;
#pragma unroll
        for (int lv = 0; lv < LV; ++lv) g += (((p / NV) >> (LV - 1 - lv)) & 1) * (LPR >> (lv + 1));
        const float w = __shfl_sync(0xffffffffu, v[p % NV], rg * LPR + g);
        const int r = p * RPW + rg;
        if (r < nj) {
          float vv[EPL];
          load_seg<T_, EPL>(Vs + r * HD + sub * EPL, vv);
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, vv[e], acc[e]);
        }
      }
      __syncwarp();  // every lane is done with stage st
      phase ^= (1u << st);
      if (lane == 0) issue_next(st);
      __syncwarp();
    }
    // ---- end of the task: sum over the row groups and emit
    float lt = l;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, o);
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
    }
    const int wf = owner((long long)pair * nch);
    const int nseg = owner((long long)pair * nch + nch - 1) - wf + 1, sp = gw - wf;
    if (nseg == 1) {
      if (rg == 0) {
        const float inv = 1.f / lt;
#pragma unroll
        for (int e = 0; e < EPL; ++e) out[(size_t)b * d + h * HD + sub * EPL + e] = from_f32<T_>(acc[e] * inv);
      }
      continue;
    }
    {
      float* pr = a.part + ((size_t)pair * kXMaxSplits + sp) * (HD + 2);
      if (rg == 0) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) pr[2 + sub * EPL + e] = acc[e];
      }
      if (lane == 0) {
        pr[0] = m;
        pr[1] = lt;
      }
      __syncwarp();  // the warp's partial writes are ordered before lane 0's release
      int last = 0;
      if (lane == 0) last = (atom_add_acq_rel(&a.cnt[pair], 1) == nseg - 1);
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        const float* pp = a.part + (size_t)pair * kXMaxSplits * (HD + 2);
        float M = -INFINITY;
        for (int s2 = 0; s2 < nseg; ++s2) M = fmaxf(M, __ldcg(pp + (size_t)s2 * (HD + 2)));
        float L = 0.f;
        for (int s2 = 0; s2 < nseg; ++s2)
          L += __ldcg(pp + (size_t)s2 * (HD + 2) + 1) * exp2f(__ldcg(pp + (size_t)s2 * (HD + 2)) - M);
        const float inv = 1.f / L;
        for (int i = lane; i < HD; i += 32) {
          float o = 0.f;
          for (int s2 = 0; s2 < nseg; ++s2)
            o += __ldcg(pp + (size_t)s2 * (HD + 2) + 2 + i) * exp2f(__ldcg(pp + (size_t)s2 * (HD + 2)) - M);
          out[(size_t)b * d + h * HD + i] = from_f32<T_>(o * inv);
        }
        __syncwarp();
        if (lane == 0) a.cnt[pair] = 0;  // ready for the next launch
      }
    }
  }
  return;
fail:
  // a copy never completed: record it, give this warp's copies in flight a
  // bounded time to land (they write its shared memory), then leave
  if (lane == 0) {
    set_error(a.status, kErrTimeout);
    for (int s2 = 0; s2 < ST; ++s2) {
      const unsigned p2 = (phase >> s2) & 1u;
      mbar_wait(&bar[s2], p2, budget);
      mbar_wait(&bar[ST + s2], p2, budget);
    }
  }
  __syncwarp();
}

// Host-side launch: grid = resident CTAs on every SM (persistent).
template <typename T_, int HD, int ST>
inline cudaError_t launch_xattn_st(const XattnArgs& a, int n_sm, cudaStream_t st) {
  using S = XShape<T_, HD, ST>;
  static PerDevice occ_of;  // the shared-memory attribute and the occupancy are per device
  const int occ = occ_of.get([] {
    if (cudaFuncSetAttribute(dec_xattn_kernel<T_, HD, ST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)S::smem_bytes()) != cudaSuccess)
      return -1;
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, dec_xattn_kernel<T_, HD, ST>, kXThreads, S::smem_bytes()) !=
            cudaSuccess ||
        o < 1)
      o = 1;
    return o;
  });
  if (occ < 1) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_sm * occ);
  cfg.blockDim = dim3(kXThreads);
  cfg.dynamicSmemBytes = S::smem_bytes();
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dec_xattn_kernel<T_, HD, ST>, a);
}
// Ring depth by shape (measured on B300): three stages (two CTAs, eight
// warps per SM) stream long memories of heads up to 64 wide faster; two
// stages (twelve warps per SM) win for 128-wide heads and short windows.
template <typename T_, int HD>
inline cudaError_t launch_xattn_hd(const XattnArgs& a, int n_sm, cudaStream_t st) {
  if (HD <= 64 && a.t_cap >= 512) return launch_xattn_st<T_, HD, 3>(a, n_sm, st);
  return launch_xattn_st<T_, HD, 2>(a, n_sm, st);
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
