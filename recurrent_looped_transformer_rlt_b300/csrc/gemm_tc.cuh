// Tensor-core GEMM for sm_103a: C = A[M,K] * B[N,K]^T, bf16 operands, fp32
// accumulation in tensor memory (TMEM), operands staged in shared memory by
// the TMA engine (tiled tensor maps, 128-byte swizzle), MMAs issued with
// tcgen05.mma by one thread, results read back with tcgen05.ld and handed to
// an element-wise epilogue functor.
//
// Roles inside a CTA (192 threads):
//   warp 0  - TMA producer: fills a STAGES-deep ring of (A, B) k-blocks;
//   warp 1  - allocates the TMEM accumulator and issues the MMAs (one lane);
//   warps 2-5 - epilogue: TMEM -> registers -> functor (warp w reads TMEM
//             lanes 32*(w%4) .. 32*(w%4)+31, i.e. tile rows).
// Grid: (N tiles, M tiles, K splits).  When K is split over S CTAs, the S
// CTAs of a tile form a thread-block cluster (1, 1, S): each stages its
// partial tile in shared memory, and after a cluster barrier CTA z sums rows
// [z*rows/S, (z+1)*rows/S) of all S tiles through distributed shared memory,
// in split order (deterministic), and runs the epilogue on them.
//
// A is always the activation matrix (rows = tokens or sequences) and B a
// weight matrix [N][K], so one kernel serves the token-parallel encoder
// (M = B*T) and the decoder's weight-streaming projections (M = the batch of
// sequences: the A tile is mostly zero-filled rows, the CTAs split K to spread
// the weight stream over every SM).
#pragma once

#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

namespace rlt {
namespace tc {

constexpr int BM = 128;  // UMMA M (tile rows of A)
constexpr int BK = 64;   // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int UK = 16;   // K of one tcgen05.mma kind::f16
constexpr int THREADS = 192;

// BMA: rows of A copied per k-block (128, or 64 when M <= 64).  The MMA
// always reads 128 rows; with BMA = 64 rows 64..127 of its A operand fall on
// the B tile of the same stage, and the accumulator rows they produce are
// never read.
// NORMA: the A area of a stage holds the fp32 rows of the k-block (4 bytes
// per element), converted in place to the bf16 operand (its first half).
template <int BN, int STAGES, int BMA = BM, bool NORMA = false>
struct Cfg {
  static_assert(BN == 32 || BN == 64 || BN == 128 || BN == 256, "BN");
  static_assert(BMA == BM || (BMA == 64 && BN >= 64), "A rows 64..127 must stay inside the stage");
  static constexpr int A_BYTES = BMA * BK * (NORMA ? 4 : 2);
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = BN;  // fp32 accumulator: one column per output column
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + 256;
  // the epilogue stages up to BMA rows of fp32 results in the ring
  static_assert((size_t)STAGES * STAGE_BYTES >= (size_t)BMA * (BN + 4) * 4, "staging tile");
};

// ---------------------------------------------------------------------------
// PTX wrappers

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::
          "r"(smem_u32(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n" ::
          "r"(smem_u32(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(tm) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, int ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, int ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }

// Shared-memory matrix descriptor, K-major operand with 128-byte swizzle:
// rows of 128 bytes, 8-row groups 1024 bytes apart (stride byte offset),
// descriptor version 1, layout type 2 (SWIZZLE_128B).
__device__ __forceinline__ uint64_t sdesc_k_sw128(const void* p) {
  const uint64_t addr = smem_u32(p);
  uint64_t d = 0;
  d |= (addr >> 4) & 0x3FFFull;            // start address
  d |= (uint64_t)1 << 16;                  // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;        // stride byte offset
  d |= (uint64_t)1 << 46;                  // version
  d |= (uint64_t)2 << 61;                  // SWIZZLE_128B
  return d;
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
               : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// The same load without waiting for it: several may be in flight, then one
// tmem_wait_ld before their registers are read.
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;\n" ::: "memory"); }
// Named barriers of 64 threads (ids 2, 3: the two halves of the epilogue warps).
__device__ __forceinline__ void half_bar(int id) { asm volatile("bar.sync %0, 64;\n" ::"r"(id) : "memory"); }
// Makes this thread's shared-memory stores visible to the tensor cores (the
// asynchronous proxy) once the synchronisation that follows is passed.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
// ---------------------------------------------------------------------------

// Epilogues that consume column pairs (i, i + hd/2) of each head block of hd
// columns (RoPE) declare kPair, a member hd and pair(m, n, x_n, x_{n+hd/2});
// tiles then start on head boundaries (BN a multiple of hd).
template <class E, class = void>
struct IsPairEpi : std::false_type {};
template <class E>
struct IsPairEpi<E, std::void_t<decltype(E::kPair)>> : std::true_type {};
template <class E, class = void>
struct IsStore4Epi : std::false_type {};
template <class E>
struct IsStore4Epi<E, std::void_t<decltype(E::kStore4)>> : std::true_type {};
template <class E, class = void>
struct IsHOutEpi : std::false_type {};
template <class E>
struct IsHOutEpi<E, std::void_t<decltype(E::kHOut)>> : std::true_type {};
template <class E, class = void>
struct IsAdd4Epi : std::false_type {};
template <class E>
struct IsAdd4Epi<E, std::void_t<decltype(E::kAdd4)>> : std::true_type {};
// kVec4: store4(m, n, float4) takes columns n .. n + 3; kPair4: pair4(m, n,
// x1, x2) takes the pairs (n + j, n + j + hd/2), j < 4 (functors in
// gemm_simple.cuh)
template <class E, class = void>
struct IsVec4Epi : std::false_type {};
template <class E>
struct IsVec4Epi<E, std::void_t<decltype(E::kVec4)>> : std::true_type {};
template <class E, class = void>
struct IsPair4Epi : std::false_type {};
template <class E>
struct IsPair4Epi<E, std::void_t<decltype(E::kPair4)>> : std::true_type {};

// Where the A tiles come from.  k-blocks below split_kb are read through tmA
// (a 2-D map [M][K], or with pos3d a 3-D map [M][T][K] at position
// ctx->pos: one row of each sequence), the rest through tmA2 (a 2-D map whose
// column 0 is k = split_kb * BK).
struct AOperand {
  int split_kb;
  int pos3d;
  const StepCtx* ctx;
  // RMSNorm operand (kernels built with NORMA; tmA then maps the fp32 matrix
  // h [M][K]): A[m][k] = bf16(h[m][k] rs[m] g[k]), rs[m] = 1 / sqrt(sum_p
  // ss[p][m] / K + eps), ss[p][m] the sum of squares of h[m] over columns
  // 64p .. 64p + 63 (row stride ss_ld) left by the kernel that produced h;
  // K a multiple of 64
  const float* nss;
  const float* ng;
  float neps;
  int nss_ld;
};

struct SplitK {
  int splits;        // CTAs along K (= cluster size along z when > 1)
  int kb_per_split;  // k-blocks per CTA
  long long budget;  // clock cycles a wait may take before it gives up (0: kWaitBudget)
  int withhold;      // failure injection: CTA (0, 0, 0) never requests its first A tile, so the
                     // MMA's wait on that stage runs out (tests of the timeout path)
};

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// shared::cluster address of the same offset in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t mapa_u32(const void* local, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  return ra;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// float4 at the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ float4 ld_dsmem_f4(const void* local, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(ra)
               : "memory");
  return v;
}

// Epilogue on a staged fp32 tile stile[rows][BN + 4] (rows = output rows m0 +
// r, columns = output columns nb0 + c): rows [r0, r1) go through the functor,
// 128 threads (et = 0..127), consecutive threads on consecutive columns.
template <int BN, bool GLU, class Epi>
__device__ __forceinline__ void epilogue_tile(const float* stile, int r0, int r1, int m0, int nb0, int N,
                                              const Epi& epi, int et) {
  constexpr int LDT = BN + 4;
  if constexpr (GLU) {
    constexpr int HB = BN / 2;
    if constexpr (IsVec4Epi<Epi>::value) {
      // four consecutive outputs per thread (the values of the scalar path)
      constexpr int G4 = HB / 4;
      const int n = (r1 - r0) * G4;
#pragma unroll 2
      for (int i = et; i < n; i += 128) {
        const int r = r0 + i / G4, j = (i % G4) * 4;
        const float4 g = *reinterpret_cast<const float4*>(stile + r * LDT + j);
        const float4 u = *reinterpret_cast<const float4*>(stile + r * LDT + j + HB);
        const float4 o = make_float4(silu_f(g.x) * u.x, silu_f(g.y) * u.y, silu_f(g.z) * u.z, silu_f(g.w) * u.w);
        if (nb0 + j + 3 < N) {
          epi.store4(m0 + r, nb0 + j, o);
        } else {
          const float ov[4] = {o.x, o.y, o.z, o.w};
          for (int q = 0; q < 4 && nb0 + j + q < N; ++q) epi(m0 + r, nb0 + j + q, ov[q]);
        }
      }
    } else {
      const int n = (r1 - r0) * HB;
#pragma unroll 4
      for (int i = et; i < n; i += 128) {
        const int r = r0 + i / HB, j = i % HB;
        if (nb0 + j < N) epi(m0 + r, nb0 + j, silu_f(stile[r * LDT + j]) * stile[r * LDT + j + HB]);
      }
    }
  } else if constexpr (IsPairEpi<Epi>::value) {
    const int half = epi.hd >> 1;
    constexpr int HB = BN / 2;  // pairs per tile row
    bool done = false;
    if constexpr (IsPair4Epi<Epi>::value) {
      if ((half & 3) == 0) {
        // four consecutive pairs of one head per thread (tiles start on head
        // boundaries and N is a multiple of hd: a group inside N is whole)
        constexpr int G4 = HB / 4;
        const int n = (r1 - r0) * G4;
#pragma unroll 2
        for (int i = et; i < n; i += 128) {
          const int r = r0 + i / G4, pi = (i % G4) * 4;
          const int hb = pi / half, ii = pi - hb * half;
          const int c = hb * 2 * half + ii;
          if (nb0 + c < N)
            epi.pair4(m0 + r, nb0 + c, *reinterpret_cast<const float4*>(stile + r * LDT + c),
                      *reinterpret_cast<const float4*>(stile + r * LDT + c + half));
        }
        done = true;
      }
    }
    if (done) {
    } else if constexpr (128 % HB == 0) {
      // a thread keeps one pair of columns for all its rows: its per-column
      // context (position, rotation) is read once
      const int pi = et % HB, hb = pi / half, ii = pi - hb * half;
      const int c = hb * 2 * half + ii;
      if (nb0 + c < N) {
        const auto pc = epi.pair_ctx(nb0 + c);
#pragma unroll 4
        for (int r = r0 + et / HB; r < r1; r += 128 / HB)
          epi.pair(pc, m0 + r, nb0 + c, stile[r * LDT + c], stile[r * LDT + c + half]);
      }
    } else {
      const int n = (r1 - r0) * HB;
#pragma unroll 4
      for (int i = et; i < n; i += 128) {
        const int r = r0 + i / HB, pi = i % HB;
        const int hb = pi / half, ii = pi - hb * half;
        const int c = hb * 2 * half + ii;
        if (nb0 + c < N) epi.pair(epi.pair_ctx(nb0 + c), m0 + r, nb0 + c, stile[r * LDT + c], stile[r * LDT + c + half]);
      }
    }
  } else if constexpr (IsHOutEpi<Epi>::value) {
    // the residual stream: N a multiple of BN and rows 16-byte aligned
    // (checked by the host); a half-warp covers 64 consecutive columns of one
    // row (the row sums of squares are kept per 64-column group)
    constexpr int V4 = BN / 4;
    const int n = (r1 - r0) * V4;
    const HOut& o = epi.o;
    for (int i0 = et; i0 < n; i0 += 4 * 128) {
      typename Epi::Aux aux[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * 128;
        if (i < n) aux[u] = epi.load(m0 + r0 + i / V4, nb0 + (i % V4) * 4);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * 128;
        if (i >= n) continue;  // uniform per half-warp: n is a multiple of 16 (the sums are per half-warp)
        const int r = r0 + i / V4, c = (i % V4) * 4;
        const int m = m0 + r, col = nb0 + c;
        const float4 hv = epi.combine(aux[u], *reinterpret_cast<const float4*>(stile + r * LDT + c), col);
        const size_t off = (size_t)m * o.ldh + col;
        *reinterpret_cast<float4*>(o.h + off) = hv;
        if (o.s) *reinterpret_cast<float4*>(o.s + off) = hv;
        if (o.s16) {
          __nv_bfloat162 s01 = __floats2bfloat162_rn(hv.x, hv.y);
          __nv_bfloat162 s23 = __floats2bfloat162_rn(hv.z, hv.w);
          uint2 sp;
          sp.x = *reinterpret_cast<unsigned*>(&s01);
          sp.y = *reinterpret_cast<unsigned*>(&s23);
          *reinterpret_cast<uint2*>(o.s16 + off) = sp;
        }
        const float q2 = half_warp_sum(hv.x * hv.x + hv.y * hv.y + hv.z * hv.z + hv.w * hv.w);
        if ((et & 15) == 0) o.ss[(size_t)(col >> 6) * o.M + m] = q2;
      }
    }
  } else if constexpr (IsStore4Epi<Epi>::value || IsAdd4Epi<Epi>::value) {
    // 16-byte accesses, four per thread in flight (reads of the residual
    // first, then the stores); full 4-column groups only, the rest below.
    // An output whose rows are not 16-byte aligned takes the scalar path.
    constexpr int V4 = BN / 4;
    const bool vec = (epi.ldc % 4 == 0) && ((reinterpret_cast<uintptr_t>(epi.C) & 15u) == 0);
    const int nq = vec ? min(V4, (N - nb0) / 4) : 0;  // whole float4 columns inside N
    const int n = vec ? (r1 - r0) * V4 : 0;
    for (int i0 = et; i0 < n; i0 += 4 * 128) {
      float4 v[4], o[4];
      float* dst[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * 128;
        const int r = r0 + i / V4, c4 = i % V4;
        dst[u] = (i < n && c4 < nq) ? epi.C + (size_t)(m0 + r) * epi.ldc + nb0 + c4 * 4 : nullptr;
        v[u] = dst[u] ? *reinterpret_cast<const float4*>(stile + r * LDT + c4 * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (IsAdd4Epi<Epi>::value)
          o[u] = dst[u] ? *reinterpret_cast<const float4*>(dst[u]) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (!dst[u]) continue;
        if constexpr (IsAdd4Epi<Epi>::value) {
          v[u].x += o[u].x;
          v[u].y += o[u].y;
          v[u].z += o[u].z;
          v[u].w += o[u].w;
        }
        *reinterpret_cast<float4*>(dst[u]) = v[u];
      }
    }
    if (nb0 + 4 * nq < N && nq < V4) {  // ragged last columns of N (all of them without vec)
      const int c_beg = 4 * nq, w = min(BN, N - nb0) - c_beg;
      for (int i = et; i < (r1 - r0) * w; i += 128) {
        const int r = r0 + i / w, c = c_beg + i % w;
        epi(m0 + r, nb0 + c, stile[r * LDT + c]);
      }
    }
  } else if constexpr (IsVec4Epi<Epi>::value) {
    // four consecutive columns per thread; the ragged end of N one at a time
    constexpr int G4 = BN / 4;
    const int n = (r1 - r0) * G4;
#pragma unroll 2
    for (int i = et; i < n; i += 128) {
      const int r = r0 + i / G4, c = (i % G4) * 4;
      const float4 x = *reinterpret_cast<const float4*>(stile + r * LDT + c);
      if (nb0 + c + 3 < N) {
        epi.store4(m0 + r, nb0 + c, x);
      } else {
        const float xv[4] = {x.x, x.y, x.z, x.w};
        for (int q = 0; q < 4 && nb0 + c + q < N; ++q) epi(m0 + r, nb0 + c + q, xv[q]);
      }
    }
  } else {
    const int n = (r1 - r0) * BN;
#pragma unroll 4
    for (int i = et; i < n; i += 128) {
      const int r = r0 + i / BN, c = i % BN;
      if (nb0 + c < N) epi(m0 + r, nb0 + c, stile[r * LDT + c]);
    }
  }
}

// B operand: one weight matrix [N][K], or (glu) the pair W_1, W_3 [N][K]
// whose tile j holds rows j*BN/2 .. of W_1 in its first half and the same
// rows of W_3 in its second half, so that the epilogue sees gate and linear
// values of one output column in the same thread and writes
// silu(gate) * linear.
// MINB: CTAs per SM the instantiation is built for.  With MINB = 2 (a ring of
// at most ~100 KB) two CTAs share an SM, so one CTA's epilogue overlaps the
// other's main loop; such instantiations take no K split (their launches
// must pass splits = 1) and leave the split reduction out, which keeps them
// within the register budget of two CTAs.
// NORMA: A is the RMSNorm of an fp32 matrix (AOperand): the producer copies
// each k-block's fp32 rows into the stage's A area (signalled on hfull, a
// ring ahead like any A tile), the epilogue warps - idle until the
// accumulator is ready - convert them in place into the bf16 operand with
// the scaling and rounding of the stand-alone RMSNorm kernel (two groups of
// 64 threads on alternate k-blocks), and the stage's full barrier then takes
// the weight bytes from the TMA plus one arrival from the group.  The
// normalised matrix is never written to global memory.
template <int BN, int STAGES, bool GLU, class Epi, int BMA = BM, int MINB = 1, bool NORMA = false>
__global__ void __launch_bounds__(THREADS, MINB)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB3, int M, int N,
                   int K, AOperand ao, SplitK sk, Epi epi, int* status) {
  using C = Cfg<BN, STAGES, BMA, NORMA>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* accum = empty + STAGES;
  uint64_t* hfull = accum + 1;  // NORMA: the fp32 rows of a stage have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(hfull + STAGES);
  constexpr int LDT = BN + 4;
  __shared__ int s_fail;
  __shared__ float s_rs[NORMA ? BMA : 1];  // NORMA: 1 / RMS of each row of the tile
  __shared__ int s_built[2];               // NORMA: k-blocks each converting group delivered
  __shared__ int s_ok[2];                  // NORMA: a group's wait for its stage's rows succeeded

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, z = blockIdx.z;
  const int nb0 = blockIdx.x * (GLU ? BN / 2 : BN);  // first B row of the tile (per matrix)
  const int kb_total = (K + BK - 1) / BK;
  const int kb0 = z * sk.kb_per_split;
  const int nkb = max(0, min(kb_total, kb0 + sk.kb_per_split) - kb0);
  int issued = 0;  // k-blocks whose copies were requested (weights of the first `pre` requested earlier)
  const long long budget = sk.budget > 0 ? sk.budget : kWaitBudget;
  const bool withhold = sk.withhold && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;

  // bytes of a stage the full barrier counts (the weights only with NORMA)
  constexpr unsigned kTx = NORMA ? C::B_BYTES : C::STAGE_BYTES;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], NORMA ? 2 : 1);
      mbar_init(&empty[s], 1);
      if (NORMA) mbar_init(&hfull[s], 1);
    }
    mbar_init(accum, 1);
    s_fail = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmA2);
    tma_prefetch_desc(&tmB);
    if (GLU) tma_prefetch_desc(&tmB3);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // weights do not depend on the previous kernel: the first stages' weight
  // tiles are requested before waiting for it
  const int pre = min(nkb, STAGES);
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < pre; ++i) {
      unsigned char* sa = smem + i * C::STAGE_BYTES;
      const int kx = (kb0 + i) * BK;
      mbar_arrive_expect_tx(&full[i], kTx);
      if (GLU) {
        tma_load_2d(sa + C::A_BYTES, &tmB, kx, nb0, &full[i]);
        tma_load_2d(sa + C::A_BYTES + C::B_BYTES / 2, &tmB3, kx, nb0, &full[i]);
      } else {
        tma_load_2d(sa + C::A_BYTES, &tmB, kx, nb0, &full[i]);
      }
    }
  }
  pdl_wait();
  if (threadIdx.x == 0) pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      const int pos = ao.pos3d ? ao.ctx->pos : 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES && !mbar_wait(&empty[s], ((i / STAGES) - 1) & 1, budget)) {
          atomicExch(&s_fail, 1);
          break;
        }
        unsigned char* sa = smem + s * C::STAGE_BYTES;
        const int kx = (kb0 + i) * BK;
        if (i >= pre) mbar_arrive_expect_tx(&full[s], kTx);
        if (NORMA) {
          mbar_arrive_expect_tx(&hfull[s], C::A_BYTES);
          if (!(withhold && i == 0)) tma_load_2d(sa, &tmA, kx, m0, &hfull[s]);  // (injection: never sent)
        } else if (withhold && i == 0) {
          // (injection: the stage's A bytes are expected, never requested)
        } else if (kb0 + i < ao.split_kb) {
          if (ao.pos3d)
            tma_load_3d(sa, &tmA, kx, pos, m0, &full[s]);
          else
            tma_load_2d(sa, &tmA, kx, m0, &full[s]);
        } else {
          tma_load_2d(sa, &tmA2, kx - ao.split_kb * BK, m0, &full[s]);
        }
        if (i >= pre) {
          if (GLU) {
            tma_load_2d(sa + C::A_BYTES, &tmB, kx, nb0, &full[s]);
            tma_load_2d(sa + C::A_BYTES + C::B_BYTES / 2, &tmB3, kx, nb0, &full[s]);
          } else {
            tma_load_2d(sa + C::A_BYTES, &tmB, kx, nb0, &full[s]);
          }
        }
        issued = i + 1;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(&full[s], (i / STAGES) & 1, budget)) {
          atomicExch(&s_fail, 1);
          break;
        }
        tc_fence_after();
        const unsigned char* sa = smem + s * C::STAGE_BYTES;
        const uint64_t da = sdesc_k_sw128(sa), db = sdesc_k_sw128(sa + C::A_BYTES);
#pragma unroll
        for (int k = 0; k < BK / UK; ++k)  // advance 16 elements = 32 bytes (2 in descriptor units)
          mma_bf16(tmem, da + 2 * k, db + 2 * k, idesc, (i > 0 || k > 0) ? 1 : 0);
        mma_commit(&empty[s]);
      }
      mma_commit(accum);  // arrives once every issued MMA has completed (at once if none)
    }
    __syncwarp();
  } else {
    // ---- epilogue warps (128 threads)
    if constexpr (NORMA) {
      // 0. the A operand: 1 / RMS of the tile's rows, then the k-blocks
      const int et = threadIdx.x - 64;
      if (et < BMA) {
        const int m = m0 + et;
        float rs = 0.f;  // rows past M: zero rows
        if (m < M) {
          float tot = 0.f;
          for (int p = 0; p < K / 64; ++p) tot += ao.nss[(size_t)p * ao.nss_ld + m];
          rs = rsqrtf(tot / (float)K + ao.neps);
        }
        s_rs[et] = rs;
      }
      epi_bar();
      // group grp converts k-blocks grp, grp + 2, ...: the stage's fp32 rows
      // [BMA][64] (256 bytes each) become bf16 rows of 128 bytes, 16-byte
      // chunks permuted by row % 8 (the layout a 128-byte-swizzled TMA copy
      // writes), in place: 64 rows at a time, all of them read before any is
      // written (row r's output lies over input rows r/2, read already)
      const int grp = et >> 6, gt = et & 63, c16 = gt & 7;
      int built = 0;
      for (int i = grp; i < nkb; i += 2) {
        const int s = i % STAGES;
        if (gt == 0) s_ok[grp] = mbar_wait(&hfull[s], (i / STAGES) & 1, budget) ? 1 : 0;
        half_bar(2 + grp);
        if (!s_ok[grp]) {  // (the same for the whole group)
          atomicExch(&s_fail, 1);
          break;
        }
        const int col = (kb0 + i) * BK + c16 * 8;
        const float4 g0 = *reinterpret_cast<const float4*>(ao.ng + col);
        const float4 g1 = *reinterpret_cast<const float4*>(ao.ng + col + 4);
        unsigned char* sa = smem + s * C::STAGE_BYTES;
#pragma unroll 1
        for (int rb = 0; rb < BMA; rb += 64) {
          float4 hv[8][2];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int r = rb + (gt >> 3) + 8 * j;
            const float* src = reinterpret_cast<const float*>(sa + r * 256 + c16 * 32);
            hv[j][0] = *reinterpret_cast<const float4*>(src);
            hv[j][1] = *reinterpret_cast<const float4*>(src + 4);
          }
          half_bar(2 + grp);  // the group's reads of these rows are done
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int r = rb + (gt >> 3) + 8 * j;
            const float rs = s_rs[r];
            __nv_bfloat162 p0 = __floats2bfloat162_rn(hv[j][0].x * rs * g0.x, hv[j][0].y * rs * g0.y);
            __nv_bfloat162 p1 = __floats2bfloat162_rn(hv[j][0].z * rs * g0.z, hv[j][0].w * rs * g0.w);
            __nv_bfloat162 p2 = __floats2bfloat162_rn(hv[j][1].x * rs * g1.x, hv[j][1].y * rs * g1.y);
            __nv_bfloat162 p3 = __floats2bfloat162_rn(hv[j][1].z * rs * g1.z, hv[j][1].w * rs * g1.w);
            uint4 pk;
            pk.x = *reinterpret_cast<unsigned*>(&p0);
            pk.y = *reinterpret_cast<unsigned*>(&p1);
            pk.z = *reinterpret_cast<unsigned*>(&p2);
            pk.w = *reinterpret_cast<unsigned*>(&p3);
            *reinterpret_cast<uint4*>(sa + r * 128 + ((c16 ^ (r & 7)) << 4)) = pk;
          }
        }
        fence_async_smem();
        half_bar(2 + grp);
        if (gt == 0) mbar_arrive(&full[s]);
        ++built;
      }
      if (gt == 0) s_built[grp] = built;
    }
    // 1. TMEM -> shared staging tile [BM][BN + 4] fp32 (thread <-> tile row,
    //    i.e. TMEM lane); the stage ring is free once every MMA has completed.
    const int q = warp & 3;
    const int rl = q * 32 + lane;
    const bool ok = mbar_wait(accum, 0, budget) && (nkb > 0);
    if (!ok) atomicExch(&s_fail, 1);
    tc_fence_after();
    float* stile = reinterpret_cast<float*>(smem);
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    if (q * 32 < M - m0) {  // warps whose 32 TMEM lanes hold at least one output row
      constexpr int NL = BN >= 64 ? 4 : BN / 16;  // 16-column loads in flight per wait
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16 * NL) {
        uint32_t v[NL][16];
#pragma unroll
        for (int u = 0; u < NL; ++u) tmem_ld16_async(tq + c0 + 16 * u, v[u]);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < NL; ++u)
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4*>(stile + rl * LDT + c0 + 16 * u + j) =
                make_float4(__uint_as_float(v[u][j]), __uint_as_float(v[u][j + 1]), __uint_as_float(v[u][j + 2]),
                            __uint_as_float(v[u][j + 3]));
      }
    }
    epi_bar();
  }
  // ---- all threads: split-K reduction through distributed shared memory
  const int rows = min(BM, M - m0);
  int r0 = 0, r1 = rows;
  if (MINB == 1 && sk.splits > 1) {
    cluster_sync_all();  // every split's tile is staged
    r0 = (int)(((long long)rows * z) / sk.splits);
    r1 = (int)(((long long)rows * (z + 1)) / sk.splits);
    if (warp >= 2) {
      const int et = threadIdx.x - 64;
      constexpr int V4 = BN / 4;
      float* stile = reinterpret_cast<float*>(smem);
      uint32_t rbase[8];  // the staged tile in every CTA of the cluster (splits <= 8)
#pragma unroll
      for (int zz = 0; zz < 8; ++zz) rbase[zz] = zz < sk.splits ? mapa_u32(stile, (uint32_t)zz) : 0u;
      const int nv = (r1 - r0) * V4;
      // the values of every split for E elements are in flight before they
      // are summed in split order; the sums go back to rows [r0, r1) of this
      // CTA's own tile (each element read and written by one thread; the other
      // CTAs of the cluster read only their own, disjoint row ranges)
      constexpr int E = 4;
      for (int i0 = et; i0 < nv; i0 += 128 * E) {
        float4 f[E][8];
#pragma unroll
        for (int u = 0; u < E; ++u) {
          const int i = i0 + u * 128;
          if (i >= nv) continue;
          const uint32_t off = (uint32_t)(((r0 + i / V4) * LDT + (i % V4) * 4) * 4);
#pragma unroll
          for (int zz = 0; zz < 8; ++zz)
            if (zz < sk.splits) f[u][zz] = ld_cluster_f4(rbase[zz] + off);
        }
#pragma unroll
        for (int u = 0; u < E; ++u) {
          const int i = i0 + u * 128;
          if (i >= nv) continue;
          float4 acc = f[u][0];
#pragma unroll
          for (int zz = 1; zz < 8; ++zz)
            if (zz < sk.splits) {
              acc.x += f[u][zz].x;
              acc.y += f[u][zz].y;
              acc.z += f[u][zz].z;
              acc.w += f[u][zz].w;
            }
          *reinterpret_cast<float4*>(stile + (r0 + i / V4) * LDT + (i % V4) * 4) = acc;
        }
      }
    }
    cluster_arrive();  // this CTA is done reading its peers' tiles
  }
  if (warp >= 2) {
    // ---- epilogue functor on rows [r0, r1); consecutive threads take
    //      consecutive columns
    const int et = threadIdx.x - 64;
    const float* stile = reinterpret_cast<const float*>(smem);
    epi_bar();
    if (!s_fail) epilogue_tile<BN, GLU>(stile, r0, r1, m0, nb0, N, epi, et);
  }
  if (MINB == 1 && sk.splits > 1) cluster_wait();  // peers are done reading this CTA's tile before it exits
  tc_fence_before();
  __syncthreads();
  if (s_fail && threadIdx.x == 0) {
    set_error(status, kErrTimeout);
    // give the copies still in flight a bounded time to land before leaving
    // (NORMA: the fp32 rows too, and the converting group's arrival on
    // stages it never delivered is added, so that each such phase completes
    // once its weight bytes land)
    for (int i = max(0, issued - STAGES); i < issued; ++i) {
      if (NORMA) {
        mbar_wait(&hfull[i % STAGES], (i / STAGES) & 1, budget);
        if ((i >> 1) >= s_built[i & 1]) mbar_arrive(&full[i % STAGES]);
      }
      mbar_wait(&full[i % STAGES], (i / STAGES) & 1, budget);
    }
  }
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace tc
}  // namespace rlt
