// C ABI of the RLT hot path (declared in include/rlt.h).
//
// Host side: argument validation, workspace layout, the token-parallel
// encoder pass, and the decoder step, which is captured once per call as a
// CUDA graph and replayed n times (every per-step kernel reads the position
// and step index from a small context in the workspace).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

#include "../../include/rlt.h"
#include "common.cuh"
#include "gemm_simple.cuh"
#include "gemm_tc.cuh"
#include "kernels.cuh"
#include "attn_enc.cuh"
#include "attn_enc_tc.cuh"
#include "xattn.cuh"
#include "dec_fused.cuh"

using namespace rlt;

namespace {

std::atomic<uint64_t> g_launches{0};

#define RLT_CUDA_TRY(x)                         \
  do {                                          \
    cudaError_t e_ = (x);                       \
    if (e_ != cudaSuccess) return RLT_ECUDA;    \
  } while (0)

inline int launch_ok() { return cudaGetLastError() == cudaSuccess ? RLT_OK : RLT_ECUDA; }

// Launch with programmatic dependent launch: the kernel may be scheduled
// while the previous kernel of the stream is still running; it calls
// pdl_wait() before touching anything that kernel produces.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? RLT_OK : RLT_ECUDA;
}
inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline unsigned cdiv(size_t a, size_t b) { return (unsigned)((a + b - 1) / b); }

}  // namespace

// Per-launch timing of one kernel class (see rlt_timer_arm).
struct KernelTimer {
  int cls = RLT_TIMER_OFF;
  int cap = 0;                       // event pairs available
  int used = 0;                      // pairs recorded so far
  std::vector<cudaEvent_t> ev;       // [2 * cap]: start, stop, start, stop, ...
  std::vector<cudaEvent_t> ph;       // placeholders bound at capture time
  std::vector<cudaGraphNode_t> nodes;  // captured event-record nodes of the current step graph
};

struct rlt_model {
  rlt_config cfg;
  rlt_weights w;
  uint64_t version;
  cudaStream_t cap_stream;
  size_t esz;  // bytes per stored element
  int n_sm;    // SMs of the device the model was created on
  KernelTimer* timer;
  // co-resident clusters of the deep projection kernels, [config][cluster
  // size] (size 1: CTAs), measured on the device at creation
  int gemm_maxc[5][9];
  // decoder path of rlt_decode_steps (RLT_DECODE_*) and the cluster size of
  // the persistent path (0: chosen per call)
  int decode_path;
  int fused_cs;
  // one-shot failure injection of rlt_debug_withhold_copy: the kernel class
  // (RLT_KERNEL_*, 0 none) whose next standalone launch withholds a copy,
  // and the wait budget of that launch in clock cycles
  mutable int inject_kernel;
  mutable long long inject_budget;
};

// ---------------------------------------------------------------------------
// workspace layout

namespace {

struct WsLayout {
  size_t status, ctx, emit, rope;  // header
  // decoder
  size_t d_h, d_x, d_m, d_c, d_o, d_part, d_cnt, d_ss, d_s16, d_tok;
  // encoder
  size_t e_h, e_a, e_m, e_c, e_q, e_k, e_v, e_o, e_ss;
  size_t total;
};

// the status word: the part of the workspace that must start at zero
// (cleared by rlt_workspace_init)
constexpr size_t kWsHeaderBytes = 256;

WsLayout layout(const rlt_model* m, int B, int T) {
  const rlt_config& c = m->cfg;
  const size_t d = c.d_model, f = c.d_ffn, V = c.vocab, H = c.n_heads, hd = c.head_dim;
  const size_t es = m->esz;
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.status = take(sizeof(int) * 4);
  L.ctx = take(sizeof(StepCtx));
  L.emit = take(sizeof(int) * (size_t)T);
  L.rope = take(sizeof(float2) * (size_t)T * (hd / 2));
  const size_t common_end = off;
  // decoder region
  size_t cmax = std::max(std::max(3 * d, 2 * f), std::max(V, 2 * d));
  L.d_h = take(4 * (size_t)B * d);
  L.d_x = take(es * (size_t)B * std::max(2 * d, f));
  L.d_m = take(es * (size_t)B * f);
  L.d_c = take(4 * (size_t)B * cmax);
  L.d_o = take(es * (size_t)B * d);
  L.d_part = take(4 * (size_t)B * H * kXMaxSplits * (hd + 2));
  L.d_cnt = take(sizeof(int) * (size_t)B * H);
  L.d_ss = take(4 * (size_t)B * ((d + 63) / 64));
  L.d_s16 = take(es * (size_t)B * d);
  L.d_tok = take(sizeof(int) * (size_t)B);
  const size_t dec_end = off;
  // encoder region overlaps the decoder region (one call at a time per workspace)
  off = common_end;
  const size_t R = (size_t)B * T;
  L.e_h = take(4 * R * d);
  L.e_a = take(es * R * d);
  L.e_m = take(es * R * f);
  L.e_c = take(es == 4 ? 4 * R * std::max(3 * d, 2 * f) : 0);  // fp32 models: projection outputs
  L.e_q = take(es * R * d);
  L.e_k = take(es * R * d);
  L.e_v = take(es * R * d);
  L.e_o = take(es * R * d);
  L.e_ss = take(4 * R * ((d + 63) / 64));
  const size_t enc_end = off;
  L.total = std::max(dec_end, enc_end);
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// ---------------------------------------------------------------------------
// launch helpers

template <typename T_, class Epi>
int gemm(cudaStream_t st, const T_* A, int lda, GemmB gb, int M, int N, int K, Epi epi) {
  if (M <= 0 || N <= 0) return RLT_OK;
  static_assert(std::is_same<T_, float>::value, "bf16 projections run on the tensor-core kernel");
  dim3 grid(cdiv(N, simt_v0::BN), cdiv(M, simt_v0::BM));
  simt_v0::gemm_f32_kernel<Epi><<<grid, simt_v0::THREADS, 0, st>>>(A, lda, gb, M, N, K, epi);
  g_launches++;
  return launch_ok();
}

// ---------------------------------------------------------------------------
// tensor-core GEMM launcher (bf16 models)

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tiled map of a row-major bf16 matrix [rows][cols] (row pitch ld elements),
// box = 64 columns (128 bytes, swizzled) x box_rows rows; reads outside the
// matrix return zeros.
int tmap_bf16(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows) {
  auto fn = tmap_encoder();
  if (!fn) return RLT_ECUDA;
  if (((uintptr_t)base & 15u) || (ld * 2) % 16) return RLT_EINVAL;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)tc::BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? RLT_OK : RLT_ECUDA;
}
// 2-D map of an fp32 matrix [rows][cols] (row stride ld elements), box = 64
// columns x box_rows rows, no swizzle (rows of 256 bytes in shared memory).
int tmap_f32(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows) {
  auto fn = tmap_encoder();
  if (!fn) return RLT_ECUDA;
  if (((uintptr_t)base & 15u) || (ld * 4) % 16) return RLT_EINVAL;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 4};
  cuuint32_t box[2] = {(cuuint32_t)tc::BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? RLT_OK : RLT_ECUDA;
}
// 3-D map of a bf16 tensor [rows][T][cols] (rows of T positions), box = 64
// columns x 1 position x box_rows rows: one position of every row.
int tmap_bf16_3d(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t T, uint64_t cols, uint32_t box_rows) {
  auto fn = tmap_encoder();
  if (!fn) return RLT_ECUDA;
  if (((uintptr_t)base & 15u) || (cols * 2) % 16) return RLT_EINVAL;
  cuuint64_t dims[3] = {cols, T, rows};
  cuuint64_t strides[2] = {cols * 2, T * cols * 2};
  cuuint32_t box[3] = {(cuuint32_t)tc::BK, 1, box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? RLT_OK : RLT_ECUDA;
}

// 3-D map of a bf16 tensor [d2][d1][d0] (d0 contiguous), box = 64 x box1 x 1
// (128-byte swizzle): a [box1][64] tile of one d2 slice.
int tmap_bf16_3d_tile(CUtensorMap* tm, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box1) {
  auto fn = tmap_encoder();
  if (!fn) return RLT_ECUDA;
  if (((uintptr_t)base & 15u) || (d0 * 2) % 16) return RLT_EINVAL;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d1 * d0 * 2};
  cuuint32_t box[3] = {64, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? RLT_OK : RLT_ECUDA;
}

// Launch context of the tensor-core GEMMs.
struct TcScratch {
  int n_sm;
  int* status;
  const int (*maxc)[9];  // rlt_model::gemm_maxc
  long long budget = 0;  // wait budget of the launch (0: the kernels' default)
  int withhold = 0;      // failure injection (rlt_debug_withhold_copy)
};

// The A operand of a projection: A [M][lda] for k < split (all of K when
// A2 == nullptr), A2 [M][lda2] for k >= split (column 0 = k split); with T3 > 0
// the first part is a [M][T3][lda] tensor read at the step's position ctx->pos.
struct AArg {
  const bf16* A;
  int lda;
  const bf16* A2 = nullptr;
  int lda2 = 0;
  int split = 0;
  int T3 = 0;
  const StepCtx* ctx = nullptr;
  // A = bf16(RMSNorm(nh) * ng) built inside the projection (nh [M][K] fp32,
  // nss its per-64-column sums of squares [K/64][M]); A above is then unused
  const float* nh = nullptr;
  const float* nss = nullptr;
  const float* ng = nullptr;
  float neps = 0.f;
};

template <int BN, int STAGES, bool GLU, class Epi, int BMA = tc::BM, int MINB = 1, bool NORMA = false>
int gemm_tc_launch(cudaStream_t st, const AArg& a, int M, int K, const bf16* B, const bf16* B3, int ldb, int N,
                   Epi epi, const TcScratch& sc, int split_req = 0) {
  using C = tc::Cfg<BN, STAGES, BMA, NORMA>;
  static_assert(MINB == 1 || MINB * (C::SMEM + 1024) <= 228 * 1024, "CTAs per SM");
  static_assert(!NORMA || MINB == 1, "the RMSNorm operand is built in single-CTA instantiations");
  static PerDevice attr;  // the shared-memory attribute is per device
  if (attr.get([] {
        return cudaFuncSetAttribute(tc::gemm_tc_kernel<BN, STAGES, GLU, Epi, BMA, MINB, NORMA>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM) == cudaSuccess
                   ? 1
                   : -1;
      }) != 1)
    return RLT_ECUDA;
  if (M > BMA && BMA != tc::BM) return RLT_EINVAL;
  if (NORMA != (a.nh != nullptr) || (NORMA && (M > BMA || K % 64 || a.A2 || a.T3 > 0))) return RLT_EINVAL;
  const int nout = GLU ? BN / 2 : BN;
  const int tiles_n = (N + nout - 1) / nout, tiles_m = (M + tc::BM - 1) / tc::BM;
  const int kb = (K + tc::BK - 1) / tc::BK;
  // split K over a cluster of CTAs per tile when there are few tiles (the
  // caller's split when given).  Sizes from measurements of the
  // weight-streaming shapes on B300: clusters of 8 fit on 120 of the 148 SMs
  // only (15 at a time), clusters of 2 on all; about 100 CTAs already
  // saturate HBM with 3-stage rings.
  const int tiles = tiles_n * tiles_m;
  int splits = 1;
  if (split_req > 0)
    splits = split_req;
  else if (tiles < 12)
    splits = 8;
  else if (tiles < 32)
    splits = 6;
  else if (tiles < 128)
    splits = 2;
  splits = std::max(1, std::min(splits, kb));
  if (MINB > 1) splits = 1;  // (instantiations for two CTAs per SM have no split reduction)
  const int kbps = (kb + splits - 1) / splits;
  splits = (kb + kbps - 1) / kbps;
  if (a.A2 && (a.split % tc::BK)) return RLT_EINVAL;
  CUtensorMap ta, ta2, tb, tb3;
  int rc;
  const int k1 = a.A2 ? a.split : K;
  if (NORMA) {
    if ((rc = tmap_f32(&ta, a.nh, M, K, K, BMA))) return rc;
  } else if (a.T3 > 0) {
    if ((rc = tmap_bf16_3d(&ta, a.A, M, a.T3, a.lda, BMA))) return rc;
  } else if ((rc = tmap_bf16(&ta, a.A, M, k1, a.lda, BMA))) {
    return rc;
  }
  if ((rc = tmap_bf16(&ta2, a.A2 ? a.A2 : a.A, M, a.A2 ? K - a.split : k1, a.A2 ? a.lda2 : a.lda, BMA))) return rc;
  if ((rc = tmap_bf16(&tb, B, N, K, ldb, GLU ? BN / 2 : BN))) return rc;
  if ((rc = tmap_bf16(&tb3, GLU ? B3 : B, N, K, ldb, GLU ? BN / 2 : BN))) return rc;
  tc::AOperand ao{a.A2 ? a.split / tc::BK : kb, a.T3 > 0 ? 1 : 0, a.ctx, a.nss, a.ng, a.neps, M};
  tc::SplitK sk{splits, kbps, sc.budget, sc.withhold};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles_n, tiles_m, splits);
  cfg.blockDim = dim3(tc::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = 1;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = splits;
  cfg.attrs = at;
  cfg.numAttrs = splits > 1 ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, tc::gemm_tc_kernel<BN, STAGES, GLU, Epi, BMA, MINB, NORMA>, ta, ta2, tb, tb3, M, N, K, ao, sk,
                         epi, sc.status) != cudaSuccess)
    return RLT_ECUDA;
  g_launches++;
  return launch_ok();
}

// C = A[M,K] B[N,K]^T with the epilogue functor; tiles sized for the shape.
template <class Epi>
int gemm_bf16_tc(cudaStream_t st, const AArg& a, int M, int K, const bf16* B, int ldb, int N, Epi epi,
                 const TcScratch& sc) {
  if (M <= 0 || N <= 0) return RLT_OK;
  if (M <= tc::BM) return gemm_tc_launch<128, 3, false>(st, a, M, K, B, nullptr, ldb, N, epi, sc);
  return gemm_tc_launch<128, 3, false, Epi, tc::BM, 2>(st, a, M, K, B, nullptr, ldb, N, epi, sc);
}
template <class Epi>
int gemm_bf16_tc(cudaStream_t st, const bf16* A, int lda, int M, int K, const bf16* B, int ldb, int N, Epi epi,
                 const TcScratch& sc) {
  AArg a;
  a.A = A;
  a.lda = lda;
  return gemm_bf16_tc(st, a, M, K, B, ldb, N, epi, sc);
}
// Weight streaming at up to 128 rows (decoder step, rlt_linear): one CTA per
// SM whose shared memory is one deep ring of k-blocks, so that each SM keeps
// 100-160 KB of weights in flight.  Configurations (BN, rows of A per copy):
//   0: (128, 64)  8 stages   1: (256, 64)  5 stages
//   2: (128, 128) 6 stages   3: (256, 128) 4 stages
//   4: (64, 64)   8 stages (not for RoPE tiles of heads wider than 64)
// (NORMA: the A area of a stage holds fp32 rows, twice the bf16 bytes)
template <int BN, int BMA, bool NORMA = false>
constexpr int deep_stages() {
  return std::min(8, (200 * 1024) / (((NORMA ? 2 : 1) * BMA + BN) * tc::BK * 2));
}
struct DeepPlan {
  int cfg, splits;
};
// Whether a projection of M rows can take its RMSNorm operand from the fp32
// rows directly (AArg::nh): the deep kernels (M <= 128), K in whole
// 64-column sum-of-squares groups.
inline bool norm_fusable(int M, int K) { return M > 0 && M <= tc::BM && K % 64 == 0; }
// The tile width and K split with the most CTAs that are all resident at
// once (one wave), fewer splits on ties; the widest tiles without a split
// when no choice fits in one wave.  More CTAs stream more weight bytes at
// once and share the epilogue; a split's partial sums cost a cluster barrier
// and a pull through distributed shared memory (~2-3 us, measured), which
// fewer, longer CTAs lose more than that to streaming and epilogue time.
// 64-wide tiles are considered only when the wider ones leave more than half
// of the SMs idle (narrow projections of small models: measured 11 % faster
// per step at d = 256; at d = 2048, where 128-wide tiles already take 96 or
// more CTAs, they were 2-3 % slower).
DeepPlan deep_plan(const TcScratch& sc, int M, int N, int K, bool glu, bool allow64) {
  const int base = (M <= 64) ? 0 : 2;
  const int kb = (K + tc::BK - 1) / tc::BK;
  DeepPlan best{base + 1, 1};
  int best_ctas = 0, best_s = 0;
  const int order[3] = {0, 1, -1};  // 128 wide, 256 wide, then 64 wide
  for (const int j : order) {
    if (j < 0 && !(base == 0 && allow64 && 2 * best_ctas < sc.n_sm)) break;
    const int cfg = j < 0 ? 4 : base + j;
    const int bn = j < 0 ? 64 : j ? 256 : 128, nout = glu ? bn / 2 : bn;
    const long long tiles = (N + nout - 1) / nout;
    // (256, 128) tiles have no split (their partial tiles are the largest)
    const int smax = (cfg == 3) ? 1 : std::min(8, kb);
    for (int s = 1; s <= smax; ++s) {
      const int kbps = (kb + s - 1) / s;
      if ((kb + kbps - 1) / kbps != s) continue;  // every split non-empty
      const long long ctas = tiles * s;
      if (ctas > (long long)sc.maxc[cfg][s] * s) continue;
      if (ctas > best_ctas || (ctas == best_ctas && s < best_s)) {
        best = {cfg, s};
        best_ctas = (int)ctas;
        best_s = s;
      }
    }
  }
  return best;
}
template <int BN, int BMA, bool GLU, bool NORMA, class Epi>
int deep_launch(cudaStream_t st, const AArg& x, int M, int K, const bf16* W, const bf16* W3, int ldw, int N, Epi epi,
                const TcScratch& sc, int splits) {
  return gemm_tc_launch<BN, deep_stages<BN, BMA, NORMA>(), GLU, Epi, BMA, 1, NORMA>(st, x, M, K, W, W3, ldw, N, epi,
                                                                                     sc, splits);
}
template <bool GLU, class Epi, bool NORMA = false>
int proj_deep(cudaStream_t st, const AArg& x, int M, int K, const bf16* W, const bf16* W3, int ldw, int N, Epi epi,
              const TcScratch& sc) {
  bool allow64 = true;  // RoPE pair tiles start on head boundaries: 64-wide tiles only for heads of <= 64
  if constexpr (tc::IsPairEpi<Epi>::value) allow64 = epi.hd <= 64;
  const DeepPlan p = deep_plan(sc, M, N, K, GLU, allow64);
  switch (p.cfg) {
    case 4: return deep_launch<64, 64, GLU, NORMA>(st, x, M, K, W, W3, ldw, N, epi, sc, p.splits);
    case 0: return deep_launch<128, 64, GLU, NORMA>(st, x, M, K, W, W3, ldw, N, epi, sc, p.splits);
    case 1: return deep_launch<256, 64, GLU, NORMA>(st, x, M, K, W, W3, ldw, N, epi, sc, p.splits);
    case 2: return deep_launch<128, 128, GLU, NORMA>(st, x, M, K, W, W3, ldw, N, epi, sc, p.splits);
    default: return deep_launch<256, 128, GLU, NORMA>(st, x, M, K, W, W3, ldw, N, epi, sc, p.splits);
  }
}
// Co-resident clusters of each deep configuration for cluster sizes 1..8.
template <int BN, int BMA>
int deep_occupancy(int n_sm, int* maxc) {
  using C = tc::Cfg<BN, deep_stages<BN, BMA>(), BMA>;
  auto kern = tc::gemm_tc_kernel<BN, deep_stages<BN, BMA>(), false, EpiStoreF32, BMA>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM) != cudaSuccess)
    return RLT_ECUDA;
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, tc::THREADS, C::SMEM) != cudaSuccess) return RLT_ECUDA;
  maxc[0] = 0;
  maxc[1] = nb * n_sm;
  for (int s = 2; s <= 8; ++s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, s);
    cfg.blockDim = dim3(tc::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess) return RLT_ECUDA;
    maxc[s] = nc;
  }
  return RLT_OK;
}
int deep_occupancy_all(rlt_model* m) {
  int rc;
  if ((rc = deep_occupancy<128, 64>(m->n_sm, m->gemm_maxc[0]))) return rc;
  if ((rc = deep_occupancy<256, 64>(m->n_sm, m->gemm_maxc[1]))) return rc;
  if ((rc = deep_occupancy<128, 128>(m->n_sm, m->gemm_maxc[2]))) return rc;
  if ((rc = deep_occupancy<256, 128>(m->n_sm, m->gemm_maxc[3]))) return rc;
  return deep_occupancy<64, 64>(m->n_sm, m->gemm_maxc[4]);
}
// Projection of a batch of sequences (decoder step, rlt_linear): the deep
// weight-streaming kernels up to 128 rows, 4 stages of 256-wide tiles beyond.
// An RMSNorm operand (x.nh) is built inside the deep kernels (norm_fusable).
template <bool GLU, class Epi>
int proj_bf16(cudaStream_t st, const AArg& x, int M, int K, const bf16* W, const bf16* W3, int ldw, int N, Epi epi,
              const TcScratch& sc) {
  if (M <= 0 || N <= 0) return RLT_OK;
  if (x.nh) {
    if (!norm_fusable(M, K)) return RLT_EINVAL;
    return proj_deep<GLU, Epi, true>(st, x, M, K, W, W3, ldw, N, epi, sc);
  }
  if (M <= tc::BM) return proj_deep<GLU>(st, x, M, K, W, W3, ldw, N, epi, sc);
  // hundreds of sequences (tensor-core bound): 128 x 128 tiles two per SM, or
  // 128 x 64 tiles where the wider ones would leave SMs without a tile
  // (d-wide outputs of d = 1024 at M = 1024: 64 tiles of 128 columns)
  bool narrow = (long long)((M + tc::BM - 1) / tc::BM) * ((N + (GLU ? 63 : 127)) / (GLU ? 64 : 128)) < sc.n_sm;
  if constexpr (tc::IsPairEpi<Epi>::value) narrow = narrow && epi.hd <= 64;  // RoPE tiles start on head boundaries
  if (narrow) return gemm_tc_launch<64, 4, GLU, Epi, tc::BM, 2>(st, x, M, K, W, W3, ldw, N, epi, sc);
  return gemm_tc_launch<128, 3, GLU, Epi, tc::BM, 2>(st, x, M, K, W, W3, ldw, N, epi, sc);
}

// out[m][j] = silu(A W_1^T)[m][j] * (A W_3^T)[m][j], j < N (= d_ffn).
template <class Epi>
int gemm_bf16_tc_glu(cudaStream_t st, const bf16* A, int lda, int M, int K, const bf16* W1, const bf16* W3, int ldb,
                     int N, Epi epi, const TcScratch& sc) {
  if (M <= 0 || N <= 0) return RLT_OK;
  AArg a;
  a.A = A;
  a.lda = lda;
  if (M <= tc::BM) return gemm_tc_launch<128, 3, true>(st, a, M, K, W1, W3, ldb, N, epi, sc);
  return gemm_tc_launch<128, 3, true, Epi, tc::BM, 2>(st, a, M, K, W1, W3, ldb, N, epi, sc);
}

TcScratch tc_scratch(const rlt_model* m, void* ws, const WsLayout& Lw) {
  TcScratch sc;
  sc.n_sm = m->n_sm;
  sc.maxc = m->gemm_maxc;
  sc.status = at<int>(ws, Lw.status);
  return sc;
}

// y = A W^T with the epilogue: tensor cores for bf16 models, FFMA for fp32.
template <typename T_, class Epi>
int proj(cudaStream_t st, const T_* A, int lda, int M, int K, const void* W, int ldw, int N, Epi epi,
         const TcScratch& sc) {
  if constexpr (std::is_same<T_, bf16>::value)
    return gemm_bf16_tc(st, A, lda, M, K, static_cast<const bf16*>(W), ldw, N, epi, sc);
  else
    return gemm<T_>(st, A, lda, GemmB{W, W, N, ldw}, M, N, K, epi);
}

template <typename T_>
int rmsnorm(cudaStream_t st, const float* x, const float* g, T_* y, int rows, int d, int ldy, float eps) {
  rmsnorm_kernel<T_><<<cdiv((size_t)rows * 32, 256), 256, 0, st>>>(x, g, y, rows, d, ldy, eps);
  g_launches++;
  return launch_ok();
}

template <typename T_>
const T_* wl(const void* base, int l, size_t per_layer) {
  return static_cast<const T_*>(base) + (size_t)l * per_layer;
}

template <typename T_>
void set_attrs() {
  cudaFuncSetAttribute(enc_attn_simt_kernel<T_>, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024);
  cudaFuncSetAttribute(head_reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
}
void ensure_attrs() {  // once per device: function attributes are per device
  static PerDevice done;
  done.get([] {
    set_attrs<float>();
    set_attrs<bf16>();
    return 1;
  });
}

// ---------------------------------------------------------------------------
// encoder

// out[m][j] = silu(A W_1^T)[m][j] * (A W_3^T)[m][j] in storage precision (j < f);
// fp32 models go through an fp32 buffer C [M][2f] and a separate kernel.
template <typename T_>
int swiglu_proj(cudaStream_t st, const T_* A, int lda, int M, int K, const T_* W1, const T_* W3, int f, T_* out,
                float* C, const TcScratch& sc) {
  if constexpr (std::is_same<T_, bf16>::value) {
    return gemm_bf16_tc_glu(st, A, lda, M, K, W1, W3, K, f, EpiStoreT<bf16>{out, f}, sc);
  } else {
    int rc = gemm<T_>(st, A, lda, GemmB{W1, W3, f, K}, M, 2 * f, K, EpiStoreF32{C, 2 * f});
    if (rc) return rc;
    swiglu_kernel<T_><<<cdiv((size_t)M * f, 256), 256, 0, st>>>(C, out, M, f);
    g_launches++;
    return launch_ok();
  }
}

// x = bf16(RMSNorm(h) * g) for bf16 models, from the producer's per-64-column
// sums of squares.
int norm_rows(cudaStream_t st, const float* h, const float* ss, const float* g, bf16* x, int rows, int d, float eps) {
  g_launches++;
  return launch_pdl(norm_rows_kernel, dim3(rows), dim3(d / 4), 0, st, h, ss, g, x, rows, d, eps);
}

// Causal self-attention of the bf16 encoder: the flash kernel on the tensor
// cores (head_dim 16..128), the CUDA-core kernel below that.
template <int HD>
int enc_flash_launch(cudaStream_t st, const bf16* q, const bf16* k, const bf16* v, bf16* o, int B, int T, int H) {
  static PerDevice attr;  // the shared-memory attribute is per device
  if (attr.get([] {
        return cudaFuncSetAttribute(fa::enc_flash_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)fa::smem_bytes<HD>()) == cudaSuccess
                   ? 1
                   : -1;
      }) != 1)
    return RLT_ECUDA;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  fa::enc_flash_kernel<HD><<<dim3(cdiv(T, fa::BQ), H, B), fa::THREADS, fa::smem_bytes<HD>(), st>>>(q, k, v, o, T, H,
                                                                                                   scale_log2);
  g_launches++;
  return launch_ok();
}
// The tcgen05 encoder attention (attn_enc_tc.cuh): V transposed into vt
// (B*H*hd*T elements of scratch), then one launch.
template <int HD>
int enc_attn_tc_launch(cudaStream_t st, const bf16* q, const bf16* k, const bf16* v, bf16* vt, bf16* o, int B,
                       int T, int H, int* status) {
  using Lo = fat::Lay<HD>;
  static PerDevice attr;  // the shared-memory attribute is per device
  if (attr.get([] {
        return cudaFuncSetAttribute(fat::enc_attn_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)Lo::SMEM) == cudaSuccess
                   ? 1
                   : -1;
      }) != 1)
    return RLT_ECUDA;
  const uint64_t BH = (uint64_t)B * H;
  fat::vt_transpose_kernel<<<dim3(cdiv(T, 32), HD / 32, (unsigned)BH), dim3(32, 8), 0, st>>>(v, vt, T, HD);
  g_launches++;
  int rc;
  if ((rc = launch_ok())) return rc;
  CUtensorMap tq, tk, tv;
  if ((rc = tmap_bf16_3d_tile(&tq, q, HD, T, BH, fat::BQ)) || (rc = tmap_bf16_3d_tile(&tk, k, HD, T, BH, fat::BKV)) ||
      (rc = tmap_bf16_3d_tile(&tv, vt, T, HD, BH, HD)))
    return rc;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  fat::enc_attn_tc_kernel<HD><<<dim3(cdiv(T, fat::BQ), H, B), fat::THREADS, Lo::SMEM, st>>>(tq, tk, tv, o, T, H,
                                                                                             scale_log2, status);
  g_launches++;
  return launch_ok();
}

// Causal self-attention of the bf16 encoder.  Head widths 64 and 128 with T a
// multiple of 8 (the transposed V's rows must be 16-byte multiples for the
// tensor maps) run on the tcgen05 kernel, which takes vt (B*H*hd*T elements
// of scratch); the others on the warp-level MMA kernel.
int enc_attention_bf16(cudaStream_t st, const bf16* q, const bf16* k, const bf16* v, bf16* o, int B, int T, int H,
                       int hd, bf16* vt, int* status) {
  if (vt && T % 8 == 0) {
    if (hd == 128) return enc_attn_tc_launch<128>(st, q, k, v, vt, o, B, T, H, status);
    if (hd == 64) return enc_attn_tc_launch<64>(st, q, k, v, vt, o, B, T, H, status);
  }
  switch (hd) {
    case 16: return enc_flash_launch<16>(st, q, k, v, o, B, T, H);
    case 32: return enc_flash_launch<32>(st, q, k, v, o, B, T, H);
    case 64: return enc_flash_launch<64>(st, q, k, v, o, B, T, H);
    case 128: return enc_flash_launch<128>(st, q, k, v, o, B, T, H);
    default: {
      const size_t att_smem = sizeof(float) * (32 * hd + 32 * (hd + 1) + 32 * hd);
      enc_attn_simt_kernel<bf16><<<dim3(cdiv(T, 32), H, B), 256, att_smem, st>>>(q, k, v, o, T, H, hd,
                                                                                 1.0f / sqrtf((float)hd));
      g_launches++;
      return launch_ok();
    }
  }
}

// bf16 encoder: projections on the tensor cores with the RMSNorms deferred
// into them (the residual producers write x = bf16(h * g_next) and row sums of
// squares; the consumers scale their output rows), RoPE and the head-major
// q/k/v layout in the QKV epilogue, SwiGLU in the W_1/W_3 epilogue.
// Token-parallel encoder of bf16 models.  e [B][T_stride][d] and mem
// [G][2][B][H][T_stride][hd] receive positions 0..T-1 (T_stride >= T); with
// enc_kv [L][2][B][H][T_stride][hd], every layer's keys (after RoPE) and
// values are kept for incremental encoding.
int encode_bf16(const rlt_model* m, const int32_t* tok, int B, int T, bf16* e, bf16* mem, void* ws,
                cudaStream_t st, int T_stride = 0, bf16* enc_kv = nullptr) {
  if (T_stride <= 0) T_stride = T;
  const rlt_config& c = m->cfg;
  const rlt_weights& w = m->w;
  const int d = c.d_model, f = c.d_ffn, H = c.n_heads, hd = c.head_dim, L = c.n_layers, G = c.mem_groups;
  const int R = B * T;
  WsLayout Lw = layout(m, B, T);
  int* status = at<int>(ws, Lw.status);
  float2* tab = at<float2>(ws, Lw.rope);
  float* h = at<float>(ws, Lw.e_h);
  bf16* x = at<bf16>(ws, Lw.e_a);
  bf16* xm = at<bf16>(ws, Lw.e_m);
  bf16* q = at<bf16>(ws, Lw.e_q);
  bf16* k = at<bf16>(ws, Lw.e_k);
  bf16* v = at<bf16>(ws, Lw.e_v);
  bf16* o = at<bf16>(ws, Lw.e_o);
  float* ss = at<float>(ws, Lw.e_ss);
  const TcScratch sc = tc_scratch(m, ws, Lw);
  int rc;
  // memory group g (keys and values, [B][H][T_stride][hd] each) from the source rows src [R][d]
  const size_t plane = (size_t)B * H * T_stride * hd;
  auto mem_proj_bf16 = [&](cudaStream_t s_, const bf16* src, int g) -> int {
    const bf16* WK = wl<bf16>(w.W_K, g, (size_t)d * d);
    const bf16* WV = wl<bf16>(w.W_V, g, (size_t)d * d);
    int r;
    if ((r = gemm_bf16_tc(s_, src, d, R, d, WK, d, d, EpiMemScatter<bf16>{mem + (2 * g) * plane, T, H, hd, T_stride},
                          sc)))
      return r;
    return gemm_bf16_tc(s_, src, d, R, d, WV, d, d,
                        EpiMemScatter<bf16>{mem + (2 * g + 1) * plane, T, H, hd, T_stride}, sc);
  };
  // e rows go straight to e when they are contiguous, else through x and a copy
  bf16* e_rows = (T_stride == T) ? e : x;
  rope_table_kernel<<<cdiv((size_t)T * (hd / 2), 256), 256, 0, st>>>(tab, 0, T, hd / 2, (double)c.rope_theta);
  g_launches++;
  embed_norm_kernel<<<R, d / 4, 0, st>>>(tok, static_cast<const bf16*>(w.tok_emb), h, x, w.enc_attn_norm, R, d,
                                         c.vocab, c.rms_eps, status);
  g_launches++;
  if ((rc = launch_ok())) return rc;
  for (int l = 0; l < L; ++l) {
    const bf16* Wqkv = wl<bf16>(w.W_qkv, l, (size_t)3 * d * d);
    if ((rc = gemm_bf16_tc(st, x, d, R, d, Wqkv, d, 3 * d, EpiEncQKVRope<bf16>{q, k, v, tab, d, H, hd, T}, sc)))
      return rc;
    if (enc_kv) {  // keep this layer's keys and values: [B*H] rows of T positions into T_stride
      const size_t kvp = (size_t)B * H * T_stride * hd, row = (size_t)T * hd * 2;
      RLT_CUDA_TRY(cudaMemcpy2DAsync(enc_kv + (2 * l) * kvp, (size_t)T_stride * hd * 2, k, row, row,
                                     (size_t)B * H, cudaMemcpyDeviceToDevice, st));
      RLT_CUDA_TRY(cudaMemcpy2DAsync(enc_kv + (2 * l + 1) * kvp, (size_t)T_stride * hd * 2, v, row, row,
                                     (size_t)B * H, cudaMemcpyDeviceToDevice, st));
    }
    // V transposed into the SwiGLU buffer (free until this layer's W_1/W_3;
    // it holds R x f >= R x d elements when f >= d)
    if ((rc = enc_attention_bf16(st, q, k, v, o, B, T, H, hd, f >= d ? xm : nullptr, sc.status))) return rc;
    const bf16* WO = wl<bf16>(w.W_O, l, (size_t)d * d);
    if ((rc = gemm_bf16_tc(st, o, d, R, d, WO, d, d, EpiResidual{HOut{h, d, nullptr, nullptr, ss, R}}, sc))) return rc;
    if ((rc = norm_rows(st, h, ss, w.enc_ffn_norm + (size_t)l * d, x, R, d, c.rms_eps))) return rc;
    const bf16* W1 = wl<bf16>(w.W_1, l, (size_t)f * d);
    const bf16* W3 = wl<bf16>(w.W_3, l, (size_t)f * d);
    if ((rc = gemm_bf16_tc_glu(st, x, d, R, d, W1, W3, d, f, EpiStoreT<bf16>{xm, f}, sc))) return rc;
    const bf16* W2 = wl<bf16>(w.W_2, l, (size_t)d * f);
    if ((rc = gemm_bf16_tc(st, xm, f, R, f, W2, f, d, EpiResidual{HOut{h, d, nullptr, nullptr, ss, R}}, sc))) return rc;
    // per-layer memory: group l from RMSNorm_e of this layer's output (the
    // SwiGLU buffer is free until the next layer's W_1/W_3 projection)
    if (c.mem_source == RLT_MEM_PER_LAYER && l + 1 < L) {
      if ((rc = norm_rows(st, h, ss, w.enc_norm, xm, R, d, c.rms_eps))) return rc;
      if ((rc = mem_proj_bf16(st, xm, l))) return rc;
    }
    // RMSNorm of the next layer's attention, or the final norm producing e
    if ((rc = norm_rows(st, h, ss, (l + 1 < L) ? w.enc_attn_norm + (size_t)(l + 1) * d : w.enc_norm,
                        (l + 1 < L) ? x : e_rows, R, d, c.rms_eps)))
      return rc;
  }
  if (e_rows != e)
    RLT_CUDA_TRY(cudaMemcpy2DAsync(e, (size_t)T_stride * d * 2, e_rows, (size_t)T * d * 2, (size_t)T * d * 2, B,
                                   cudaMemcpyDeviceToDevice, st));
  if (c.mem_source == RLT_MEM_PER_LAYER) return mem_proj_bf16(st, e_rows, L - 1);  // the last layer's source is e
  for (int g = 0; g < G; ++g)
    if ((rc = mem_proj_bf16(st, e_rows, g))) return rc;
  return RLT_OK;
}

template <typename T_>
int encode_impl(const rlt_model* m, const int32_t* tok, int B, int T, T_* e, T_* mem, void* ws, cudaStream_t st) {
  const rlt_config& c = m->cfg;
  const rlt_weights& w = m->w;
  const int d = c.d_model, f = c.d_ffn, H = c.n_heads, hd = c.head_dim, L = c.n_layers, G = c.mem_groups;
  const int R = B * T;
  WsLayout Lw = layout(m, B, T);
  int* status = at<int>(ws, Lw.status);
  float2* tab = at<float2>(ws, Lw.rope);
  float* h = at<float>(ws, Lw.e_h);
  T_* a = at<T_>(ws, Lw.e_a);
  T_* am = at<T_>(ws, Lw.e_m);
  float* C = at<float>(ws, Lw.e_c);
  T_* q = at<T_>(ws, Lw.e_q);
  T_* k = at<T_>(ws, Lw.e_k);
  T_* v = at<T_>(ws, Lw.e_v);
  T_* o = at<T_>(ws, Lw.e_o);
  const TcScratch sc = tc_scratch(m, ws, Lw);
  int rc;
  rope_table_kernel<<<cdiv((size_t)T * (hd / 2), 256), 256, 0, st>>>(tab, 0, T, hd / 2, (double)c.rope_theta);
  g_launches++;
  embed_kernel<T_><<<R, 128, 0, st>>>(tok, static_cast<const T_*>(w.tok_emb), h, R, d, c.vocab, status);
  g_launches++;
  if ((rc = launch_ok())) return rc;
  const float scale = 1.0f / sqrtf((float)hd);
  const size_t att_smem = sizeof(float) * (32 * hd + 32 * (hd + 1) + 32 * hd);
  // memory group g (keys and values, [B][H][T][hd] each) from the source rows src [R][d]
  const size_t plane = (size_t)B * H * T * hd;
  auto mem_proj = [&](const T_* src, int g) -> int {
    const T_* WK = wl<T_>(w.W_K, g, (size_t)d * d);
    const T_* WV = wl<T_>(w.W_V, g, (size_t)d * d);
    int r;
    if ((r = proj<T_>(st, src, d, R, d, WK, d, d, EpiMemScatter<T_>{mem + (2 * g) * plane, T, H, hd}, sc))) return r;
    return proj<T_>(st, src, d, R, d, WV, d, d, EpiMemScatter<T_>{mem + (2 * g + 1) * plane, T, H, hd}, sc);
  };
  for (int l = 0; l < L; ++l) {
    if ((rc = rmsnorm<T_>(st, h, w.enc_attn_norm + (size_t)l * d, a, R, d, d, c.rms_eps))) return rc;
    const T_* Wqkv = wl<T_>(w.W_qkv, l, (size_t)3 * d * d);
    if ((rc = proj<T_>(st, a, d, R, d, Wqkv, d, 3 * d, EpiStoreF32{C, 3 * d}, sc))) return rc;
    rope_split_kernel<T_><<<cdiv((size_t)R * H * (hd / 2), 256), 256, 0, st>>>(C, q, k, v, tab, B, T, H, hd);
    g_launches++;
    enc_attn_simt_kernel<T_><<<dim3(cdiv(T, 32), H, B), 256, att_smem, st>>>(q, k, v, o, T, H, hd, scale);
    g_launches++;
    if ((rc = launch_ok())) return rc;
    const T_* WO = wl<T_>(w.W_O, l, (size_t)d * d);
    if ((rc = proj<T_>(st, o, d, R, d, WO, d, d, EpiAddF32{h, d}, sc))) return rc;
    if ((rc = rmsnorm<T_>(st, h, w.enc_ffn_norm + (size_t)l * d, a, R, d, d, c.rms_eps))) return rc;
    const T_* W1 = wl<T_>(w.W_1, l, (size_t)f * d);
    const T_* W3 = wl<T_>(w.W_3, l, (size_t)f * d);
    if ((rc = swiglu_proj<T_>(st, a, d, R, d, W1, W3, f, am, C, sc))) return rc;
    const T_* W2 = wl<T_>(w.W_2, l, (size_t)d * f);
    if ((rc = proj<T_>(st, am, f, R, f, W2, f, d, EpiAddF32{h, d}, sc))) return rc;
    // per-layer memory: group l from RMSNorm_e of this layer's output
    if (c.mem_source == RLT_MEM_PER_LAYER && l + 1 < L) {
      if ((rc = rmsnorm<T_>(st, h, w.enc_norm, a, R, d, d, c.rms_eps))) return rc;
      if ((rc = mem_proj(a, l))) return rc;
    }
  }
  if ((rc = rmsnorm<T_>(st, h, w.enc_norm, e, R, d, d, c.rms_eps))) return rc;
  if (c.mem_source == RLT_MEM_PER_LAYER) return mem_proj(e, L - 1);  // the last layer's source is e
  for (int g = 0; g < G; ++g)
    if ((rc = mem_proj(e, g))) return rc;
  return RLT_OK;
}

// ---------------------------------------------------------------------------
// decoder: the kernels of one step (enqueued during graph capture)

struct DecodeArgs {
  const void* e;
  const void* mem;
  int T_mem, n;
  const int32_t* actions;
  float inv_temp;
  int top_k;
  float *logp, *logp_full;
  int32_t* argmax;
  float* logits;
  int n_emit;
  // generation: sample the next token instead of scoring actions
  int* next_tok = nullptr;
  int* sample_tok = nullptr;
  unsigned long long seed = 0;
};

template <typename T_>
int enqueue_step(const rlt_model* m, rlt_state* sst, const DecodeArgs& A, void* ws, const WsLayout& Lw,
                 cudaStream_t st, int* n_kernels) {
  const rlt_config& c = m->cfg;
  const rlt_weights& w = m->w;
  const int B = sst->batch;
  const int d = c.d_model, f = c.d_ffn, H = c.n_heads, hd = c.head_dim, L = c.n_layers, Wn = c.window;
  const int V = c.vocab;
  StepCtx* ctx = at<StepCtx>(ws, Lw.ctx);
  int* status = at<int>(ws, Lw.status);
  const float2* tab = at<float2>(ws, Lw.rope);
  float* h = at<float>(ws, Lw.d_h);
  T_* x = at<T_>(ws, Lw.d_x);
  T_* xm = at<T_>(ws, Lw.d_m);
  float* C = at<float>(ws, Lw.d_c);
  const TcScratch sc = tc_scratch(m, ws, Lw);
  T_* o = at<T_>(ws, Lw.d_o);
  float* part = at<float>(ws, Lw.d_part);
  const T_* e = static_cast<const T_*>(A.e);
  const T_* mem = static_cast<const T_*>(A.mem);
  const float scale = 1.0f / sqrtf((float)hd);
  int rc, nk = 0;
  auto post = [&]() {
    g_launches++;
    nk++;
    return launch_ok();
  };
  // event-record node around launches of the timed class
  KernelTimer* tm = m->timer;
  auto mark = [&](int cls) -> int {
    if (!tm || tm->cls != cls) return RLT_OK;
    size_t j = tm->nodes.size();
    if (j >= tm->ph.size()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return RLT_ECUDA;
      tm->ph.push_back(e);
    }
    if (cudaEventRecordWithFlags(tm->ph[j], st, cudaEventRecordExternal) != cudaSuccess) return RLT_ECUDA;
    cudaStreamCaptureStatus cst;
    const cudaGraphNode_t* deps = nullptr;
    size_t nd = 0;
    if (cudaStreamGetCaptureInfo(st, &cst, nullptr, nullptr, &deps, nullptr, &nd) != cudaSuccess || nd != 1)
      return RLT_ECUDA;
    tm->nodes.push_back(deps[0]);
    return RLT_OK;
  };
  if (tm) tm->nodes.clear();
  if ((rc = mark(RLT_TIMER_STEP))) return rc;
  // merge
  const int bd = B * d;
  if (c.gate_mode == RLT_GATE_LEARNED) {
    merge_prep_kernel<T_><<<cdiv(bd, 256), 256, 0, st>>>(e, sst->s, x, B, A.T_mem, d, ctx);
    if ((rc = post())) return rc;
    const T_* Wg = static_cast<const T_*>(w.W_g);
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    if ((rc = proj<T_>(st, x, 2 * d, B, 2 * d, Wg, 2 * d, d, EpiStoreF32{C, d}, sc))) return rc;
    nk++;
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
  }
  merge_blend_kernel<T_><<<cdiv(bd, 256), 256, 0, st>>>(C, w.b_g, e, sst->s, h, B, A.T_mem, d,
                                                        c.gate_mode == RLT_GATE_DISCARD_S, ctx);
  if ((rc = post())) return rc;
  const size_t ring_layer = (size_t)B * H * Wn * hd;
  const size_t plane = (size_t)B * H * A.T_mem * hd;
  T_* rk = static_cast<T_*>(sst->ring_k);
  T_* rv = static_cast<T_*>(sst->ring_v);
  const size_t swa_smem = sizeof(float) * (hd + Wn);
  XattnArgs xa{};
  xa.part = part;
  xa.cnt = at<int>(ws, Lw.d_cnt);
  xa.out = o;
  xa.q = C;
  xa.B = B;
  xa.H = H;
  xa.T_mem = A.T_mem;
  xa.t_cap = A.T_mem;
  xa.scale = scale;
  xa.ctx = ctx;
  xa.status = status;
  for (int l = 0; l < L; ++l) {
    // self-attention over the window
    if ((rc = rmsnorm<T_>(st, h, w.dec_attn_norm + (size_t)l * d, x, B, d, d, c.rms_eps))) return rc;
    nk++;
    const T_* Wqkv = wl<T_>(w.W_qkv, l, (size_t)3 * d * d);
    if constexpr (std::is_same<T_, bf16>::value) {
      // QKV on the tensor cores; the epilogue applies RoPE, keeps q in C and
      // writes k, v to ring slot p mod W; then attention over the ring
      if ((rc = mark(RLT_TIMER_GEMM))) return rc;
      EpiQKVRope<T_> eq{C, rk + l * ring_layer, rv + l * ring_layer, tab, ctx, d, H, hd, Wn};
      if ((rc = gemm_bf16_tc(st, x, d, B, d, Wqkv, d, 3 * d, eq, sc))) return rc;
      nk++;
      if ((rc = mark(RLT_TIMER_GEMM))) return rc;
      if ((rc = mark(RLT_TIMER_SWA))) return rc;
      XattnArgs sa = xa;
      sa.q = C;
      sa.mk = rk + l * ring_layer;
      sa.mv = rv + l * ring_layer;
      sa.T_mem = Wn;
      sa.t_cap = Wn;
      if (launch_xattn<T_>(sa, hd, m->n_sm, st) != cudaSuccess) return RLT_ECUDA;
      if ((rc = post())) return rc;
      if ((rc = mark(RLT_TIMER_SWA))) return rc;
    } else {
      if ((rc = mark(RLT_TIMER_GEMM))) return rc;
      if ((rc = proj<T_>(st, x, d, B, d, Wqkv, d, 3 * d, EpiStoreF32{C, 3 * d}, sc))) return rc;
      nk++;
      if ((rc = mark(RLT_TIMER_GEMM))) return rc;
      if ((rc = mark(RLT_TIMER_SWA))) return rc;
      dec_swa_kernel<T_><<<dim3(H, B), 128, swa_smem, st>>>(C, rk + l * ring_layer, rv + l * ring_layer, o, tab, H,
                                                            hd, Wn, scale, ctx);
      if ((rc = post())) return rc;
      if ((rc = mark(RLT_TIMER_SWA))) return rc;
    }
    const T_* WO = wl<T_>(w.W_O, l, (size_t)d * d);
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    if ((rc = proj<T_>(st, o, d, B, d, WO, d, d, EpiAddF32{h, d}, sc))) return rc;
    nk++;
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    // cross-attention to memory positions 0..p
    if ((rc = rmsnorm<T_>(st, h, w.dec_xattn_norm + (size_t)l * d, x, B, d, d, c.rms_eps))) return rc;
    nk++;
    const T_* WQx = wl<T_>(w.W_Qx, l, (size_t)d * d);
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    if ((rc = proj<T_>(st, x, d, B, d, WQx, d, d, EpiStoreF32{C, d}, sc))) return rc;
    nk++;
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    const int g = (c.mem_groups == 1) ? 0 : l;
    if ((rc = mark(RLT_TIMER_XATTN))) return rc;
    xa.mk = mem + (2 * g) * plane;
    xa.mv = mem + (2 * g + 1) * plane;
    if (launch_xattn<T_>(xa, hd, m->n_sm, st) != cudaSuccess) return RLT_ECUDA;
    if ((rc = post())) return rc;
    if ((rc = mark(RLT_TIMER_XATTN))) return rc;
    const T_* WOx = wl<T_>(w.W_Ox, l, (size_t)d * d);
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    if ((rc = proj<T_>(st, o, d, B, d, WOx, d, d, EpiAddF32{h, d}, sc))) return rc;
    nk++;
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    // SwiGLU FFN
    if ((rc = rmsnorm<T_>(st, h, w.dec_ffn_norm + (size_t)l * d, x, B, d, d, c.rms_eps))) return rc;
    nk++;
    const T_* W1 = wl<T_>(w.W_1, l, (size_t)f * d);
    const T_* W3 = wl<T_>(w.W_3, l, (size_t)f * d);
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    {
      const uint64_t l0 = g_launches.load();
      if ((rc = swiglu_proj<T_>(st, x, d, B, d, W1, W3, f, xm, C, sc))) return rc;
      nk += (int)(g_launches.load() - l0);
    }
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    const T_* W2 = wl<T_>(w.W_2, l, (size_t)d * f);
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    if ((rc = proj<T_>(st, xm, f, B, f, W2, f, d, EpiAddF32{h, d}, sc))) return rc;
    nk++;
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
  }
  // head
  if ((rc = mark(RLT_TIMER_HEAD))) return rc;
  head_prep_kernel<T_><<<cdiv((size_t)B * 32, 256), 256, 0, st>>>(h, sst->s, w.head_norm, x, B, d, c.rms_eps);
  if ((rc = post())) return rc;
  const T_* Wo = static_cast<const T_*>(w.W_o);
  if ((rc = mark(RLT_TIMER_GEMM))) return rc;
  if ((rc = proj<T_>(st, x, d, B, d, Wo, d, V, EpiStoreF32{C, V}, sc))) return rc;
  nk++;
  if ((rc = mark(RLT_TIMER_GEMM))) return rc;
  HeadArgs ha;
  ha.logits = C;
  ha.actions = A.actions;
  ha.logp = A.logp;
  ha.logp_full = A.logp_full;
  ha.argmax = A.argmax;
  ha.emit_map = at<int>(ws, Lw.emit);
  ha.logits_out = (A.n_emit > 0) ? A.logits : nullptr;
  ha.B = B;
  ha.V = V;
  ha.n = A.n;
  ha.top_k = A.top_k;
  ha.inv_temp = A.inv_temp;
  ha.status = status;
  head_reduce_kernel<<<B, 1024, sizeof(float) * V, st>>>(ha, ctx);
  if ((rc = post())) return rc;
  if ((rc = mark(RLT_TIMER_HEAD))) return rc;
  advance_kernel<<<1, 1, 0, st>>>(ctx);
  if ((rc = post())) return rc;
  if ((rc = mark(RLT_TIMER_STEP))) return rc;
  *n_kernels = nk;
  return RLT_OK;
}

// One decoder step of a bf16 model (enqueued during graph capture):
//   gate GEMM [e_t; s_{t-1}] W_g^T with the merge in its epilogue -> h,
//   per layer: QKV (RoPE, ring write) -> window attention -> O (+ residual)
//              -> Qx -> cross-attention -> Ox (+ residual) -> W_1/W_3 (SwiGLU)
//              -> W_2 (+ residual),
//   head GEMM -> log-softmax reduction -> advance.
// Every RMSNorm is deferred into the projection that consumes it (row scale
// from the producer's sums of squares).  8 L + 4 kernels per step.
int enqueue_step_bf16(const rlt_model* m, rlt_state* sst, const DecodeArgs& A, void* ws, const WsLayout& Lw,
                      cudaStream_t st, int* n_kernels) {
  const rlt_config& c = m->cfg;
  const rlt_weights& w = m->w;
  const int B = sst->batch;
  const int d = c.d_model, f = c.d_ffn, H = c.n_heads, hd = c.head_dim, L = c.n_layers, Wn = c.window;
  const int V = c.vocab;
  StepCtx* ctx = at<StepCtx>(ws, Lw.ctx);
  int* status = at<int>(ws, Lw.status);
  const float2* tab = at<float2>(ws, Lw.rope);
  float* h = at<float>(ws, Lw.d_h);
  bf16* x = at<bf16>(ws, Lw.d_x);
  bf16* xm = at<bf16>(ws, Lw.d_m);
  float* C = at<float>(ws, Lw.d_c);
  bf16* o = at<bf16>(ws, Lw.d_o);
  float* ss = at<float>(ws, Lw.d_ss);
  bf16* s16 = at<bf16>(ws, Lw.d_s16);
  const TcScratch sc = tc_scratch(m, ws, Lw);
  auto act = [](const bf16* p, int ld) {
    AArg a;
    a.A = p;
    a.lda = ld;
    return a;
  };
  const bf16* e = static_cast<const bf16*>(A.e);
  const bf16* mem = static_cast<const bf16*>(A.mem);
  int rc, nk = 0;
  auto post = [&]() {
    g_launches++;
    nk++;
    return launch_ok();
  };
  KernelTimer* tm = m->timer;
  auto mark = [&](int cls) -> int {
    if (!tm || tm->cls != cls) return RLT_OK;
    size_t j = tm->nodes.size();
    if (j >= tm->ph.size()) {
      cudaEvent_t ev;
      if (cudaEventCreate(&ev) != cudaSuccess) return RLT_ECUDA;
      tm->ph.push_back(ev);
    }
    if (cudaEventRecordWithFlags(tm->ph[j], st, cudaEventRecordExternal) != cudaSuccess) return RLT_ECUDA;
    cudaStreamCaptureStatus cst;
    const cudaGraphNode_t* deps = nullptr;
    size_t nd = 0;
    if (cudaStreamGetCaptureInfo(st, &cst, nullptr, nullptr, &deps, nullptr, &nd) != cudaSuccess || nd != 1)
      return RLT_ECUDA;
    tm->nodes.push_back(deps[0]);
    return RLT_OK;
  };
  auto gemm_done = [&](int r) -> int {
    if (r) return r;
    nk++;
    return mark(RLT_TIMER_GEMM);
  };
  if (tm) tm->nodes.clear();
  if ((rc = mark(RLT_TIMER_STEP))) return rc;
  // merge: A = [e_t ; bf16(s_{t-1})], epilogue h = z s + (1 - z) e
  {
    AArg a;
    a.A = e;
    a.lda = d;
    a.T3 = A.T_mem;
    a.ctx = ctx;
    a.A2 = s16;
    a.lda2 = d;
    a.split = d;
    EpiMerge em{HOut{h, d, nullptr, nullptr, ss, B}, e, (size_t)A.T_mem * d, sst->s, w.b_g, ctx,
                c.gate_mode == RLT_GATE_DISCARD_S ? 1 : 0};
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    if ((rc = gemm_done(proj_bf16<false>(st, a, B, 2 * d, static_cast<const bf16*>(w.W_g), nullptr, 2 * d, d, em, sc)))) return rc;
  }
  // x = bf16(RMSNorm(h) * g) as the input of the next projection: built
  // inside that projection's kernel where it can (the same values, one
  // launch fewer), else by the RMSNorm kernel into x
  const bool fuse_norm = norm_fusable(B, d);
  auto normed = [&](const float* g, AArg* a) -> int {
    *a = act(x, d);
    if (fuse_norm) {
      a->nh = h;
      a->nss = ss;
      a->ng = g;
      a->neps = c.rms_eps;
      return RLT_OK;
    }
    nk++;
    return norm_rows(st, h, ss, g, x, B, d, c.rms_eps);
  };
  AArg xn;
  const size_t ring_layer = (size_t)B * H * Wn * hd;
  const size_t plane = (size_t)B * H * A.T_mem * hd;
  bf16* rk = static_cast<bf16*>(sst->ring_k);
  bf16* rv = static_cast<bf16*>(sst->ring_v);
  XattnArgs xa{};
  xa.part = at<float>(ws, Lw.d_part);
  xa.cnt = at<int>(ws, Lw.d_cnt);
  xa.out = o;
  xa.q = C;
  xa.B = B;
  xa.H = H;
  xa.scale = 1.0f / sqrtf((float)hd);
  xa.ctx = ctx;
  xa.status = status;
  for (int l = 0; l < L; ++l) {
    const size_t ld = (size_t)l * d;
    // self-attention over the window
    const bf16* Wqkv = wl<bf16>(w.W_qkv, l, (size_t)3 * d * d);
    EpiQKVRope<bf16> eq{C, rk + l * ring_layer, rv + l * ring_layer, tab, ctx, d, H, hd, Wn};
    if ((rc = normed(w.dec_attn_norm + ld, &xn))) return rc;
    TcScratch sq = sc;
    if (l == 0 && fuse_norm && m->inject_kernel == RLT_KERNEL_NORM_PROJ) {  // one-shot (rlt_debug_withhold_copy)
      sq.budget = m->inject_budget;
      sq.withhold = 1;
      m->inject_kernel = 0;
    }
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    if ((rc = gemm_done(proj_bf16<false>(st, xn, B, d, Wqkv, nullptr, d, 3 * d, eq, sq)))) return rc;
    if ((rc = mark(RLT_TIMER_SWA))) return rc;
    {
      XattnArgs sa = xa;
      sa.mk = rk + l * ring_layer;
      sa.mv = rv + l * ring_layer;
      sa.T_mem = Wn;
      sa.t_cap = Wn;
      sa.early = 2;  // the ring entry of this step is written by the QKV projection just before
      if (launch_xattn<bf16>(sa, hd, m->n_sm, st) != cudaSuccess) return RLT_ECUDA;
      if ((rc = post())) return rc;
    }
    if ((rc = mark(RLT_TIMER_SWA))) return rc;
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    if ((rc = gemm_done(proj_bf16<false>(st, act(o, d), B, d, wl<bf16>(w.W_O, l, (size_t)d * d), nullptr, d, d,
                                         EpiResidual{HOut{h, d, nullptr, nullptr, ss, B}}, sc))))
      return rc;
    // cross-attention to memory positions 0..p
    if ((rc = normed(w.dec_xattn_norm + ld, &xn))) return rc;
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    if ((rc = gemm_done(proj_bf16<false>(st, xn, B, d, wl<bf16>(w.W_Qx, l, (size_t)d * d), nullptr, d, d,
                                         EpiStoreF32{C, d}, sc))))
      return rc;
    const int g = (c.mem_groups == 1) ? 0 : l;
    if ((rc = mark(RLT_TIMER_XATTN))) return rc;
    {
      XattnArgs ca = xa;
      ca.mk = mem + (2 * g) * plane;
      ca.mv = mem + (2 * g + 1) * plane;
      ca.T_mem = A.T_mem;
      ca.t_cap = A.T_mem;
      ca.early = 1;  // encoder memory: written before the decoder call
      if (launch_xattn<bf16>(ca, hd, m->n_sm, st) != cudaSuccess) return RLT_ECUDA;
      if ((rc = post())) return rc;
    }
    if ((rc = mark(RLT_TIMER_XATTN))) return rc;
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    if ((rc = gemm_done(proj_bf16<false>(st, act(o, d), B, d, wl<bf16>(w.W_Ox, l, (size_t)d * d), nullptr, d, d,
                                         EpiResidual{HOut{h, d, nullptr, nullptr, ss, B}}, sc))))
      return rc;
    // SwiGLU FFN
    if ((rc = normed(w.dec_ffn_norm + ld, &xn))) return rc;
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    if ((rc = gemm_done(proj_bf16<true>(st, xn, B, d, wl<bf16>(w.W_1, l, (size_t)f * d),
                                        wl<bf16>(w.W_3, l, (size_t)f * d), d, f, EpiStoreT<bf16>{xm, f}, sc))))
      return rc;
    const bool last = (l + 1 == L);
    HOut ho{h, d, last ? sst->s : nullptr, last ? s16 : nullptr, ss, B};
    if ((rc = mark(RLT_TIMER_GEMM))) return rc;
    if ((rc = gemm_done(proj_bf16<false>(st, act(xm, f), B, f, wl<bf16>(w.W_2, l, (size_t)d * f), nullptr, f, d, EpiResidual{ho}, sc))))
      return rc;
  }
  // head: logits = W_o x with x = bf16(RMSNorm_o(s_t))
  if ((rc = mark(RLT_TIMER_HEAD))) return rc;
  if ((rc = normed(w.head_norm, &xn))) return rc;
  if ((rc = mark(RLT_TIMER_GEMM))) return rc;
  if ((rc = gemm_done(proj_bf16<false>(st, xn, B, d, static_cast<const bf16*>(w.W_o), nullptr, d, V, EpiStoreF32{C, V}, sc))))
    return rc;
  HeadArgs ha;
  ha.logits = C;
  ha.actions = A.actions;
  ha.logp = A.logp;
  ha.logp_full = A.logp_full;
  ha.argmax = A.argmax;
  ha.emit_map = at<int>(ws, Lw.emit);
  ha.logits_out = (A.n_emit > 0) ? A.logits : nullptr;
  ha.B = B;
  ha.V = V;
  ha.n = A.n;
  ha.top_k = A.top_k;
  ha.inv_temp = A.inv_temp;
  ha.status = status;
  ha.next_tok = A.next_tok;
  ha.sample_tok = A.sample_tok;
  ha.sample_off = 1;  // the token drawn from s_{p+1} is the one at position p + 1
  ha.seed = A.seed;
  if ((rc = launch_pdl(head_reduce_kernel, dim3(B), dim3(1024), sizeof(float) * V, st, ha, (const StepCtx*)ctx)))
    return rc;
  if ((rc = post())) return rc;
  if ((rc = mark(RLT_TIMER_HEAD))) return rc;
  if ((rc = launch_pdl(advance_kernel, dim3(1), dim3(1), 0, st, ctx))) return rc;
  if ((rc = post())) return rc;
  if ((rc = mark(RLT_TIMER_STEP))) return rc;
  *n_kernels = nk;
  return RLT_OK;
}

// One incremental encoder step of bf16 models (generation): the token
// next_tok[b] of every sequence, at position p = ctx->pos, through the
// encoder layers with its keys and values appended to the encoder cache
// enc_kv [L][2][B][H][T_max][hd], then e[:, p] and the memory rows of p.  The
// projections and norms follow the token-parallel encoder's numerics; the
// attention over the cached positions 0..p is the decoder's streaming kernel
// (fp32 online softmax), where the token-parallel encoder rounds P to bf16 on
// the final row maximum.  Uses the decoder scratch of the workspace.
int enqueue_enc_step_bf16(const rlt_model* m, int B, int T_max, bf16* e, bf16* mem, bf16* enc_kv, void* ws,
                          const WsLayout& Lw, cudaStream_t st, int* n_kernels) {
  const rlt_config& c = m->cfg;
  const rlt_weights& w = m->w;
  const int d = c.d_model, f = c.d_ffn, H = c.n_heads, hd = c.head_dim, L = c.n_layers, G = c.mem_groups;
  StepCtx* ctx = at<StepCtx>(ws, Lw.ctx);
  int* status = at<int>(ws, Lw.status);
  const float2* tab = at<float2>(ws, Lw.rope);
  const int* tok = at<int>(ws, Lw.d_tok);
  float* h = at<float>(ws, Lw.d_h);
  bf16* x = at<bf16>(ws, Lw.d_x);
  bf16* xm = at<bf16>(ws, Lw.d_m);
  float* C = at<float>(ws, Lw.d_c);
  bf16* o = at<bf16>(ws, Lw.d_o);
  float* ss = at<float>(ws, Lw.d_ss);
  const TcScratch sc = tc_scratch(m, ws, Lw);
  auto act = [](const bf16* p, int ld) {
    AArg a;
    a.A = p;
    a.lda = ld;
    return a;
  };
  int rc, nk = 0;
  const size_t kvp = (size_t)B * H * T_max * hd;   // one K or V plane of the encoder cache
  const size_t mplane = (size_t)B * H * T_max * hd;  // one K or V plane of the memory
  // memory rows of position p for group g from the normed rows src [B][d]
  auto mem_rows = [&](const bf16* src, int g) -> int {
    int r;
    if ((r = proj_bf16<false>(st, act(src, d), B, d, wl<bf16>(w.W_K, g, (size_t)d * d), nullptr, d, d,
                              EpiMemRow<bf16>{mem + (2 * g) * mplane, T_max, H, hd, ctx}, sc)))
      return r;
    nk++;
    if ((r = proj_bf16<false>(st, act(src, d), B, d, wl<bf16>(w.W_V, g, (size_t)d * d), nullptr, d, d,
                              EpiMemRow<bf16>{mem + (2 * g + 1) * mplane, T_max, H, hd, ctx}, sc)))
      return r;
    nk++;
    return RLT_OK;
  };
  auto norm = [&](const float* g, bf16* out) -> int {
    nk++;
    return norm_rows(st, h, ss, g, out, B, d, c.rms_eps);
  };
  // the input of the next projection: bf16(RMSNorm(h) * g) built inside it
  // where it can (as in the decoder step), else by the RMSNorm kernel into x
  const bool fuse_norm = norm_fusable(B, d);
  auto normed = [&](const float* g, AArg* a) -> int {
    *a = act(x, d);
    if (!fuse_norm) return norm(g, x);
    a->nh = h;
    a->nss = ss;
    a->ng = g;
    a->neps = c.rms_eps;
    return RLT_OK;
  };
  AArg xn = act(x, d);  // layer 0: the embedding kernel's normalised rows
  embed_norm_kernel<<<B, d / 4, 0, st>>>(tok, static_cast<const bf16*>(w.tok_emb), h, x, w.enc_attn_norm, B, d,
                                         c.vocab, c.rms_eps, status);
  g_launches++;
  nk++;
  if ((rc = launch_ok())) return rc;
  XattnArgs xa{};
  xa.part = at<float>(ws, Lw.d_part);
  xa.cnt = at<int>(ws, Lw.d_cnt);
  xa.out = o;
  xa.q = C;
  xa.B = B;
  xa.H = H;
  xa.scale = 1.0f / sqrtf((float)hd);
  xa.ctx = ctx;
  xa.status = status;
  for (int l = 0; l < L; ++l) {
    bf16* kc = enc_kv + (2 * l) * kvp;
    bf16* vc = enc_kv + (2 * l + 1) * kvp;
    // q, k with RoPE at p; k, v appended at cache slot p
    EpiQKVRope<bf16> eq{C, kc, vc, tab, ctx, d, H, hd, T_max};
    if ((rc = proj_bf16<false>(st, xn, B, d, wl<bf16>(w.W_qkv, l, (size_t)3 * d * d), nullptr, d, 3 * d, eq, sc)))
      return rc;
    nk++;
    XattnArgs sa = xa;
    sa.mk = kc;
    sa.mv = vc;
    sa.T_mem = T_max;
    sa.t_cap = T_max;
    sa.early = 2;  // slot p is written by the projection just before
    if (launch_xattn<bf16>(sa, hd, m->n_sm, st) != cudaSuccess) return RLT_ECUDA;
    g_launches++;
    nk++;
    if ((rc = launch_ok())) return rc;
    if ((rc = proj_bf16<false>(st, act(o, d), B, d, wl<bf16>(w.W_O, l, (size_t)d * d), nullptr, d, d,
                               EpiResidual{HOut{h, d, nullptr, nullptr, ss, B}}, sc)))
      return rc;
    nk++;
    if ((rc = normed(w.enc_ffn_norm + (size_t)l * d, &xn))) return rc;
    if ((rc = proj_bf16<true>(st, xn, B, d, wl<bf16>(w.W_1, l, (size_t)f * d), wl<bf16>(w.W_3, l, (size_t)f * d), d, f,
                              EpiStoreT<bf16>{xm, f}, sc)))
      return rc;
    nk++;
    if ((rc = proj_bf16<false>(st, act(xm, f), B, f, wl<bf16>(w.W_2, l, (size_t)d * f), nullptr, f, d,
                               EpiResidual{HOut{h, d, nullptr, nullptr, ss, B}}, sc)))
      return rc;
    nk++;
    if (c.mem_source == RLT_MEM_PER_LAYER && l + 1 < L) {  // group l from this layer's output
      if ((rc = norm(w.enc_norm, o))) return rc;
      if ((rc = mem_rows(o, l))) return rc;
    }
    if (l + 1 < L && (rc = normed(w.enc_attn_norm + (size_t)(l + 1) * d, &xn))) return rc;
  }
  // e_p = RMSNorm_e(h), then the memory rows of p
  if ((rc = norm(w.enc_norm, x))) return rc;
  if ((rc = launch_pdl(put_row_kernel, dim3(B), dim3(128), 0, st, (const bf16*)x, e, B, d, T_max,
                       (const StepCtx*)ctx)))
    return rc;
  g_launches++;
  nk++;
  if (c.mem_source == RLT_MEM_PER_LAYER) {
    if ((rc = mem_rows(x, L - 1))) return rc;
  } else {
    for (int g = 0; g < G; ++g)
      if ((rc = mem_rows(x, g))) return rc;
  }
  *n_kernels = nk;
  return RLT_OK;
}

// Autoregressive generation of bf16 models ("Understanding and Applying the
// Recurrent Looped Transformer Architecture", "Autoregressive generation"):
// from the state's distribution draw a token, encode it incrementally,
// consume it through the decoder exactly once; n times.  The first draw comes
// from the state the call starts with (its head computed here, bitwise as a
// step's head); each captured iteration then encodes and consumes the drawn
// token and draws the next one.
int gen_impl(const rlt_model* m, rlt_state* sst, bf16* e, bf16* mem, bf16* enc_kv, int T_max, int n,
             unsigned long long seed, float inv_temp, int top_k, int32_t* tokens, float* logp, void* ws,
             cudaStream_t st) {
  const rlt_config& c = m->cfg;
  const int B = sst->batch, d = c.d_model, V = c.vocab;
  WsLayout Lw = layout(m, B, T_max);
  const int p0 = sst->pos;
  StepCtx* ctx = at<StepCtx>(ws, Lw.ctx);
  int rc;
  set_ctx_kernel<<<1, 1, 0, st>>>(ctx, p0);
  g_launches++;
  const int half = c.head_dim / 2;
  rope_table_kernel<<<cdiv((size_t)n * half, 256), 256, 0, st>>>(at<float2>(ws, Lw.rope), p0, n, half,
                                                                 (double)c.rope_theta);
  g_launches++;
  if ((rc = launch_ok())) return rc;
  RLT_CUDA_TRY(cudaMemsetAsync(at<int>(ws, Lw.d_cnt), 0, sizeof(int) * (size_t)B * c.n_heads, st));
  {
    const size_t nn = (size_t)B * d;
    to_bf16_kernel<<<cdiv(nn, 256), 256, 0, st>>>(sst->s, at<bf16>(ws, Lw.d_s16), nn);
    g_launches++;
  }
  // first draw: head of s_{p0} (sums of squares as the residual epilogue
  // makes them, so the normed input is bitwise the in-step one)
  float* ss = at<float>(ws, Lw.d_ss);
  bf16* x = at<bf16>(ws, Lw.d_x);
  float* C = at<float>(ws, Lw.d_c);
  row_ss_kernel<<<cdiv((size_t)B * (d / 128), 4), 128, 0, st>>>(sst->s, ss, B, d);
  g_launches++;
  if ((rc = launch_ok())) return rc;
  if ((rc = norm_rows(st, sst->s, ss, m->w.head_norm, x, B, d, c.rms_eps))) return rc;
  TcScratch sc = tc_scratch(m, ws, Lw);
  {
    AArg a;
    a.A = x;
    a.lda = d;
    if ((rc = proj_bf16<false>(st, a, B, d, static_cast<const bf16*>(m->w.W_o), nullptr, d, V, EpiStoreF32{C, V},
                               sc)))
      return rc;
  }
  HeadArgs h0{};
  h0.logits = C;
  h0.logp = logp;
  h0.B = B;
  h0.V = V;
  h0.n = n;
  h0.top_k = top_k;
  h0.inv_temp = inv_temp;
  h0.status = at<int>(ws, Lw.status);
  h0.next_tok = at<int>(ws, Lw.d_tok);
  h0.sample_tok = tokens;
  h0.sample_off = 0;
  h0.seed = seed;
  if ((rc = launch_pdl(head_reduce_kernel, dim3(B), dim3(1024), sizeof(float) * V, st, h0, (const StepCtx*)ctx)))
    return rc;
  g_launches++;
  // one captured iteration: encode the drawn token at p, consume it, draw the next
  DecodeArgs A;
  A.e = e;
  A.mem = mem;
  A.T_mem = T_max;
  A.n = n;
  A.actions = nullptr;
  A.inv_temp = inv_temp;
  A.top_k = top_k;
  A.logp = logp;
  A.logp_full = nullptr;
  A.argmax = nullptr;
  A.logits = nullptr;
  A.n_emit = 0;
  A.next_tok = at<int>(ws, Lw.d_tok);
  A.sample_tok = tokens;
  A.seed = seed;
  cudaStream_t cs = m->cap_stream;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  RLT_CUDA_TRY(cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal));
  int nk_e = 0, nk_d = 0;
  const uint64_t before = g_launches.load();
  rc = enqueue_enc_step_bf16(m, B, T_max, e, mem, enc_kv, ws, Lw, cs, &nk_e);
  if (!rc) rc = enqueue_step_bf16(m, sst, A, ws, Lw, cs, &nk_d);
  cudaError_t ce = cudaStreamEndCapture(cs, &graph);
  g_launches.store(before);
  if (rc) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (ce != cudaSuccess) return RLT_ECUDA;
  ce = cudaGraphInstantiate(&exec, graph, 0);
  if (ce != cudaSuccess) {
    cudaGraphDestroy(graph);
    return RLT_ECUDA;
  }
  for (int i = 0; i < n; ++i) {
    ce = cudaGraphLaunch(exec, st);
    if (ce != cudaSuccess) break;
    g_launches += (uint64_t)(nk_e + nk_d);
  }
  cudaGraphDestroy(graph);
  cudaGraphExecDestroy(exec);
  if (ce != cudaSuccess) return RLT_ECUDA;
  sst->pos += n;
  return RLT_OK;
}

template <typename T_>
int decode_impl(const rlt_model* m, rlt_state* sst, const DecodeArgs& A, const int32_t* emit_steps, void* ws,
                cudaStream_t st) {
  const rlt_config& c = m->cfg;
  const int B = sst->batch;
  WsLayout Lw = layout(m, B, A.T_mem);
  const int p0 = sst->pos;
  int rc;
  // per-call setup (not captured): context, emit map, RoPE rows p0..p0+n-1
  set_ctx_kernel<<<1, 1, 0, st>>>(at<StepCtx>(ws, Lw.ctx), p0);
  g_launches++;
  std::vector<int> emap(A.n, -1);
  for (int j = 0; j < A.n_emit; ++j) emap[emit_steps[j]] = j;
  RLT_CUDA_TRY(cudaMemcpyAsync(at<int>(ws, Lw.emit), emap.data(), sizeof(int) * A.n, cudaMemcpyHostToDevice, st));
  const int half = c.head_dim / 2;
  rope_table_kernel<<<cdiv((size_t)A.n * half, 256), 256, 0, st>>>(at<float2>(ws, Lw.rope), p0, A.n, half,
                                                                   (double)c.rope_theta);
  g_launches++;
  if ((rc = launch_ok())) return rc;
  RLT_CUDA_TRY(cudaMemsetAsync(at<int>(ws, Lw.d_cnt), 0, sizeof(int) * (size_t)B * c.n_heads, st));
  if constexpr (std::is_same<T_, bf16>::value) {  // bf16(s_{t-1}) for the first step's gate input
    const size_t n = (size_t)B * c.d_model;
    to_bf16_kernel<<<cdiv(n, 256), 256, 0, st>>>(sst->s, at<bf16>(ws, Lw.d_s16), n);
    g_launches++;
    if ((rc = launch_ok())) return rc;
  }
  // capture one step and replay it n times
  cudaStream_t cs = m->cap_stream;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  RLT_CUDA_TRY(cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal));
  int nk = 0;
  const uint64_t before = g_launches.load();
  if constexpr (std::is_same<T_, bf16>::value)
    rc = enqueue_step_bf16(m, sst, A, ws, Lw, cs, &nk);
  else
    rc = enqueue_step<T_>(m, sst, A, ws, Lw, cs, &nk);
  cudaError_t ce = cudaStreamEndCapture(cs, &graph);
  g_launches.store(before);  // captured launches are counted when the graph runs
  if (rc) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (ce != cudaSuccess) return RLT_ECUDA;
  ce = cudaGraphInstantiate(&exec, graph, 0);
  if (ce != cudaSuccess) {
    cudaGraphDestroy(graph);
    return RLT_ECUDA;
  }
  KernelTimer* tm = m->timer;
  const int pairs = (tm && tm->cls != RLT_TIMER_OFF) ? (int)tm->nodes.size() / 2 : 0;
  bool parked = false;
  for (int i = 0; i < A.n; ++i) {
    if (pairs > 0) {
      if (tm->used + pairs <= tm->cap) {
        for (int j = 0; j < pairs; ++j) {
          cudaGraphExecEventRecordNodeSetEvent(exec, tm->nodes[2 * j], tm->ev[2 * (tm->used + j)]);
          cudaGraphExecEventRecordNodeSetEvent(exec, tm->nodes[2 * j + 1], tm->ev[2 * (tm->used + j) + 1]);
        }
        tm->used += pairs;
      } else if (!parked) {  // pool exhausted: point the nodes back at the placeholders
        for (size_t j = 0; j < tm->nodes.size(); ++j)
          cudaGraphExecEventRecordNodeSetEvent(exec, tm->nodes[j], tm->ph[j]);
        parked = true;
      }
    }
    ce = cudaGraphLaunch(exec, st);
    if (ce != cudaSuccess) break;
    g_launches += (uint64_t)nk;
  }
  cudaGraphDestroy(graph);
  // destroying an executable graph with launches in flight is allowed; its
  // resources are released once they complete
  cudaGraphExecDestroy(exec);
  if (ce != cudaSuccess) return RLT_ECUDA;
  sst->pos += A.n;
  return RLT_OK;
}

// ---------------------------------------------------------------------------
// persistent cluster decoder (dec_fused.cuh)

fused::Shape fused_shape(const rlt_config& c) {
  return fused::Shape{c.d_model, c.n_heads, c.head_dim, c.d_ffn, c.n_layers, c.window, c.vocab, c.mem_groups,
                      c.gate_mode == RLT_GATE_DISCARD_S ? 0 : 1, c.mem_source == RLT_MEM_PER_LAYER ? 1 : 0};
}

// Generation through the persistent kernel (rlt_generate on the fused path).
struct FusedGen {
  bf16* enc_kv;
  int32_t* tokens;
  unsigned long long seed;
};

// The kernel's launch attributes for smem bytes of dynamic shared memory
// (clusters of up to 16 CTAs are outside the portable size 8).
int fused_attrs(size_t smem) {
  if (cudaFuncSetAttribute(fused::dec_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(fused::dec_fused_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return RLT_ECUDA;
  return RLT_OK;
}

// Clusters of CS CTAs with smem bytes each that the device holds at once.
int fused_max_clusters(int CS, size_t smem) {
  if (fused_attrs(smem) != RLT_OK) return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS);
  cfg.blockDim = dim3(fused::kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = CS;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fused::dec_fused_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return n;
}

// The plan for B sequences (fused::choose_plan) with the device's
// co-resident clusters.
int fused_choose(const rlt_model* m, int B, fused::Plan* out) {
  if (m->cfg.dtype != RLT_BF16) return RLT_EUNSUPPORTED;
  const int rc = fused::choose_plan(fused_shape(m->cfg), B, m->fused_cs, fused_max_clusters, out);
  return rc ? RLT_EUNSUPPORTED : RLT_OK;
}

int decode_fused(const rlt_model* m, rlt_state* sst, const DecodeArgs& A, const int32_t* emit_steps, void* ws,
                 cudaStream_t st, const FusedGen* gen = nullptr) {
  const rlt_config& c = m->cfg;
  const int B = sst->batch;
  fused::Plan P;
  int rc = fused_choose(m, B, &P);
  if (rc) return rc;
  if (!aligned16(A.e) || !aligned16(A.mem) || !aligned16(sst->ring_k) || !aligned16(sst->ring_v)) return RLT_EINVAL;
  WsLayout Lw = layout(m, B, A.T_mem);
  std::vector<int> emap(A.n, -1);
  for (int j = 0; j < A.n_emit; ++j) emap[emit_steps[j]] = j;
  RLT_CUDA_TRY(cudaMemcpyAsync(at<int>(ws, Lw.emit), emap.data(), sizeof(int) * A.n, cudaMemcpyHostToDevice, st));
  const int half = c.head_dim / 2;  // RoPE rows of positions p0 .. p0 + n - 1
  rope_table_kernel<<<cdiv((size_t)A.n * half, 256), 256, 0, st>>>(at<float2>(ws, Lw.rope), sst->pos, A.n, half,
                                                                   (double)c.rope_theta);
  g_launches++;
  if ((rc = launch_ok())) return rc;
  const rlt_weights& w = m->w;
  fused::Args a = {};
  a.rope = at<const float2>(ws, Lw.rope);
  a.W_g = static_cast<const bf16*>(w.W_g);
  a.W_qkv = static_cast<const bf16*>(w.W_qkv);
  a.W_O = static_cast<const bf16*>(w.W_O);
  a.W_Qx = static_cast<const bf16*>(w.W_Qx);
  a.W_Ox = static_cast<const bf16*>(w.W_Ox);
  a.W_1 = static_cast<const bf16*>(w.W_1);
  a.W_3 = static_cast<const bf16*>(w.W_3);
  a.W_2 = static_cast<const bf16*>(w.W_2);
  a.W_o = static_cast<const bf16*>(w.W_o);
  a.b_g = w.b_g;
  a.attn_norm = w.dec_attn_norm;
  a.xattn_norm = w.dec_xattn_norm;
  a.ffn_norm = w.dec_ffn_norm;
  a.head_norm = w.head_norm;
  a.e = static_cast<bf16*>(const_cast<void*>(A.e));  // written only in generation
  a.mem = static_cast<bf16*>(const_cast<void*>(A.mem));
  if (gen) {
    a.gen = 1;
    a.tok_emb = static_cast<const bf16*>(w.tok_emb);
    a.enc_attn_norm = w.enc_attn_norm;
    a.enc_ffn_norm = w.enc_ffn_norm;
    a.enc_norm = w.enc_norm;
    a.W_K = static_cast<const bf16*>(w.W_K);
    a.W_V = static_cast<const bf16*>(w.W_V);
    a.enc_kv = gen->enc_kv;
    a.tokens = gen->tokens;
    a.seed = gen->seed;
  }
  a.actions = A.actions;
  a.emit_map = at<int>(ws, Lw.emit);
  a.logits_out = A.logits;
  a.logp = A.logp;
  a.logp_full = A.logp_full;
  a.argmax = A.argmax;
  a.s = sst->s;
  a.ring_k = static_cast<bf16*>(sst->ring_k);
  a.ring_v = static_cast<bf16*>(sst->ring_v);
  a.status = at<int>(ws, Lw.status);
  a.B = B;
  a.T_mem = A.T_mem;
  a.p0 = sst->pos;
  a.n = A.n;
  a.top_k = A.top_k;
  a.eps = c.rms_eps;
  a.theta = c.rope_theta;
  a.scale = 1.0f / sqrtf((float)c.head_dim);
  a.inv_temp = A.inv_temp;
  a.sh = fused_shape(c);
  a.P = P;
  if ((rc = fused_attrs(P.total))) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.nclu * P.CS);
  cfg.blockDim = dim3(fused::kThreads);
  cfg.dynamicSmemBytes = P.total;
  cfg.stream = st;
  cudaLaunchAttribute lat[1];
  lat[0].id = cudaLaunchAttributeClusterDimension;
  lat[0].val.clusterDim.x = P.CS;
  lat[0].val.clusterDim.y = 1;
  lat[0].val.clusterDim.z = 1;
  cfg.attrs = lat;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, fused::dec_fused_kernel, a) != cudaSuccess) return RLT_ECUDA;
  g_launches++;
  sst->pos += A.n;
  return RLT_OK;
}

int validate_cfg(const rlt_config* c) {
  if (!c) return RLT_EINVAL;
  if (c->d_model <= 0 || c->n_layers <= 0 || c->n_heads <= 0 || c->head_dim <= 0 || c->d_ffn <= 0 ||
      c->window <= 0 || c->vocab <= 0)
    return RLT_EINVAL;
  if (c->d_model != c->n_heads * c->head_dim) return RLT_EINVAL;
  if (c->mem_groups != 1 && c->mem_groups != c->n_layers) return RLT_EINVAL;
  if (c->dtype != RLT_F32 && c->dtype != RLT_BF16) return RLT_EINVAL;
  if (c->gate_mode != RLT_GATE_LEARNED && c->gate_mode != RLT_GATE_DISCARD_S) return RLT_EINVAL;
  if (c->mem_source != RLT_MEM_FINAL && c->mem_source != RLT_MEM_PER_LAYER) return RLT_EINVAL;
  if (c->mem_source == RLT_MEM_PER_LAYER && c->mem_groups != c->n_layers) return RLT_EINVAL;
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return RLT_EINVAL;
  // kernel limits
  if (c->head_dim % 8 != 0 || 128 % c->head_dim != 0) return RLT_EUNSUPPORTED;
  // bf16 rows are moved in 16-byte pieces
  if (c->dtype == RLT_BF16 && (c->d_model % 8 != 0 || c->d_ffn % 8 != 0)) return RLT_EUNSUPPORTED;
  // bf16 models: the residual stream is produced in tiles of up to 256
  // columns and the deferred RMSNorm keeps one sum of squares per 64 columns
  if (c->dtype == RLT_BF16 && c->d_model % 256 != 0) return RLT_EUNSUPPORTED;
  if (c->vocab > 49152) return RLT_EUNSUPPORTED;
  if (c->window > 4096) return RLT_EUNSUPPORTED;
  return RLT_OK;
}

}  // namespace

// ===========================================================================
// extern "C" entry points

extern "C" {

int rlt_abi_version(void) { return 200; }

uint64_t rlt_launch_count(void) { return g_launches.load(); }

const char* rlt_strerror(int code) {
  switch (code) {
    case RLT_OK: return "ok";
    case RLT_EINVAL: return "invalid argument";
    case RLT_ESTALE: return "state built under another model version";
    case RLT_ERANGE: return "position range exceeds the encoded length";
    case RLT_ECUDA: return "CUDA error";
    case RLT_ETIMEOUT: return "device wait timed out";
    case RLT_EBOUNDS: return "index out of range on the device";
    case RLT_EWORKSPACE: return "workspace too small";
    case RLT_EUNSUPPORTED: return "shape not supported by the kernels";
    default: return "unknown error";
  }
}

int rlt_model_create(const rlt_config* cfg, const rlt_weights* w, uint64_t version, rlt_model** out) {
  if (!out) return RLT_EINVAL;
  *out = nullptr;
  int rc = validate_cfg(cfg);
  if (rc) return rc;
  if (!w) return RLT_EINVAL;
  const void* ptrs[] = {w->tok_emb, w->s_star, w->W_g, w->b_g, w->W_qkv, w->W_O, w->W_1, w->W_3,
                        w->W_2, w->W_Qx, w->W_Ox, w->W_K, w->W_V, w->W_o, w->enc_attn_norm,
                        w->enc_ffn_norm, w->enc_norm, w->dec_attn_norm, w->dec_xattn_norm, w->dec_ffn_norm,
                        w->head_norm};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return RLT_EINVAL;
  rlt_model* m = new rlt_model();
  m->cfg = *cfg;
  m->w = *w;
  m->version = version;
  m->esz = (cfg->dtype == RLT_BF16) ? 2 : 4;
  m->timer = nullptr;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&m->n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || m->n_sm < 1) {
      delete m;
      return RLT_ECUDA;
    }
  }
  if (cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking) != cudaSuccess) {
    delete m;
    return RLT_ECUDA;
  }
  ensure_attrs();
  if (cfg->dtype == RLT_BF16 && deep_occupancy_all(m) != RLT_OK) {
    cudaStreamDestroy(m->cap_stream);
    delete m;
    return RLT_ECUDA;
  }
  *out = m;
  return RLT_OK;
}

// ---------------------------------------------------------------------------
// prefix snapshots

namespace {

// Header at the start of a snapshot (64 bytes), then s, ring K, ring V, e, M
// and (optional) the encoder's key/value cache, each section starting on a
// 256-byte boundary.
struct SnapHeader {
  uint32_t magic, abi;
  uint64_t version;
  int32_t B, pos, d, L, H, hd, W, G, dtype, mem_source;
  int32_t enc_kv;  // 1: the encoder cache section is present
  int32_t pad;
};
static_assert(sizeof(SnapHeader) == 64, "snapshot header");
constexpr uint32_t kSnapMagic = 0x534c5452u;  // "RTLS"

struct SnapLayout {
  size_t s, rk, rv, e, mem, kv, total;
  size_t s_bytes, ring_bytes, e_row, mem_row;  // e_row: pos * d elements, mem_row: pos * hd (bytes)
  size_t mem_rows;                              // G * 2 * B * H
  size_t kv_rows;                               // L * 2 * B * H (rows of mem_row bytes), 0 without the section
};
SnapLayout snap_layout(const rlt_model* m, int B, int pos, bool with_kv) {
  const rlt_config& c = m->cfg;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  SnapLayout L{};
  L.s_bytes = (size_t)B * c.d_model * 4;
  L.ring_bytes = (size_t)c.n_layers * B * c.n_heads * c.window * c.head_dim * m->esz;
  L.e_row = (size_t)pos * c.d_model * m->esz;
  L.mem_row = (size_t)pos * c.head_dim * m->esz;
  L.mem_rows = (size_t)c.mem_groups * 2 * B * c.n_heads;
  size_t off = up(sizeof(SnapHeader));
  L.s = off;
  off += up(L.s_bytes);
  L.rk = off;
  off += up(L.ring_bytes);
  L.rv = off;
  off += up(L.ring_bytes);
  L.e = off;
  off += up(L.e_row * B);
  L.mem = off;
  off += up(L.mem_row * L.mem_rows);
  L.kv = off;
  L.kv_rows = with_kv ? (size_t)c.n_layers * 2 * B * c.n_heads : 0;
  off += up(L.mem_row * L.kv_rows);
  L.total = off;
  return L;
}

__global__ void snap_header_kernel(SnapHeader* dst, SnapHeader h) { *dst = h; }

}  // namespace

int rlt_snapshot_size(const rlt_model* m, int32_t B, int32_t pos, int32_t with_enc_kv, size_t* bytes) {
  if (!m || !bytes || B <= 0 || pos < 0 || (with_enc_kv != 0 && with_enc_kv != 1)) return RLT_EINVAL;
  *bytes = snap_layout(m, B, pos, with_enc_kv != 0).total;
  return RLT_OK;
}

int rlt_snapshot_save(const rlt_model* m, const rlt_state* st, const void* e, const void* mem, const void* enc_kv,
                      int32_t T_mem, void* snap, size_t snap_bytes, rlt_stream_t stream) {
  if (!m || !st || !snap || !aligned16(snap) || st->batch <= 0 || !st->s || !st->ring_k || !st->ring_v)
    return RLT_EINVAL;
  if (st->version != m->version) return RLT_ESTALE;
  const int B = st->batch, pos = st->pos;
  if (pos < 0 || (pos > 0 && (!e || !mem || T_mem < pos))) return RLT_EINVAL;
  const bool with_kv = enc_kv != nullptr;
  const SnapLayout L = snap_layout(m, B, pos, with_kv);
  if (snap_bytes < L.total) return RLT_EINVAL;
  const rlt_config& c = m->cfg;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(snap);
  SnapHeader h{};
  h.magic = kSnapMagic;
  h.abi = (uint32_t)rlt_abi_version();
  h.version = m->version;
  h.B = B;
  h.pos = pos;
  h.d = c.d_model;
  h.L = c.n_layers;
  h.H = c.n_heads;
  h.hd = c.head_dim;
  h.W = c.window;
  h.G = c.mem_groups;
  h.dtype = c.dtype;
  h.mem_source = c.mem_source;
  h.enc_kv = with_kv ? 1 : 0;
  snap_header_kernel<<<1, 1, 0, s>>>(reinterpret_cast<SnapHeader*>(base), h);
  g_launches++;
  RLT_CUDA_TRY(cudaGetLastError());
  RLT_CUDA_TRY(cudaMemcpyAsync(base + L.s, st->s, L.s_bytes, cudaMemcpyDeviceToDevice, s));
  RLT_CUDA_TRY(cudaMemcpyAsync(base + L.rk, st->ring_k, L.ring_bytes, cudaMemcpyDeviceToDevice, s));
  RLT_CUDA_TRY(cudaMemcpyAsync(base + L.rv, st->ring_v, L.ring_bytes, cudaMemcpyDeviceToDevice, s));
  if (pos > 0) {
    // rows 0..pos-1 of every sequence (e) and of every (group, K/V, sequence, head) plane (M)
    RLT_CUDA_TRY(cudaMemcpy2DAsync(base + L.e, L.e_row, e, (size_t)T_mem * c.d_model * m->esz, L.e_row, B,
                                   cudaMemcpyDeviceToDevice, s));
    RLT_CUDA_TRY(cudaMemcpy2DAsync(base + L.mem, L.mem_row, mem, (size_t)T_mem * c.head_dim * m->esz, L.mem_row,
                                   L.mem_rows, cudaMemcpyDeviceToDevice, s));
    if (with_kv)  // rows 0..pos-1 of every (layer, K/V, sequence, head) plane of the encoder cache
      RLT_CUDA_TRY(cudaMemcpy2DAsync(base + L.kv, L.mem_row, enc_kv, (size_t)T_mem * c.head_dim * m->esz, L.mem_row,
                                     L.kv_rows, cudaMemcpyDeviceToDevice, s));
  }
  return RLT_OK;
}

int rlt_snapshot_restore(const rlt_model* m, const void* snap, size_t snap_bytes, rlt_state* st, void* e, void* mem,
                         void* enc_kv, int32_t T_mem, rlt_stream_t stream) {
  if (!m || !st || !snap || !aligned16(snap) || st->batch <= 0 || !st->s || !st->ring_k || !st->ring_v ||
      snap_bytes < sizeof(SnapHeader))
    return RLT_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  SnapHeader h{};
  RLT_CUDA_TRY(cudaMemcpyAsync(&h, snap, sizeof(h), cudaMemcpyDeviceToHost, s));
  RLT_CUDA_TRY(cudaStreamSynchronize(s));
  const rlt_config& c = m->cfg;
  if (h.magic != kSnapMagic || h.abi != (uint32_t)rlt_abi_version()) return RLT_EINVAL;
  if (h.d != c.d_model || h.L != c.n_layers || h.H != c.n_heads || h.hd != c.head_dim || h.W != c.window ||
      h.G != c.mem_groups || h.dtype != c.dtype || h.mem_source != c.mem_source || h.B != st->batch)
    return RLT_EINVAL;
  if (h.enc_kv != 0 && h.enc_kv != 1) return RLT_EINVAL;
  // the cache section is restored exactly when the caller asks for it, and
  // can only be asked for when the snapshot holds it
  if ((enc_kv != nullptr) != (h.enc_kv == 1)) return RLT_EINVAL;
  if (h.version != m->version) return RLT_ESTALE;
  const int B = h.B, pos = h.pos;
  if (pos < 0 || (pos > 0 && (!e || !mem || T_mem < pos))) return RLT_EINVAL;
  const SnapLayout L = snap_layout(m, B, pos, h.enc_kv == 1);
  if (snap_bytes < L.total) return RLT_EINVAL;
  const char* base = static_cast<const char*>(snap);
  RLT_CUDA_TRY(cudaMemcpyAsync(st->s, base + L.s, L.s_bytes, cudaMemcpyDeviceToDevice, s));
  RLT_CUDA_TRY(cudaMemcpyAsync(st->ring_k, base + L.rk, L.ring_bytes, cudaMemcpyDeviceToDevice, s));
  RLT_CUDA_TRY(cudaMemcpyAsync(st->ring_v, base + L.rv, L.ring_bytes, cudaMemcpyDeviceToDevice, s));
  if (pos > 0) {
    RLT_CUDA_TRY(cudaMemcpy2DAsync(e, (size_t)T_mem * c.d_model * m->esz, base + L.e, L.e_row, L.e_row, B,
                                   cudaMemcpyDeviceToDevice, s));
    RLT_CUDA_TRY(cudaMemcpy2DAsync(mem, (size_t)T_mem * c.head_dim * m->esz, base + L.mem, L.mem_row, L.mem_row,
                                   L.mem_rows, cudaMemcpyDeviceToDevice, s));
    if (enc_kv)
      RLT_CUDA_TRY(cudaMemcpy2DAsync(enc_kv, (size_t)T_mem * c.head_dim * m->esz, base + L.kv, L.mem_row, L.mem_row,
                                     L.kv_rows, cudaMemcpyDeviceToDevice, s));
  }
  st->pos = pos;
  st->version = h.version;
  return RLT_OK;
}

int rlt_model_set_version(rlt_model* m, uint64_t version) {
  if (!m) return RLT_EINVAL;
  m->version = version;
  return RLT_OK;
}

void rlt_model_destroy(rlt_model* m) {
  if (!m) return;
  cudaStreamSynchronize(m->cap_stream);
  cudaStreamDestroy(m->cap_stream);
  if (m->timer) {
    cudaDeviceSynchronize();
    for (cudaEvent_t e : m->timer->ev) cudaEventDestroy(e);
    for (cudaEvent_t e : m->timer->ph) cudaEventDestroy(e);
    delete m->timer;
  }
  delete m;
}

int rlt_timer_arm(rlt_model* m, int32_t kernel_class, int32_t max_launches) {
  if (!m || kernel_class < RLT_TIMER_OFF || kernel_class > RLT_TIMER_STEP || max_launches < 0) return RLT_EINVAL;
  if (!m->timer) m->timer = new KernelTimer();
  KernelTimer* t = m->timer;
  while ((int)t->ev.size() < 2 * max_launches) {
    cudaEvent_t e;
    RLT_CUDA_TRY(cudaEventCreate(&e));
    t->ev.push_back(e);
  }
  t->cap = max_launches;
  t->used = 0;
  t->cls = kernel_class;
  t->nodes.clear();
  return RLT_OK;
}

int rlt_timer_read(rlt_model* m, float* ms, int32_t cap, int32_t* n_out) {
  if (!m || !n_out || (cap > 0 && !ms)) return RLT_EINVAL;
  *n_out = 0;
  KernelTimer* t = m->timer;
  if (!t) return RLT_OK;
  RLT_CUDA_TRY(cudaDeviceSynchronize());
  int n = std::min(t->used, cap);
  for (int i = 0; i < n; ++i) RLT_CUDA_TRY(cudaEventElapsedTime(&ms[i], t->ev[2 * i], t->ev[2 * i + 1]));
  *n_out = t->used;
  t->cls = RLT_TIMER_OFF;
  t->used = 0;
  t->nodes.clear();
  return RLT_OK;
}

int rlt_workspace_size(const rlt_model* m, int32_t B, int32_t T_max, size_t* bytes) {
  if (!m || !bytes || B <= 0 || T_max <= 0) return RLT_EINVAL;
  *bytes = layout(m, B, T_max).total;
  return RLT_OK;
}

int rlt_workspace_init(void* ws, size_t ws_bytes, rlt_stream_t stream) {
  if (!ws || ws_bytes < kWsHeaderBytes || !aligned16(ws)) return RLT_EINVAL;
  RLT_CUDA_TRY(cudaMemsetAsync(ws, 0, kWsHeaderBytes, reinterpret_cast<cudaStream_t>(stream)));
  return RLT_OK;
}

int rlt_state_sizes(const rlt_model* m, int32_t B, size_t* s_bytes, size_t* ring_bytes) {
  if (!m || B <= 0) return RLT_EINVAL;
  const rlt_config& c = m->cfg;
  if (s_bytes) *s_bytes = (size_t)B * c.d_model * 4;
  if (ring_bytes) *ring_bytes = (size_t)c.n_layers * B * c.n_heads * c.window * c.head_dim * m->esz;
  return RLT_OK;
}

int rlt_state_init(const rlt_model* m, rlt_state* st, rlt_stream_t stream) {
  if (!m || !st || st->batch <= 0 || !st->s || !st->ring_k || !st->ring_v) return RLT_EINVAL;
  if (!aligned16(st->s) || !aligned16(st->ring_k) || !aligned16(st->ring_v)) return RLT_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const rlt_config& c = m->cfg;
  const int d = c.d_model;
  bcast_rows_kernel<<<cdiv((size_t)st->batch * d, 256), 256, 0, s>>>(st->s, m->w.s_star, st->batch, d);
  g_launches++;
  size_t ring_el = (size_t)c.n_layers * st->batch * c.n_heads * c.window * c.head_dim;
  if (m->cfg.dtype == RLT_BF16) {
    fill_nan_kernel<bf16><<<1184, 256, 0, s>>>(static_cast<bf16*>(st->ring_k), ring_el);
    fill_nan_kernel<bf16><<<1184, 256, 0, s>>>(static_cast<bf16*>(st->ring_v), ring_el);
  } else {
    fill_nan_kernel<float><<<1184, 256, 0, s>>>(static_cast<float*>(st->ring_k), ring_el);
    fill_nan_kernel<float><<<1184, 256, 0, s>>>(static_cast<float*>(st->ring_v), ring_el);
  }
  g_launches += 2;
  if (launch_ok()) return RLT_ECUDA;
  st->pos = 0;
  st->version = m->version;
  return RLT_OK;
}

int rlt_encode(const rlt_model* m, const int32_t* tokens, int32_t B, int32_t T, void* e, void* mem, void* ws,
               size_t ws_bytes, rlt_stream_t stream) {
  if (!m || !tokens || !e || !mem || !ws || B <= 0 || T <= 0) return RLT_EINVAL;
  if (!aligned16(e) || !aligned16(mem) || !aligned16(ws) || !aligned16(tokens)) return RLT_EINVAL;
  if (ws_bytes < layout(m, B, T).total) return RLT_EWORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (m->cfg.dtype == RLT_BF16)
    return encode_bf16(m, tokens, B, T, static_cast<bf16*>(e), static_cast<bf16*>(mem), ws, s);
  return encode_impl<float>(m, tokens, B, T, static_cast<float*>(e), static_cast<float*>(mem), ws, s);
}

int rlt_encode_kv(const rlt_model* m, const int32_t* tokens, int32_t B, int32_t T, int32_t T_max, void* e, void* mem,
                  void* enc_kv, void* ws, size_t ws_bytes, rlt_stream_t stream) {
  if (!m || !tokens || !e || !mem || !enc_kv || !ws || B <= 0 || T <= 0 || T_max < T) return RLT_EINVAL;
  if (!aligned16(e) || !aligned16(mem) || !aligned16(enc_kv) || !aligned16(ws) || !aligned16(tokens))
    return RLT_EINVAL;
  if (m->cfg.dtype != RLT_BF16) return RLT_EUNSUPPORTED;
  if (ws_bytes < layout(m, B, T_max).total) return RLT_EWORKSPACE;
  return encode_bf16(m, tokens, B, T, static_cast<bf16*>(e), static_cast<bf16*>(mem), ws,
                     reinterpret_cast<cudaStream_t>(stream), T_max, static_cast<bf16*>(enc_kv));
}

int rlt_generate(const rlt_model* m, rlt_state* st, void* e, void* mem, void* enc_kv, int32_t T_max, int32_t n,
                 uint64_t seed, float temperature, int32_t top_k, int32_t* tokens, float* logp, void* ws,
                 size_t ws_bytes, rlt_stream_t stream) {
  if (!m || !st || !e || !mem || !enc_kv || !tokens || !ws || T_max <= 0 || n < 0 || st->batch <= 0)
    return RLT_EINVAL;
  if (!st->s || !st->ring_k || !st->ring_v) return RLT_EINVAL;
  if (!aligned16(e) || !aligned16(mem) || !aligned16(enc_kv) || !aligned16(ws)) return RLT_EINVAL;
  if (!(temperature > 0.f) || top_k < 0) return RLT_EINVAL;
  if (m->cfg.dtype != RLT_BF16) return RLT_EUNSUPPORTED;
  if (st->version != m->version) return RLT_ESTALE;
  if (st->pos < 0 || (int64_t)st->pos + n > T_max) return RLT_ERANGE;
  if (ws_bytes < layout(m, st->batch, T_max).total) return RLT_EWORKSPACE;
  if (n == 0) return RLT_OK;
  if (m->decode_path == RLT_DECODE_FUSED) {
    DecodeArgs A;
    A.e = e;
    A.mem = mem;
    A.T_mem = T_max;
    A.n = n;
    A.actions = nullptr;
    A.inv_temp = 1.0f / temperature;
    A.top_k = top_k;
    A.logp = logp;
    A.logp_full = nullptr;
    A.argmax = nullptr;
    A.logits = nullptr;
    A.n_emit = 0;
    const FusedGen g{static_cast<bf16*>(enc_kv), tokens, (unsigned long long)seed};
    return decode_fused(m, st, A, nullptr, ws, reinterpret_cast<cudaStream_t>(stream), &g);
  }
  return gen_impl(m, st, static_cast<bf16*>(e), static_cast<bf16*>(mem), static_cast<bf16*>(enc_kv), T_max, n,
                  (unsigned long long)seed, 1.0f / temperature, top_k, tokens, logp, ws,
                  reinterpret_cast<cudaStream_t>(stream));
}

int rlt_decode_steps(const rlt_model* m, rlt_state* st, const void* e, const void* mem, int32_t T_mem, int32_t n,
                     const int32_t* actions, float temperature, int32_t top_k, float* logp, float* logp_full,
                     int32_t* argmax, const int32_t* emit_steps, int32_t n_emit, float* logits, void* ws,
                     size_t ws_bytes, rlt_stream_t stream) {
  if (!m || !st || !e || !mem || !ws || T_mem <= 0 || n < 0 || st->batch <= 0) return RLT_EINVAL;
  if (!st->s || !st->ring_k || !st->ring_v) return RLT_EINVAL;
  if (!(temperature > 0.f) || top_k < 0 || n_emit < 0) return RLT_EINVAL;
  if (n_emit > 0 && (!emit_steps || !logits)) return RLT_EINVAL;
  for (int j = 0; j < n_emit; ++j)
    if (emit_steps[j] < 0 || emit_steps[j] >= n) return RLT_EINVAL;
  if (st->version != m->version) return RLT_ESTALE;
  if (st->pos < 0 || (int64_t)st->pos + n > T_mem) return RLT_ERANGE;
  if (ws_bytes < layout(m, st->batch, T_mem).total) return RLT_EWORKSPACE;
  if (n == 0) return RLT_OK;
  DecodeArgs A;
  A.e = e;
  A.mem = mem;
  A.T_mem = T_mem;
  A.n = n;
  A.actions = actions;
  A.inv_temp = 1.0f / temperature;
  A.top_k = top_k;
  A.logp = logp;
  A.logp_full = logp_full;
  A.argmax = argmax;
  A.logits = logits;
  A.n_emit = n_emit;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (m->decode_path == RLT_DECODE_FUSED) return decode_fused(m, st, A, emit_steps, ws, s);
  if (m->cfg.dtype == RLT_BF16) return decode_impl<bf16>(m, st, A, emit_steps, ws, s);
  return decode_impl<float>(m, st, A, emit_steps, ws, s);
}

int rlt_set_decode_path(rlt_model* m, int32_t path, int32_t cluster_size) {
  if (!m) return RLT_EINVAL;
  if (path != RLT_DECODE_AUTO && path != RLT_DECODE_GRAPH && path != RLT_DECODE_FUSED) return RLT_EINVAL;
  if (cluster_size != 0 && cluster_size != 1 && cluster_size != 2 && cluster_size != 4 && cluster_size != 8 &&
      cluster_size != 16)
    return RLT_EINVAL;
  m->decode_path = path;
  m->fused_cs = cluster_size;
  return RLT_OK;
}

int rlt_fused_plan(const rlt_model* m, int32_t B, int32_t* cluster_size, int32_t* seqs_per_cluster,
                   int32_t* clusters, int32_t* smem_bytes) {
  if (!m || B <= 0) return RLT_EINVAL;
  fused::Plan P;
  const int rc = fused_choose(m, B, &P);
  if (rc) return rc;
  if (cluster_size) *cluster_size = P.CS;
  if (seqs_per_cluster) *seqs_per_cluster = P.Bc;
  if (clusters) *clusters = P.nclu;
  if (smem_bytes) *smem_bytes = (int32_t)P.total;
  return RLT_OK;
}

int rlt_cross_attention(const rlt_model* m, const float* q, const void* mem_k, const void* mem_v, int32_t B,
                        int32_t T_mem, int32_t t, void* out, void* ws, size_t ws_bytes, rlt_stream_t stream) {
  if (!m || !q || !mem_k || !mem_v || !out || !ws || B <= 0 || T_mem <= 0 || t < 1 || t > T_mem)
    return RLT_EINVAL;
  if (!aligned16(q) || !aligned16(mem_k) || !aligned16(mem_v) || !aligned16(out) || !aligned16(ws)) return RLT_EINVAL;
  WsLayout Lw = layout(m, B, T_mem);
  if (ws_bytes < Lw.total) return RLT_EWORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const rlt_config& c = m->cfg;
  const int H = c.n_heads, hd = c.head_dim;
  StepCtx* ctx = at<StepCtx>(ws, Lw.ctx);
  float* part = at<float>(ws, Lw.d_part);
  XattnArgs xa{};
  xa.q = q;
  xa.mk = mem_k;
  xa.mv = mem_v;
  xa.part = part;
  xa.cnt = at<int>(ws, Lw.d_cnt);
  xa.out = out;
  xa.B = B;
  xa.H = H;
  xa.T_mem = T_mem;
  xa.t_cap = T_mem;
  xa.scale = 1.0f / sqrtf((float)hd);
  xa.ctx = ctx;
  xa.status = at<int>(ws, Lw.status);
  if (m->inject_kernel == RLT_KERNEL_XATTN) {  // one-shot (rlt_debug_withhold_copy)
    xa.budget = m->inject_budget;
    xa.withhold = 1;
    m->inject_kernel = 0;
  }
  set_ctx_kernel<<<1, 1, 0, s>>>(ctx, t - 1);
  RLT_CUDA_TRY(cudaMemsetAsync(xa.cnt, 0, sizeof(int) * (size_t)B * H, s));
  cudaError_t ce = (c.dtype == RLT_BF16) ? launch_xattn<bf16>(xa, hd, m->n_sm, s) : launch_xattn<float>(xa, hd, m->n_sm, s);
  if (ce != cudaSuccess) return RLT_ECUDA;
  g_launches += 2;
  return launch_ok();
}

int rlt_linear(const rlt_model* m, const void* A, int32_t lda, int32_t M, int32_t K, const void* W, const void* W3,
               int32_t ldw, int32_t N, float* C, int32_t ldc, void* ws, size_t ws_bytes, rlt_stream_t stream) {
  if (!m || !A || !W || !C || !ws || M <= 0 || K <= 0 || N <= 0 || lda < K || ldw < K || ldc < N) return RLT_EINVAL;
  if (m->cfg.dtype != RLT_BF16) return RLT_EUNSUPPORTED;
  if (!aligned16(A) || !aligned16(W) || (W3 && !aligned16(W3)) || !aligned16(ws) || lda % 8 || ldw % 8)
    return RLT_EINVAL;
  WsLayout Lw = layout(m, 1, 1);
  if (ws_bytes < Lw.total) return RLT_EWORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  TcScratch sc = tc_scratch(m, ws, Lw);
  if (m->inject_kernel == RLT_KERNEL_GEMM) {  // one-shot (rlt_debug_withhold_copy)
    sc.budget = m->inject_budget;
    sc.withhold = 1;
    m->inject_kernel = 0;
  }
  AArg a;
  a.A = static_cast<const bf16*>(A);
  a.lda = lda;
  const bf16* w = static_cast<const bf16*>(W);
  if (W3)
    return proj_bf16<true>(s, a, M, K, w, static_cast<const bf16*>(W3), ldw, N, EpiStoreF32{C, ldc}, sc);
  return proj_bf16<false>(s, a, M, K, w, nullptr, ldw, N, EpiStoreF32{C, ldc}, sc);
}

int rlt_debug_withhold_copy(rlt_model* m, int32_t kernel, int64_t budget_cycles) {
  if (!m || (kernel != RLT_KERNEL_XATTN && kernel != RLT_KERNEL_GEMM && kernel != RLT_KERNEL_NORM_PROJ) ||
      budget_cycles < 1000 || budget_cycles > 4000000000LL)
    return RLT_EINVAL;
  if (kernel != RLT_KERNEL_XATTN && m->cfg.dtype != RLT_BF16) return RLT_EUNSUPPORTED;
  m->inject_budget = budget_cycles;
  m->inject_kernel = kernel;
  return RLT_OK;
}

int rlt_status(void* ws, rlt_stream_t stream) {
  if (!ws) return RLT_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return RLT_ECUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return RLT_ECUDA;
  if (v != 0) {
    int z = 0;
    if (cudaMemcpy(ws, &z, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return RLT_ECUDA;
  }
  return v;
}

}  // extern "C"

// backpropagation through time of the decoder (rlt_bptt)
#include "bptt_api.cuh"
