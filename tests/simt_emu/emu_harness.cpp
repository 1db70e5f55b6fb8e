// Runs the library's bpplan::run with the device kernels of bptt.cuh under
// the host emulation of emu.h; the projections run as a reference loop into
// the same epilogue functors (the tensor-core kernel is inline PTX and is not
// emulated; both GEMM kernels are covered by the forward's GPU tests).  The two generated inputs come
// from the test: bptt_emu.cuh (bptt.cuh with its dynamic shared array taken
// from the emulator) and emu_ops.inc (the device Ops of bptt_api.cuh with
// each kernel launch turned into emu_launch).  Test infrastructure only.
#include "emu.h"
#include "cuda_bf16.h"
#include <mutex>
#include <type_traits>
#include "bptt_emu.cuh"
#include "gemm_simple.cuh"
#include "bptt_plan.h"

using namespace rlt;
constexpr int RLT_OK = 0, RLT_ECUDA = -4;
constexpr int cudaMemcpyDeviceToDevice = 3;
inline std::atomic<uint64_t> g_launches{0};
inline int launch_ok() { return RLT_OK; }
inline unsigned cdiv(size_t a, size_t b) { return (unsigned)((a + b - 1) / b); }
inline int cudaMemsetAsync(void* p, int v, size_t n, cudaStream_t) { memset(p, v, n); return cudaSuccess; }
inline int cudaMemcpyAsync(void* d, const void* s, size_t n, int, cudaStream_t) { memmove(d, s, n); return cudaSuccess; }
struct TcScratch { int n_sm; int* status; const int (*maxc)[9]; };
// graph capture is not emulated: the harness runs the steps eagerly (these
// stand-ins only let the capture path compile)
typedef struct GraphStub* cudaGraph_t;
typedef struct GraphExecStub* cudaGraphExec_t;
constexpr int cudaStreamCaptureModeThreadLocal = 1;
inline int cudaStreamBeginCapture(cudaStream_t, int) { return -1; }
inline int cudaStreamEndCapture(cudaStream_t, cudaGraph_t*) { return -1; }
inline int cudaGraphInstantiate(cudaGraphExec_t*, cudaGraph_t, int) { return -1; }
inline int cudaGraphDestroy(cudaGraph_t) { return 0; }
inline int cudaGraphLaunch(cudaGraphExec_t, cudaStream_t) { return -1; }
inline int cudaGraphExecDestroy(cudaGraphExec_t) { return 0; }
#define RLT_CUDA_TRY(x)                         \
  do {                                          \
    if ((x) != cudaSuccess) return RLT_ECUDA;   \
  } while (0)
struct AArg { const bf16* A; int lda; };
__global__ void bcast_rows_kernel(float* dst, const float* src, int rows, int d) {
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < (size_t)rows * d) dst[i] = src[i % d];
}
// Projections: a reference loop that hands every output element to the
// epilogue functor, as both GEMM kernels do (the GEMM kernels themselves are
// covered by the forward path's GPU tests).
template <typename T_, class Epi>
int gemm(cudaStream_t, const T_* A, int lda, GemmB gb, int M, int N, int K, Epi epi) {
  const float* W = static_cast<const float*>(gb.B0);
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n) {
      float acc = 0.f;
      for (int k = 0; k < K; ++k) acc = fmaf(A[(size_t)m * lda + k], W[(size_t)n * gb.ldb + k], acc);
      epi(m, n, acc);
    }
  return RLT_OK;
}
template <bool GLU, class Epi>
int proj_bf16(cudaStream_t, const AArg& a, int M, int K, const bf16* W, const bf16*, int ldw, int N, Epi epi,
              const TcScratch&) {
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n) {
      float acc = 0.f;
      for (int k = 0; k < K; ++k) acc += __bfloat162float(a.A[(size_t)m * a.lda + k]) * __bfloat162float(W[(size_t)n * ldw + k]);
      epi(m, n, acc);
    }
  return RLT_OK;
}
namespace {
#include "emu_ops.inc"
}

template <typename T>
static std::vector<T> conv(const float* x, size_t n) {
  std::vector<T> v(n);
  for (size_t i = 0; i < n; ++i) {
    if constexpr (std::is_same<T, float>::value) v[i] = x[i];
    else v[i] = __float2bfloat16_rn(x[i]);
  }
  return v;
}

template <typename T>
static int run_emu(const int* sh, const float* fp, void** P, const size_t* nel) {
  bpplan::Shape S{};
  S.B = sh[0]; S.n = sh[1]; S.T_mem = sh[2]; S.d = sh[3]; S.H = sh[4]; S.hd = sh[5]; S.f = sh[6]; S.L = sh[7];
  S.W = sh[8]; S.V = sh[9]; S.G = sh[10]; S.gate_learned = sh[11] != 0; S.top_k = sh[12];
  S.eps = fp[0]; S.theta = fp[1]; S.scale = 1.0f / std::sqrt((float)S.hd); S.inv_temp = 1.0f / fp[2];
  const bool bf = std::is_same<T, bf16>::value;
  S.Bp = bf ? (S.B + 63) / 64 * 64 : S.B;
  S.S = sh[16];
  S.chunk = bptt::kAttnChunk;  // the partials scratch is sized for the kernels' key split
  bpplan::Detach D{sh[13], sh[14] != 0, sh[15] != 0};
  // matrices in the storage type (indices 0..8 and e, mem), the rest fp32
  std::vector<std::vector<T>> keepT;
  auto tm = [&](int i) { keepT.push_back(conv<T>((const float*)P[i], nel[i])); return (const T*)keepT.back().data(); };
  const T* Wg = tm(0); const T* Wqkv = tm(1); const T* WO = tm(2); const T* WQx = tm(3); const T* WOx = tm(4);
  const T* W1 = tm(5); const T* W3 = tm(6); const T* W2 = tm(7); const T* Wo = tm(8);
  bpplan::Params<T> Pp{Wg, Wqkv, WO, WQx, WOx, W1, W3, W2, Wo, (const float*)P[9], (const float*)P[10],
                       (const float*)P[11], (const float*)P[12], (const float*)P[13], (const float*)P[14]};
  const T* e = tm(15); const T* mem = tm(16);
  bpplan::Io<T> io{e, mem, (const int32_t*)P[17], (float*)P[18], (float*)P[19], (float*)P[35], (float*)P[36]};
  bpplan::Grads G{(float*)P[20], (float*)P[21], (float*)P[22], (float*)P[23], (float*)P[24], (float*)P[25],
                  (float*)P[26], (float*)P[27], (float*)P[28], (float*)P[29], (float*)P[30], (float*)P[31],
                  (float*)P[32], (float*)P[33], (float*)P[34]};
  const bpplan::Layout Lw = bpplan::layout(S, sizeof(T), 256);
  std::vector<double> ws((Lw.total + 7) / 8, 0.0);
  EmuOps<T> k;
  k.st = nullptr;
  k.user = nullptr;
  k.cap = nullptr;
  k.graphs = false;
  k.status = reinterpret_cast<int*>(ws.data());
  return bpplan::run(k, S, D, Pp, io, G, reinterpret_cast<char*>(ws.data()), Lw);
}

extern "C" int bptt_emu(const int* sh, const float* fp, void** P, const size_t* nel) {
  return sh[17] ? run_emu<bf16>(sh, fp, P, nel) : run_emu<float>(sh, fp, P, nel);
}
