// Cross-attention entry point for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside another
// framework's allocator regime, embedders that forbid allocation after start-up,
// or hosts that only hand out input and output buffers.  rlt_cross_attention
// needs a caller-provided workspace for its per-chunk partial results and
// arrival counters; this variant keeps those (and its small step context) in
// one fixed array compiled into the library instead, so the caller passes only
// q, the memory planes and the output.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its kNoAllocScratchBytes until the process exits.  In host
// code the array's name only stands for the symbol; its device address is
// obtained once per device with cudaGetSymbolAddress (with that device
// current) on the first call made on that device, which is why that first call
// should come before any stream capture.  The address is kept for the life of
// the process, so the entry point must not be used on a device after a
// cudaDeviceReset (or other teardown of the device's primary context) in the
// same process.  All calls share the array; each call clears the arrival
// counters it uses (the partials need no clearing: every partial that is read
// was written by the same call); calls that overlap on the GPU race on it.
// A bounded wait that gives up inside the kernel records RLT_ETIMEOUT in a
// status word of the array (the first condition wins); the call itself
// returns before the kernel runs, so the word is read (and cleared) with
// rlt_cross_attention_noalloc_status.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/rlt.h"
#include "common.cuh"
#include "ptx.cuh"

// This translation unit compiles its own copy of the kernels, in a private
// namespace, so that its kernel symbols do not collide with the library's.
namespace rlt_noalloc {
using namespace ::rlt;
#include "kernels.cuh"
#include "xattn.cuh"
}  // namespace rlt_noalloc

using namespace ::rlt;
using rlt_noalloc::rlt::kXMaxSplits;
using rlt_noalloc::rlt::launch_xattn;
using rlt_noalloc::rlt::set_ctx_kernel;
using rlt_noalloc::rlt::XattnArgs;

namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB
constexpr size_t kCtxBytes = 256;                    // step context + status word at the start of the array
constexpr size_t kStatusOffset = 128;                // the status word (zero in a freshly loaded module)
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
int g_n_sm[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on the
// first call per device).
int scratch_on_current_device(void** out, int* n_sm) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RLT_ECUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return RLT_ECUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
      return RLT_ECUDA;
    g_n_sm[dev] = sms;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  *n_sm = g_n_sm[dev];
  return RLT_OK;
}

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" {

int rlt_cross_attention_noalloc_status(rlt_stream_t stream) {
  void* base = nullptr;
  int n_sm = 0;
  int rc = scratch_on_current_device(&base, &n_sm);
  if (rc) return rc;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return RLT_ECUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_noalloc_scratch, sizeof(int), kStatusOffset, cudaMemcpyDeviceToHost) != cudaSuccess)
    return RLT_ECUDA;
  if (v != 0) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_noalloc_scratch, &z, sizeof(int), kStatusOffset, cudaMemcpyHostToDevice) != cudaSuccess)
      return RLT_ECUDA;
  }
  return v;
}

int rlt_cross_attention_noalloc(const float* q, const void* mem_k, const void* mem_v, int32_t B, int32_t n_heads,
                                int32_t head_dim, int32_t dtype, int32_t T_mem, int32_t t, void* out,
                                rlt_stream_t stream) {
  if (!q || !mem_k || !mem_v || !out || B <= 0 || n_heads <= 0 || T_mem <= 0 || t < 1 || t > T_mem)
    return RLT_EINVAL;
  if (dtype != RLT_F32 && dtype != RLT_BF16) return RLT_EINVAL;
  if (head_dim < 8 || head_dim % 8 != 0 || 128 % head_dim != 0) return RLT_EUNSUPPORTED;
  if (!aligned16(q) || !aligned16(mem_k) || !aligned16(mem_v) || !aligned16(out)) return RLT_EINVAL;
  const size_t pairs = (size_t)B * n_heads;
  const size_t cnt_bytes = (sizeof(int) * pairs + 255) / 256 * 256;
  const size_t part_bytes = sizeof(float) * pairs * kXMaxSplits * (head_dim + 2);
  if (cnt_bytes + part_bytes > kNoAllocScratchBytes - kCtxBytes) return RLT_EUNSUPPORTED;  // beyond the built-in scratch
  void* base = nullptr;
  int n_sm = 0;
  int rc = scratch_on_current_device(&base, &n_sm);
  if (rc) return rc;
  unsigned char* sb = static_cast<unsigned char*>(base);
  StepCtx* ctx = reinterpret_cast<StepCtx*>(sb);
  int* status = reinterpret_cast<int*>(sb + kStatusOffset);
  int* cnt = reinterpret_cast<int*>(sb + kCtxBytes);
  float* part = reinterpret_cast<float*>(sb + kCtxBytes + cnt_bytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  XattnArgs xa{};
  xa.q = q;
  xa.mk = mem_k;
  xa.mv = mem_v;
  xa.part = part;
  xa.cnt = cnt;
  xa.out = out;
  xa.B = B;
  xa.H = n_heads;
  xa.T_mem = T_mem;
  xa.t_cap = T_mem;
  xa.scale = 1.0f / sqrtf((float)head_dim);
  xa.ctx = ctx;
  xa.status = status;
  set_ctx_kernel<<<1, 1, 0, s>>>(ctx, t - 1);
  if (cudaMemsetAsync(cnt, 0, sizeof(int) * pairs, s) != cudaSuccess) return RLT_ECUDA;
  cudaError_t ce = (dtype == RLT_BF16) ? launch_xattn<bf16>(xa, head_dim, n_sm, s)
                                       : launch_xattn<float>(xa, head_dim, n_sm, s);
  if (ce != cudaSuccess) return RLT_ECUDA;
  return cudaGetLastError() == cudaSuccess ? RLT_OK : RLT_ECUDA;
}

}  // extern "C"
