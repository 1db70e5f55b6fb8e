// A host emulation of the CUDA execution model, for testing the index logic
// of plain CUDA kernels without a GPU: one host thread per CUDA thread,
// blocks run one after another, __syncthreads and warp shuffles are
// barriers, __shared__ becomes static storage (one block at a time).  Test
// infrastructure only: results obtained here are not GPU parity.
#pragma once
#include <atomic>
#include <barrier>
#include <chrono>
#include <cstdlib>
#include <semaphore>
#include <condition_variable>
#include <mutex>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <memory>
#include <thread>
#include <vector>
#include <algorithm>

struct dim3 {
  unsigned x = 1, y = 1, z = 1;
  dim3(unsigned a = 1, unsigned b = 1, unsigned c = 1) : x(a), y(b), z(c) {}
};
typedef struct CUstream_st* cudaStream_t;
typedef int cudaError_t;
constexpr int cudaSuccess = 0;
// host set-up calls of the library's headers: one device, index 0
inline cudaError_t cudaGetDevice(int* dev) {
  *dev = 0;
  return cudaSuccess;
}

inline thread_local dim3 threadIdx, blockIdx;
inline dim3 blockDim, gridDim;
inline thread_local int emu_lane = 0, emu_warp = 0;

struct EmuWarp {
  std::unique_ptr<std::barrier<>> bar;
  float f[32];
  int i[32];
  unsigned u[32];
  unsigned ma[32][4], mb[32][2];  // warp-level MMA operands
};
// the calling thread's block: its warps, block barrier and dynamic shared
// memory; with cluster launches also its rank, the cluster barrier and every
// block's shared memory
inline thread_local std::vector<EmuWarp>* emu_warps = nullptr;
inline thread_local std::barrier<>* emu_block_bar = nullptr;
inline thread_local char* emu_tl_smem = nullptr;
inline thread_local unsigned emu_rank = 0;
inline thread_local std::barrier<>* emu_cluster_bar = nullptr;
inline thread_local char* const* emu_cluster_smem = nullptr;
inline std::vector<char> emu_dyn;
#define __align__(n) __attribute__((aligned(n)))

#define __global__
#define __device__
#define __host__
#define __forceinline__ inline
#define __restrict__ __restrict
#define __shared__ static
#define __launch_bounds__(...)
#define __grid_constant__

// EMU_JITTER=1 in the environment: every thread sleeps a random 0-63 us after
// each block or cluster barrier, so that threads leave barriers in a
// scrambled order and an access that is not ordered by a barrier shows as a
// result that differs from run to run.
inline bool emu_jitter() {
  static const bool on = [] {
    const char* v = std::getenv("EMU_JITTER");
    return v && v[0] == '1';
  }();
  return on;
}
inline void emu_jitter_sleep() {
  thread_local unsigned x = 0x9e3779b9u ^ (unsigned)(uintptr_t)&x;
  x ^= x << 13;
  x ^= x >> 17;
  x ^= x << 5;
  std::this_thread::sleep_for(std::chrono::microseconds(x & 63u));
}
inline void __syncthreads() {
  emu_block_bar->arrive_and_wait();
  if (emu_jitter()) emu_jitter_sleep();
}
inline void __syncwarp(unsigned = 0xffffffffu) { (*emu_warps)[emu_warp].bar->arrive_and_wait(); }
inline float __shfl_xor_sync(unsigned, float v, int m) {
  auto& w = (*emu_warps)[emu_warp];
  w.f[emu_lane] = v;
  w.bar->arrive_and_wait();
  float r = w.f[emu_lane ^ m];
  w.bar->arrive_and_wait();
  return r;
}
inline int __shfl_xor_sync(unsigned, int v, int m) {
  auto& w = (*emu_warps)[emu_warp];
  w.i[emu_lane] = v;
  w.bar->arrive_and_wait();
  int r = w.i[emu_lane ^ m];
  w.bar->arrive_and_wait();
  return r;
}
inline float __shfl_sync(unsigned, float v, int src) {
  auto& w = (*emu_warps)[emu_warp];
  w.f[emu_lane] = v;
  w.bar->arrive_and_wait();
  float r = w.f[src & 31];
  w.bar->arrive_and_wait();
  return r;
}
inline int __shfl_sync(unsigned, int v, int src) {
  auto& w = (*emu_warps)[emu_warp];
  w.i[emu_lane] = v;
  w.bar->arrive_and_wait();
  int r = w.i[src & 31];
  w.bar->arrive_and_wait();
  return r;
}
// lanes of the warp holding the same value (full warps only)
inline unsigned __match_any_sync(unsigned, int v) {
  auto& w = (*emu_warps)[emu_warp];
  w.i[emu_lane] = v;
  w.bar->arrive_and_wait();
  unsigned m = 0;
  for (int l = 0; l < 32; ++l)
    if (w.i[l] == v) m |= 1u << l;
  w.bar->arrive_and_wait();
  return m;
}
inline int __ffs(unsigned x) { return x ? __builtin_ctz(x) + 1 : 0; }
inline int __popc(unsigned x) { return __builtin_popcount(x); }
inline unsigned atomicAdd(unsigned* p, unsigned v) { return std::atomic_ref<unsigned>(*p).fetch_add(v); }
inline int atomicCAS(int* p, int cmp, int val) {
  std::atomic_ref<int> a(*p);
  int c = cmp;
  a.compare_exchange_strong(c, val);
  return c;
}
inline unsigned __float_as_uint(float x) { unsigned u; memcpy(&u, &x, 4); return u; }
inline float __uint_as_float(unsigned u) { float x; memcpy(&x, &u, 4); return x; }
inline float __int_as_float(int u) { float x; memcpy(&x, &u, 4); return x; }
inline int __float_as_int(float x) { int u; memcpy(&u, &x, 4); return u; }
inline float rsqrtf(float x) { return 1.0f / std::sqrt(x); }
inline float __expf(float x) { return std::exp(x); }
inline void sincos(double a, double* s, double* c) { *s = std::sin(a); *c = std::cos(a); }
using std::min;
using std::max;

template <class T> T* emu_dyn_smem() { return reinterpret_cast<T*>(emu_tl_smem); }

// A pool of persistent host threads, one per CUDA thread slot of a block (or
// of a cluster); run(n, f) calls f(t) on threads t < n and returns when all
// of them are done.  Only the n threads a launch uses are woken.
struct EmuPool {
  std::vector<std::thread> th;
  std::vector<std::unique_ptr<std::binary_semaphore>> go;
  std::mutex mu;
  std::condition_variable done_cv;
  std::function<void(unsigned)> job;
  unsigned active = 0;
  bool stop = false;
  explicit EmuPool(unsigned n) {
    for (unsigned t = 0; t < n; ++t) go.push_back(std::make_unique<std::binary_semaphore>(0));
    for (unsigned t = 0; t < n; ++t)
      th.emplace_back([this, t]() {
        for (;;) {
          go[t]->acquire();
          if (stop) return;
          job(t);
          std::lock_guard<std::mutex> lk(mu);
          if (--active == 0) done_cv.notify_all();
        }
      });
  }
  ~EmuPool() {
    stop = true;
    for (auto& g : go) g->release();
    for (auto& x : th) x.join();
  }
  void run(unsigned n, std::function<void(unsigned)> f) {
    job = std::move(f);
    {
      std::lock_guard<std::mutex> lk(mu);
      active = n;
    }
    for (unsigned t = 0; t < n; ++t) go[t]->release();
    std::unique_lock<std::mutex> lk(mu);
    done_cv.wait(lk, [&] { return active == 0; });
  }
};
inline EmuPool& emu_pool() {
  static EmuPool pool(4096);
  return pool;
}

// Runs kernel(args...) over grid x block, one pool thread per CUDA thread,
// blocks one after another.  Threads leave the barriers when they return.
template <class F, class... A>
void emu_launch(dim3 grid, dim3 block, size_t smem, F kernel, A... args) {
  gridDim = grid;
  blockDim = block;
  const unsigned nthr = block.x * block.y * block.z;
  const unsigned nw = (nthr + 31) / 32;
  emu_dyn.assign(smem + 16, 0);
  for (unsigned bz = 0; bz < grid.z; ++bz)
    for (unsigned by = 0; by < grid.y; ++by)
      for (unsigned bx = 0; bx < grid.x; ++bx) {
        std::vector<EmuWarp> warps(nw);
        for (unsigned w = 0; w < nw; ++w)
          warps[w].bar = std::make_unique<std::barrier<>>(std::min(32u, nthr - 32 * w));
        std::barrier<> bb(nthr);
        emu_pool().run(nthr, [&](unsigned t) {
          emu_warps = &warps;
          emu_block_bar = &bb;
          emu_tl_smem = emu_dyn.data();
          threadIdx = dim3(t % block.x, (t / block.x) % block.y, t / (block.x * block.y));
          blockIdx = dim3(bx, by, bz);
          emu_lane = t % 32;
          emu_warp = t / 32;
          kernel(args...);
          (*emu_warps)[emu_warp].bar->arrive_and_drop();
          emu_block_bar->arrive_and_drop();
        });
      }
}

// Runs kernel(args...) over a 1-D grid of clusters of CS blocks: clusters
// one after another, the blocks of a cluster concurrently, each with its own
// dynamic shared memory (filled with 0xff bytes, NaN as floats, so that a
// read of memory the kernel did not initialise shows).
template <class F, class... A>
void emu_launch_cluster(dim3 grid, dim3 block, size_t smem, unsigned CS, F kernel, A... args) {
  gridDim = grid;
  blockDim = block;
  const unsigned nthr = block.x * block.y * block.z;
  const unsigned nw = (nthr + 31) / 32;
  std::vector<std::vector<char>> bufs(CS, std::vector<char>(smem + 16));
  std::vector<char*> bases(CS);
  for (unsigned c = 0; c < CS; ++c) bases[c] = bufs[c].data();
  for (unsigned cl = 0; cl < grid.x / CS; ++cl) {
    for (auto& b : bufs) std::fill(b.begin(), b.end(), (char)0xff);
    std::vector<std::vector<EmuWarp>> warps(CS);
    std::vector<std::unique_ptr<std::barrier<>>> bbs;
    for (unsigned c = 0; c < CS; ++c) {
      warps[c] = std::vector<EmuWarp>(nw);
      for (unsigned w = 0; w < nw; ++w)
        warps[c][w].bar = std::make_unique<std::barrier<>>(std::min(32u, nthr - 32 * w));
      bbs.push_back(std::make_unique<std::barrier<>>(nthr));
    }
    std::barrier<> cb(CS * nthr);
    emu_pool().run(CS * nthr, [&](unsigned tt) {
      const unsigned rk = tt / nthr, t = tt % nthr;
      emu_warps = &warps[rk];
      emu_block_bar = bbs[rk].get();
      emu_tl_smem = bases[rk];
      emu_rank = rk;
      emu_cluster_bar = &cb;
      emu_cluster_smem = bases.data();
      threadIdx = dim3(t % block.x, (t / block.x) % block.y, t / (block.x * block.y));
      blockIdx = dim3(cl * CS + rk, 0, 0);
      emu_lane = t % 32;
      emu_warp = t / 32;
      kernel(args...);
      (*emu_warps)[emu_warp].bar->arrive_and_drop();
      emu_block_bar->arrive_and_drop();
      emu_cluster_bar->arrive_and_drop();
    });
  }
}

struct float2 { float x, y; };
struct float4 { float x, y, z, w; };
struct uint2 { unsigned x, y; };
struct uint4 { unsigned x, y, z, w; };
inline uint4 make_uint4(unsigned a, unsigned b, unsigned c, unsigned d) { return uint4{a, b, c, d}; }
inline float2 make_float2(float a, float b) { return float2{a, b}; }
inline float4 make_float4(float a, float b, float c, float d) { return float4{a, b, c, d}; }
