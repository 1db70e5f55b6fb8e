// Stand-ins, under the host emulation (emu.h), for the PTX operations of the
// persistent cluster decoder (the library's fused_ptx.cuh): cluster rank and
// barrier, another block's shared memory, the 16-byte asynchronous copy
// (done at once, zero-filled past the source bytes), the L2 prefetch (no
// effect) and the warp-level m16n8k16 bf16 MMA, computed from the fragment
// layout the PTX ISA documents for it: A row g = lane / 4 (+ 8 for registers
// 1 and 3), columns 2 (lane % 4) + {0, 1} (+ 8 for registers 2 and 3);
// B column lane / 4, rows 2 (lane % 4) + {0, 1} (+ 8 for register 1);
// D row lane / 4 (+ 8 for elements 2, 3), columns 2 (lane % 4) + {0, 1}.
// Each 32-bit register holds two bf16, the lower column in the low half.
// Test infrastructure only.
#pragma once
#include <optional>
#include "emu.h"

namespace rlt {
namespace fused {

inline unsigned cluster_rank() { return emu_rank; }
inline void cluster_sync() {
  emu_cluster_bar->arrive_and_wait();
  if (emu_jitter()) emu_jitter_sleep();
}
inline thread_local std::optional<std::barrier<>::arrival_token> emu_cluster_token;
inline void cluster_arrive() { emu_cluster_token.emplace(emu_cluster_bar->arrive()); }
inline void cluster_wait() {
  emu_cluster_bar->wait(std::move(*emu_cluster_token));
  emu_cluster_token.reset();
  if (emu_jitter()) emu_jitter_sleep();
}
template <class T>
inline T* map_rank(T* p, unsigned rank) {
  return reinterpret_cast<T*>(emu_cluster_smem[rank] + (reinterpret_cast<char*>(p) - emu_tl_smem));
}
inline void cp_async16(void* smem, const void* gmem, int src_bytes) {
  memset(smem, 0, 16);
  if (src_bytes > 0) memcpy(smem, gmem, (size_t)src_bytes);
}
inline void cp_async_commit() {}
inline void cp_async_wait1() {}
inline void cp_async_wait0() {}
inline void prefetch_l2(const void*, unsigned) {}

inline float emu_bf16_half(unsigned v, int hi) {
  const unsigned u = hi ? (v & 0xffff0000u) : (v << 16);
  float f;
  memcpy(&f, &u, 4);
  return f;
}
inline void mma_bf16(float (&d)[4], const unsigned (&a)[4], const unsigned (&b)[2]) {
  auto& w = (*emu_warps)[emu_warp];
  for (int q = 0; q < 4; ++q) w.ma[emu_lane][q] = a[q];
  w.mb[emu_lane][0] = b[0];
  w.mb[emu_lane][1] = b[1];
  w.bar->arrive_and_wait();
  auto A = [&](int row, int k) {
    return emu_bf16_half(w.ma[(row % 8) * 4 + (k % 8) / 2][row / 8 + 2 * (k / 8)], k % 2);
  };
  auto Bv = [&](int k, int col) { return emu_bf16_half(w.mb[col * 4 + (k % 8) / 2][k / 8], k % 2); };
  const int g = emu_lane >> 2, c = emu_lane & 3;
  float r[4];
  for (int q = 0; q < 4; ++q) {
    const int row = g + 8 * (q >> 1), col = 2 * c + (q & 1);
    float acc = d[q];
    for (int k = 0; k < 16; ++k) acc += A(row, k) * Bv(k, col);
    r[q] = acc;
  }
  w.bar->arrive_and_wait();
  for (int q = 0; q < 4; ++q) d[q] = r[q];
}

inline uint4 ld_nc16(const void* p) {
  uint4 v;
  memcpy(&v, p, 16);
  return v;
}
inline uint4 ld_cg16(const void* p) { return ld_nc16(p); }
inline float4 ld_nc_f4(const float* p) {
  float4 v;
  std::memcpy(&v, p, 16);
  return v;
}
inline bf16 ld_cg_bf16(const bf16* p) { return *p; }

}  // namespace fused
}  // namespace rlt
