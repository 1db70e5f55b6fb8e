// Token selection shared by the head kernels (kernels.cuh) and the
// persistent decoder (dec_fused.cuh): the order-preserving key of a float,
// the counter-based uniform number of a draw, and the draw from the tempered
// (top-k) distribution.
#pragma once
#include "common.cuh"

namespace rlt {

// Order-preserving unsigned key of a float (larger float, larger key).
__device__ __forceinline__ unsigned f2key(float x) {
  unsigned u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Uniform draw in [0, 1) with 24 random bits for (seed, sequence b, position
// pos): the SplitMix64 output function (Steele, Lea and Flood, "Fast
// splittable pseudorandom number generators", 2014) applied to the counter
// seed + (pos * 2^32 + b + 1) * golden gamma.  Depends on the absolute
// position, not on how generation is split into calls.
__device__ __forceinline__ float uniform24(unsigned long long seed, int b, int pos) {
  unsigned long long z = seed + (((unsigned long long)(unsigned)pos << 32) + (unsigned)b + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return (float)(z >> 40) * (1.0f / 16777216.0f);
}

// Draws a token from the tempered distribution over the set S: every token
// (all), or the top-k set - keys (f2key of the tempered logit) above kth, and
// the first `need` tokens in id order whose key equals kth.  The weights
// exp(x - mx) are accumulated in token-id order in a fixed fp32 order: thread
// t sums the contiguous id chunk [t C, (t + 1) C), thread 0 adds the chunk
// sums up and finds the chunk where the running sum passes u times the total,
// and that chunk's thread walks its ids to the first one whose running sum
// exceeds it (the chunk's last member when rounding leaves none).  All threads
// of the block call it; it returns the token in every thread.
__device__ int sample_chunked(const float* sx, int V, float mx, bool all, unsigned kth, unsigned need, float u,
                              float* s_part, unsigned* s_tie, int* s_res) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int C = (V + nthr - 1) / nthr;
  const int v0 = min(V, tid * C), v1 = min(V, v0 + C);
  unsigned ties = 0;
  if (!all)
    for (int v = v0; v < v1; ++v) ties += (f2key(sx[v]) == kth) ? 1u : 0u;
  s_tie[tid] = ties;
  __syncthreads();
  if (tid == 0) {  // s_tie[t] := ties at kth in the chunks before t
    unsigned acc = 0;
    for (int t = 0; t < nthr; ++t) {
      const unsigned c = s_tie[t];
      s_tie[t] = acc;
      acc += c;
    }
  }
  __syncthreads();
  auto member = [&](unsigned kk, unsigned& tb) {
    if (all || kk > kth) return true;
    if (kk != kth) return false;
    return tb++ < need;
  };
  unsigned tb = s_tie[tid];
  float sum = 0.f;
  for (int v = v0; v < v1; ++v)
    if (member(f2key(sx[v]), tb)) sum += expf(sx[v] - mx);
  s_part[tid] = sum;
  __syncthreads();
  if (tid == 0) {
    s_res[4] = 0;  // kept only if no chunk holds a member (non-finite logits)
    float tot = 0.f;
    for (int t = 0; t < nthr; ++t) tot += s_part[t];
    const float target = u * tot;
    float run = 0.f;
    int tstar = -1, tlast = -1;
    for (int t = 0; t < nthr; ++t) {
      if (s_part[t] > 0.f) tlast = t;
      if (tstar < 0) {
        if (s_part[t] > 0.f && run + s_part[t] > target)
          tstar = t;
        else
          run += s_part[t];
      }
    }
    int last = 0;
    if (tstar < 0) {  // rounding: the last member overall
      tstar = tlast;
      last = 1;
    }
    s_res[0] = tstar;
    s_res[1] = last;
    s_res[2] = __float_as_int(run);
    s_res[3] = __float_as_int(target);
  }
  __syncthreads();
  if (s_res[0] >= 0 && tid == s_res[0]) {
    const bool last = s_res[1] != 0;
    float run = __int_as_float(s_res[2]);
    const float target = __int_as_float(s_res[3]);
    unsigned tb2 = s_tie[tid];
    int pick = -1, lastm = -1;
    for (int v = v0; v < v1; ++v) {
      if (!member(f2key(sx[v]), tb2)) continue;
      lastm = v;
      if (!last && pick < 0) {
        run += expf(sx[v] - mx);
        if (run > target) pick = v;
      }
    }
    if (pick >= 0 || lastm >= 0) s_res[4] = pick >= 0 ? pick : lastm;
  }
  __syncthreads();
  return min(max(s_res[4], 0), V - 1);
}

}  // namespace rlt
