// Runs the forward head kernel (head_reduce_kernel of kernels.cuh: log-
// probabilities over the tempered vocabulary, the top-k set by radix select,
// argmax, and the sampling draw) under the host emulation of emu.h, one step
// of n = 1.  The generated input kernels_emu.cuh comes from the test:
// kernels.cuh with the programmatic-launch waits as no-ops and its dynamic
// shared arrays taken from the emulator.  Test infrastructure only.
#include "emu.h"
#include "cuda_bf16.h"
#include <vector>
#include "kernels_emu.cuh"

using namespace rlt;

// logits [B][V] fp32, actions [B]; outputs logp, logp_full, argmax [B]; with
// sample != 0 the action is drawn (uniform of (seed, b, pos)) into next_tok [B]
extern "C" int head_emu(const float* logits, const int* actions, int B, int V, float inv_temp, int top_k, int sample,
                        unsigned long long seed, int pos, float* logp, float* logp_full, int* argmax, int* next_tok) {
  std::vector<float> lg(logits, logits + (size_t)B * V);
  std::vector<int> act(actions, actions + B);
  std::vector<int> emit(1, -1);
  int status = 0;
  StepCtx ctx{};
  ctx.step = 0;
  ctx.pos = pos;
  HeadArgs a{};
  a.logits = lg.data();
  a.actions = sample ? nullptr : act.data();
  a.logp = logp;
  a.logp_full = logp_full;
  a.argmax = argmax;
  a.emit_map = emit.data();
  a.B = B;
  a.V = V;
  a.n = 1;
  a.top_k = top_k;
  a.inv_temp = inv_temp;
  a.status = &status;
  a.next_tok = sample ? next_tok : nullptr;
  a.seed = seed;
  emu_launch(dim3(B), dim3(1024), sizeof(float) * V, head_reduce_kernel, a, (const StepCtx*)&ctx);
  return status;
}
