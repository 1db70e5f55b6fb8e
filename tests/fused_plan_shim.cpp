// Host-side shim over the fused decoder's plan (fused_plan.h) for the CPU
// tests: make_plan and choose_plan with a given table of co-resident clusters
// per cluster size.  Test infrastructure only.
#include "fused_plan.h"

using namespace rlt::fused;

// shape: d, H, hd, f, L, W, V, G, gate.  mac[i]: co-resident clusters of
// 2^i CTAs (i = 0..4).  out: CS, Bc, nclu, cols, hpc, gph, npairs, total bytes.
extern "C" int plan_choose(const int* shape, int B, int force, const int* mac, long long* out) {
  const Shape s{shape[0], shape[1], shape[2], shape[3], shape[4], shape[5], shape[6], shape[7], shape[8]};
  Plan p;
  auto mc = [&](int CS, size_t) { return mac[CS == 16 ? 4 : CS == 8 ? 3 : CS == 4 ? 2 : CS == 2 ? 1 : 0]; };
  if (choose_plan(s, B, force, mc, &p)) return -1;
  const long long v[8] = {p.CS, p.Bc, p.nclu, p.cols, p.hpc, p.gph, p.npairs, (long long)p.total};
  for (int i = 0; i < 8; ++i) out[i] = v[i];
  return 0;
}

extern "C" int plan_make(const int* shape, int B, int CS, int Bc, long long* out) {
  const Shape s{shape[0], shape[1], shape[2], shape[3], shape[4], shape[5], shape[6], shape[7], shape[8]};
  Plan p;
  if (make_plan(s, B, CS, Bc, &p)) return -1;
  const long long v[8] = {p.CS, p.Bc, p.nclu, p.cols, p.hpc, p.gph, p.npairs, (long long)p.total};
  for (int i = 0; i < 8; ++i) out[i] = v[i];
  return 0;
}
