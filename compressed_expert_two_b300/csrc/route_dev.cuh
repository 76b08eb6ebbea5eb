// Device-side two-level selection shared by the router kernels and the fused decode pre-pass.
//
// "Breaking the MoE LLM Trilemma" (paper notes), key design 3: a first router picks the group,
// a second one picks experts inside the chosen group.  "MoE架构演进白皮书" chapter 1: top-k of
// the logits, then softmax over the selected logits.
#pragma once
#include "common.cuh"

namespace moe {

// L lanes per token (L = the power of two >= max(G, K), at most 32): top-k_g groups, softmax p;
// inside each chosen group top-k_e experts, softmax q; gate = p * q.  Higher logit first, equal
// logits -> lower index first.  Lane l of a token holds groups l, l + L, ... and, per chosen
// group, its member l; each pick is an argmax over the token's lanes; lane j keeps the j-th pick.
// The softmax sums run over the picks in order.
constexpr int kSelGroupsPerLane = kMaxE / 32;

template <int L>
__device__ __forceinline__ void seg_argmax(float& v, int& idx) {
  // idx < 0: nothing to offer; ties go to the lower index
#pragma unroll
  for (int o = L / 2; o >= 1; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o, L);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o, L);
    if (oi >= 0 && (idx < 0 || ov > v || (ov == v && oi < idx))) { v = ov; idx = oi; }
  }
}

template <int L>
__device__ __forceinline__ void select_token(const float* sg, const GroupTable& tab, int t, bool valid, int kg,
                                             int ke, int li, int32_t* __restrict__ gidx, int32_t* __restrict__ eidx,
                                             float* __restrict__ gate) {
  const int G = tab.G, K = tab.K, k = kg * ke;
  const float* se = sg + G;
  float gv[kSelGroupsPerLane];
  uint32_t avail = 0u;
#pragma unroll
  for (int u = 0; u < kSelGroupsPerLane; ++u) {
    const int g = li + L * u;
    gv[u] = g < G ? sg[g] : 0.f;
    if (g < G) avail |= 1u << u;
  }
  // group picks: lane j keeps pick j
  int my_g = -1;
  float my_gv = 0.f;
  for (int j = 0; j < kg; ++j) {
    float bv = 0.f;
    int bi = -1;
#pragma unroll
    for (int u = 0; u < kSelGroupsPerLane; ++u)
      if (((avail >> u) & 1u) && (bi < 0 || gv[u] > bv)) { bv = gv[u]; bi = li + L * u; }
    seg_argmax<L>(bv, bi);
    if (bi % L == li) avail &= ~(1u << (bi / L));
    if (li == j) { my_g = bi; my_gv = bv; }
  }
  const float g0 = __shfl_sync(0xffffffffu, my_gv, 0, L);
  const float my_pe = expf(my_gv - g0);
  float pden = 0.f;
  for (int j = 0; j < kg; ++j) pden += __shfl_sync(0xffffffffu, my_pe, j, L);
  const float my_p = my_pe / pden;
  for (int j = 0; j < kg; ++j) {
    const int g = __shfl_sync(0xffffffffu, my_g, j, L);
    const float p = __shfl_sync(0xffffffffu, my_p, j, L);
    if (valid && li == 0) gidx[(size_t)t * kg + j] = g;
    const float v_l = li < K ? se[tab.member[g * K + li]] : 0.f;
    bool open = li < K;
    int my_e = -1;
    float my_ev = 0.f;
    for (int s2 = 0; s2 < ke; ++s2) {
      float bv = open ? v_l : 0.f;
      int bi = open ? li : -1;
      seg_argmax<L>(bv, bi);
      if (bi == li) open = false;
      if (li == s2) { my_e = (int)tab.member[g * K + bi]; my_ev = bv; }
    }
    const float e0 = __shfl_sync(0xffffffffu, my_ev, 0, L);
    const float my_qe = expf(my_ev - e0);
    float qden = 0.f;
    for (int s2 = 0; s2 < ke; ++s2) qden += __shfl_sync(0xffffffffu, my_qe, s2, L);
    if (valid && li < ke) {
      eidx[(size_t)t * k + j * ke + li] = my_e;
      gate[(size_t)t * k + j * ke + li] = p * (my_qe / qden);
    }
  }
}

}  // namespace moe
