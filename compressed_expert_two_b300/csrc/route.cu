// Router: group and expert logits in the canonical FP32 order, then two-level top-k and gates.
//
// "Breaking the MoE LLM Trilemma" (paper notes), key design 3: a first router picks the group,
// a second one picks experts inside the chosen group.  "混合专家模型的路由机制与工程落地"
// section 3.1: the router runs in FP32.  "MoE架构演进白皮书" chapter 1: top-k of the logits,
// then softmax over the selected logits.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// Logits of TPW tokens x RB router rows per warp; 8 warps share the rows of one CTA.
// Row index rr in [0, G) is group row rr (plus b_group[rr]); rr in [G, G+E) is expert row rr-G.
// Canonical order: lane l owns elements 128*j + 4*l + u (u = 0..3), adds them in ascending
// index with one rounding per product and per add, then an xor butterfly 16, 8, 4, 2, 1.
template <typename T, int TPW, int RB>
__global__ void __launch_bounds__(256) router_logits_kernel(
    const T* __restrict__ x, const T* __restrict__ wg, const float* __restrict__ bg,
    const T* __restrict__ we, float* __restrict__ logits, int Tn, int d, int G, int E) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = G + E;
  const int t0 = (blockIdx.x * 8 + warp) * TPW;
  const int r0 = blockIdx.y * RB;
  if (t0 >= Tn) return;

  const T* xp[TPW];
#pragma unroll
  for (int i = 0; i < TPW; ++i) xp[i] = x + (size_t)min(t0 + i, Tn - 1) * d;
  const T* wp[RB];
#pragma unroll
  for (int q = 0; q < RB; ++q) {
    const int rr = min(r0 + q, R - 1);
    wp[q] = rr < G ? wg + (size_t)rr * d : we + (size_t)(rr - G) * d;
  }
  float acc[TPW][RB];
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int q = 0; q < RB; ++q) acc[i][q] = 0.f;

  for (int base = 4 * lane; base < d; base += 128) {
    float xv[TPW][4];
#pragma unroll
    for (int i = 0; i < TPW; ++i)
#pragma unroll
      for (int u = 0; u < 4; ++u) xv[i][u] = to_f32(xp[i][base + u]);
#pragma unroll
    for (int q = 0; q < RB; ++q) {
      float wv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) wv[u] = to_f32(wp[q][base + u]);
#pragma unroll
      for (int i = 0; i < TPW; ++i)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if constexpr (sizeof(T) == 2) {
            // BF16 x BF16 is exact in FP32, so the fused form equals fl(s + fl(x*w)).
            acc[i][q] = __fmaf_rn(xv[i][u], wv[u], acc[i][q]);
          } else {
            acc[i][q] = __fadd_rn(acc[i][q], __fmul_rn(xv[i][u], wv[u]));
          }
        }
    }
  }
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int q = 0; q < RB; ++q) {
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1)
        acc[i][q] = __fadd_rn(acc[i][q], __shfl_xor_sync(0xffffffffu, acc[i][q], o));
    }
  // every lane holds every sum; lane (i*RB+q) % 32 writes it
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int q = 0; q < RB; ++q) {
      const int t = t0 + i, rr = r0 + q;
      if (((i * RB + q) & 31) == lane && t < Tn && rr < R) {
        float v = acc[i][q];
        if (rr < G && bg != nullptr) v = __fadd_rn(v, bg[rr]);
        logits[(size_t)t * R + rr] = v;
      }
    }
}

// One thread per token: top-k_g groups, softmax p; inside each chosen group top-k_e experts,
// softmax q; gate = p * q.  Higher logit first, equal logits -> lower index first.
__global__ void router_select_kernel(const float* __restrict__ logits, GroupTable tab, int Tn,
                                     int kg, int ke, int32_t* __restrict__ gidx,
                                     int32_t* __restrict__ eidx, float* __restrict__ gate) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= Tn) return;
  const int G = tab.G, E = tab.E, K = tab.K, k = kg * ke;
  const float* sg = logits + (size_t)t * (G + E);
  const float* se = sg + G;
  uint32_t taken[kMaxE / 32];
#pragma unroll
  for (int i = 0; i < kMaxE / 32; ++i) taken[i] = 0u;
  int gsel[kMaxK];
  float gval[kMaxK];
  for (int j = 0; j < kg; ++j) {
    int best = -1;
    float bv = 0.f;
    for (int g = 0; g < G; ++g) {
      if (taken[g >> 5] & (1u << (g & 31))) continue;
      const float v = sg[g];
      if (best < 0 || v > bv) { best = g; bv = v; }
    }
    taken[best >> 5] |= 1u << (best & 31);
    gsel[j] = best;
    gval[j] = bv;
  }
  float pden = 0.f, pe[kMaxK];
  for (int j = 0; j < kg; ++j) { pe[j] = expf(gval[j] - gval[0]); pden += pe[j]; }
  for (int j = 0; j < kg; ++j) {
    const int g = gsel[j];
    gidx[(size_t)t * kg + j] = g;
    const float p = pe[j] / pden;
    uint32_t used = 0u;  // bit i: i-th member of g already chosen (K <= 32 enforced on host)
    int esel[kMaxK];
    float ev[kMaxK];
    for (int s = 0; s < ke; ++s) {
      int bi = -1;
      float bv = 0.f;
      for (int i = 0; i < K; ++i) {
        if (used & (1u << i)) continue;
        const float v = se[tab.member[g * K + i]];
        if (bi < 0 || v > bv) { bi = i; bv = v; }
      }
      used |= 1u << bi;
      esel[s] = tab.member[g * K + bi];
      ev[s] = bv;
    }
    float qden = 0.f, qe[kMaxK];
    for (int s = 0; s < ke; ++s) { qe[s] = expf(ev[s] - ev[0]); qden += qe[s]; }
    for (int s = 0; s < ke; ++s) {
      eidx[(size_t)t * k + j * ke + s] = esel[s];
      gate[(size_t)t * k + j * ke + s] = p * (qe[s] / qden);
    }
  }
}

template <typename T>
static cudaError_t launch_logits(const void* x, const void* wg, const float* bg, const void* we,
                                 float* logits, int Tn, int d, int G, int E, cudaStream_t st) {
  constexpr int TPW = 4, RB = 8;
  const int R = G + E;
  dim3 grid((Tn + 8 * TPW - 1) / (8 * TPW), (R + RB - 1) / RB);
  router_logits_kernel<T, TPW, RB><<<grid, 256, 0, st>>>(
      (const T*)x, (const T*)wg, bg, (const T*)we, logits, Tn, d, G, E);
  prof_mark("router_logits", st);
  return cudaGetLastError();
}

cudaError_t launch_route(const LayerArgs& a, const void* x, const void* wg, const float* bg,
                         const void* we, float* logits, int32_t* gidx, int32_t* eidx, float* gate,
                         cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  cudaError_t err = a.bf16 ? launch_logits<__nv_bfloat16>(x, wg, bg, we, logits, a.T, a.d, a.G, a.E, st)
                           : launch_logits<float>(x, wg, bg, we, logits, a.T, a.d, a.G, a.E, st);
  if (err != cudaSuccess) return err;
  router_select_kernel<<<(a.T + 127) / 128, 128, 0, st>>>(logits, a.tab, a.T, a.kg, a.ke, gidx, eidx, gate);
  prof_mark("router_select", st);
  return cudaGetLastError();
}

}  // namespace moe
