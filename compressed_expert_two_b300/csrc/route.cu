// Router: group and expert logits in the canonical FP32 order, then two-level top-k and gates.
//
// "Breaking the MoE LLM Trilemma" (paper notes), key design 3: a first router picks the group,
// a second one picks experts inside the chosen group.  "混合专家模型的路由机制与工程落地"
// section 3.1: the router runs in FP32.  "MoE架构演进白皮书" chapter 1: top-k of the logits,
// then softmax over the selected logits.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// Two independent IEEE round-to-nearest FMAs in one instruction: (a.x*b.x + c.x, a.y*b.y + c.y).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long ra = *reinterpret_cast<unsigned long long*>(&a);
  unsigned long long rb = *reinterpret_cast<unsigned long long*>(&b);
  unsigned long long rc = *reinterpret_cast<unsigned long long*>(&c);
  unsigned long long rd;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  return *reinterpret_cast<float2*>(&rd);
}

// BF16 router logits.  Warp (tg, rg) of the CTA owns TPW tokens x RPW router rows; the CTA is
// WT x WR warps.  Canonical order: lane l owns elements 128*j + 4*l + u (u = 0..3) and adds them
// in ascending index, one rounding per product (exact: BF16 x BF16 fits FP32) and per add; then
// an xor butterfly 16, 8, 4, 2, 1.  Row rr < G is group row rr (+ b_group[rr]), else expert rr-G.
// The j loop is unrolled UNR times so that UNR blocks of loads are in flight per warp.
template <int TPW, int RPW, int WT, int WR, int MINB, int UNR>
__global__ void __launch_bounds__(WT * WR * 32, MINB) router_logits_bf16_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ wg, const float* __restrict__ bg,
    const __nv_bfloat16* __restrict__ we, float* __restrict__ logits, int Tn, int d, int G, int E) {
  pdl_wait();
  pdl_trigger();
  static_assert(TPW % 2 == 0, "token pairs feed the paired FMA");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tg = warp % WT, rg = warp / WT;
  const int R = G + E;
  const int t0 = (blockIdx.x * WT + tg) * TPW;
  const int r0 = (blockIdx.y * WR + rg) * RPW;
  if (t0 >= Tn || r0 >= R) return;
  const size_t drow = (size_t)d / 4;                  // uint2 per row
  const uint2* xb = reinterpret_cast<const uint2*>(x) + lane;
  uint32_t xoff[TPW];
#pragma unroll
  for (int i = 0; i < TPW; ++i) xoff[i] = (uint32_t)min(t0 + i, Tn - 1);
  const uint2* wp[RPW];
#pragma unroll
  for (int q = 0; q < RPW; ++q) {
    const int rr = min(r0 + q, R - 1);
    wp[q] = reinterpret_cast<const uint2*>(rr < G ? wg + (size_t)rr * d : we + (size_t)(rr - G) * d) + lane;
  }
  float2 acc[TPW / 2][RPW];
#pragma unroll
  for (int i = 0; i < TPW / 2; ++i)
#pragma unroll
    for (int q = 0; q < RPW; ++q) acc[i][q] = make_float2(0.f, 0.f);
  const int nb = d / 128;
#pragma unroll UNR
  for (int jb = 0; jb < nb; ++jb) {
    uint2 xr[TPW], wr[RPW];
#pragma unroll
    for (int i = 0; i < TPW; ++i) xr[i] = __ldg(xb + xoff[i] * drow + jb * 32);
#pragma unroll
    for (int q = 0; q < RPW; ++q) wr[q] = __ldg(wp[q] + jb * 32);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      // element u of this lane's 4-element chunk
      float2 xv[TPW / 2];
#pragma unroll
      for (int i = 0; i < TPW / 2; ++i) {
        const uint32_t a = u < 2 ? xr[2 * i].x : xr[2 * i].y, b = u < 2 ? xr[2 * i + 1].x : xr[2 * i + 1].y;
        xv[i] = (u & 1) ? make_float2(__uint_as_float(a & 0xFFFF0000u), __uint_as_float(b & 0xFFFF0000u))
                        : make_float2(__uint_as_float(a << 16), __uint_as_float(b << 16));
      }
#pragma unroll
      for (int q = 0; q < RPW; ++q) {
        const uint32_t w = u < 2 ? wr[q].x : wr[q].y;
        const float wf = (u & 1) ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
        const float2 w2 = make_float2(wf, wf);
#pragma unroll
        for (int i = 0; i < TPW / 2; ++i) acc[i][q] = fma2(xv[i], w2, acc[i][q]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < TPW / 2; ++i)
#pragma unroll
    for (int q = 0; q < RPW; ++q)
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        acc[i][q].x = __fadd_rn(acc[i][q].x, __shfl_xor_sync(0xffffffffu, acc[i][q].x, o));
        acc[i][q].y = __fadd_rn(acc[i][q].y, __shfl_xor_sync(0xffffffffu, acc[i][q].y, o));
      }
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int q = 0; q < RPW; ++q) {
      const int t = t0 + i, rr = r0 + q;
      if (((i * RPW + q) & 31) == lane && t < Tn && rr < R) {
        float v = (i & 1) ? acc[i / 2][q].y : acc[i / 2][q].x;
        if (rr < G && bg != nullptr) v = __fadd_rn(v, bg[rr]);
        logits[(size_t)t * R + rr] = v;
      }
    }
}

// The router rows as FP32 pairs for the paired FMA: wpair[q][c] = (row 2q, row 2q + 1) at element c
// (rows: the G group rows, then the E expert rows; a missing last row is zero).  BF16 -> FP32 is
// exact, so the logits below are the same numbers as from the BF16 rows.
__global__ void router_wpair_kernel(const __nv_bfloat16* __restrict__ wg, const __nv_bfloat16* __restrict__ we,
                                    float2* __restrict__ wpair, int d, int G, int E) {
  pdl_wait();
  pdl_trigger();
  const int R = G + E, NP = (R + 1) / 2;
  const size_t n = (size_t)NP * d;
  for (size_t w = blockIdx.x * (size_t)blockDim.x + threadIdx.x; w < n; w += (size_t)gridDim.x * blockDim.x) {
    const int q = (int)(w / d), c = (int)(w % d);
    const int r0 = 2 * q, r1 = 2 * q + 1;
    const float a = __bfloat162float(r0 < G ? wg[(size_t)r0 * d + c] : we[(size_t)(r0 - G) * d + c]);
    const float b = r1 < R ? __bfloat162float(r1 < G ? wg[(size_t)r1 * d + c] : we[(size_t)(r1 - G) * d + c]) : 0.f;
    wpair[w] = make_float2(a, b);
  }
}

// BF16 router logits from row pairs.  Warp (tg, rg) owns TPW tokens x RP row pairs; the CTA is
// WT x WR warps.  Canonical order as above: lane l adds the products of its elements
// 128*j + 4*l + u in ascending index (one rounding per product -- exact for BF16 x BF16 -- and per
// add), then the xor butterfly 16, 8, 4, 2, 1; each paired FMA performs the steps of two rows.
template <int TPW, int RP, int WT, int WR, int MINB>
__global__ void __launch_bounds__(WT * WR * 32, MINB) router_logits_pair_kernel(
    const __nv_bfloat16* __restrict__ x, const float2* __restrict__ wpair, const float* __restrict__ bg,
    float* __restrict__ logits, int Tn, int d, int G, int E) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tg = warp % WT, rg = warp / WT;
  const int R = G + E, NP = (R + 1) / 2;
  const int t0 = (blockIdx.x * WT + tg) * TPW;
  const int q0 = (blockIdx.y * WR + rg) * RP;
  if (t0 >= Tn || q0 >= NP) return;
  const uint2* xp[TPW];
#pragma unroll
  for (int i = 0; i < TPW; ++i) xp[i] = reinterpret_cast<const uint2*>(x + (size_t)min(t0 + i, Tn - 1) * d) + lane;
  const float4* wp[RP];
#pragma unroll
  for (int q = 0; q < RP; ++q) wp[q] = reinterpret_cast<const float4*>(wpair + (size_t)min(q0 + q, NP - 1) * d) + 2 * lane;
  float2 acc[TPW][RP];
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int q = 0; q < RP; ++q) acc[i][q] = make_float2(0.f, 0.f);
  const int nb = d / 128;
#pragma unroll 2
  for (int jb = 0; jb < nb; ++jb) {
    float2 xd[TPW][4];                               // (x, x) for each token and element u
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
      const uint2 v = __ldg(xp[i] + jb * 32);
      const float e0 = __uint_as_float(v.x << 16), e1 = __uint_as_float(v.x & 0xFFFF0000u);
      const float e2 = __uint_as_float(v.y << 16), e3 = __uint_as_float(v.y & 0xFFFF0000u);
      xd[i][0] = make_float2(e0, e0); xd[i][1] = make_float2(e1, e1);
      xd[i][2] = make_float2(e2, e2); xd[i][3] = make_float2(e3, e3);
    }
#pragma unroll
    for (int q = 0; q < RP; ++q) {
      const float4 wa = __ldg(wp[q] + jb * 64), wb = __ldg(wp[q] + jb * 64 + 1);
      const float2 w2[4] = {make_float2(wa.x, wa.y), make_float2(wa.z, wa.w), make_float2(wb.x, wb.y),
                            make_float2(wb.z, wb.w)};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int i = 0; i < TPW; ++i) acc[i][q] = fma2(xd[i][u], w2[u], acc[i][q]);
    }
  }
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int q = 0; q < RP; ++q)
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        acc[i][q].x = __fadd_rn(acc[i][q].x, __shfl_xor_sync(0xffffffffu, acc[i][q].x, o));
        acc[i][q].y = __fadd_rn(acc[i][q].y, __shfl_xor_sync(0xffffffffu, acc[i][q].y, o));
      }
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int q = 0; q < RP; ++q)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int t = t0 + i, rr = 2 * (q0 + q) + h;
        if (((i * RP * 2 + q * 2 + h) & 31) == lane && t < Tn && rr < R) {
          float v = h ? acc[i][q].y : acc[i][q].x;
          if (rr < G && bg != nullptr) v = __fadd_rn(v, bg[rr]);
          logits[(size_t)t * R + rr] = v;
        }
      }
}

template <int TPW, int RP, int WT, int WR, int MINB>
static void launch_pair_logits(const void* x, const float2* wpair, const float* bg, float* logits, int Tn, int d,
                               int G, int E, cudaStream_t st) {
  const int NP = (G + E + 1) / 2;
  dim3 grid((Tn + WT * TPW - 1) / (WT * TPW), (NP + WR * RP - 1) / (WR * RP));
  launch_pdl(router_logits_pair_kernel<TPW, RP, WT, WR, MINB>, grid, dim3(WT * WR * 32), 0, st,
             (const __nv_bfloat16*)x, (const float2*)wpair, bg, logits, Tn, d, G, E);
}

// FP32 router logits (same canonical order; products rounded before the add, no contraction).
template <int TPW, int RB>
__global__ void __launch_bounds__(256) router_logits_f32_kernel(
    const float* __restrict__ x, const float* __restrict__ wg, const float* __restrict__ bg,
    const float* __restrict__ we, float* __restrict__ logits, int Tn, int d, int G, int E) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = G + E;
  const int t0 = (blockIdx.x * 8 + warp) * TPW;
  const int r0 = blockIdx.y * RB;
  if (t0 >= Tn) return;
  const float* xp[TPW];
#pragma unroll
  for (int i = 0; i < TPW; ++i) xp[i] = x + (size_t)min(t0 + i, Tn - 1) * d;
  const float* wp[RB];
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
    float4 xv[TPW];
#pragma unroll
    for (int i = 0; i < TPW; ++i) xv[i] = *reinterpret_cast<const float4*>(xp[i] + base);
#pragma unroll
    for (int q = 0; q < RB; ++q) {
      const float4 wv = *reinterpret_cast<const float4*>(wp[q] + base);
#pragma unroll
      for (int i = 0; i < TPW; ++i) {
        acc[i][q] = __fadd_rn(acc[i][q], __fmul_rn(xv[i].x, wv.x));
        acc[i][q] = __fadd_rn(acc[i][q], __fmul_rn(xv[i].y, wv.y));
        acc[i][q] = __fadd_rn(acc[i][q], __fmul_rn(xv[i].z, wv.z));
        acc[i][q] = __fadd_rn(acc[i][q], __fmul_rn(xv[i].w, wv.w));
      }
    }
  }
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int q = 0; q < RB; ++q)
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1)
        acc[i][q] = __fadd_rn(acc[i][q], __shfl_xor_sync(0xffffffffu, acc[i][q], o));
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
  pdl_wait();
  pdl_trigger();
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

template <int TPW, int RPW, int WT, int WR, int MINB, int UNR>
static void launch_bf16_logits(const void* x, const void* wg, const float* bg, const void* we, float* logits,
                               int Tn, int d, int G, int E, cudaStream_t st) {
  const int R = G + E;
  dim3 grid((Tn + WT * TPW - 1) / (WT * TPW), (R + WR * RPW - 1) / (WR * RPW));
  launch_pdl(router_logits_bf16_kernel<TPW, RPW, WT, WR, MINB, UNR>, grid, dim3(WT * WR * 32), 0, st,
             (const __nv_bfloat16*)x, (const __nv_bfloat16*)wg, bg, (const __nv_bfloat16*)we, logits, Tn, d, G, E);
}

static cudaError_t launch_logits(bool bf16, const void* x, const void* wg, const float* bg, const void* we,
                                 float2* wpair, float* logits, int Tn, int d, int G, int E, cudaStream_t st) {
  if (bf16 && Tn >= 1024 && wpair) {
    // many tokens: FP32 row pairs, 4 tokens x RP row pairs per warp; RP picked to waste the
    // fewest pairs for this router height
    const int NP = (G + E + 1) / 2;
    launch_pdl(router_wpair_kernel, dim3(148 * 2), dim3(256), 0, st, (const __nv_bfloat16*)wg,
               (const __nv_bfloat16*)we, wpair, d, G, E);
    prof_mark("router_wpair", st);
    const int w4 = (NP + 7) / 8 * 8 - NP, w6 = (NP + 11) / 12 * 12 - NP, w8 = (NP + 15) / 16 * 16 - NP;
    if (w6 < w4 && w6 <= w8) launch_pair_logits<4, 6, 4, 2, 2>(x, wpair, bg, logits, Tn, d, G, E, st);
    else if (w8 < w4) launch_pair_logits<4, 8, 4, 2, 2>(x, wpair, bg, logits, Tn, d, G, E, st);
    else launch_pair_logits<4, 4, 4, 2, 2>(x, wpair, bg, logits, Tn, d, G, E, st);
  } else if (bf16) {
    // few tokens: small warp blocks and a deep unroll so that the loads of many j blocks are in
    // flight at once
    launch_bf16_logits<2, 4, 4, 2, 2, 8>(x, wg, bg, we, logits, Tn, d, G, E, st);
  } else {
    constexpr int TPW = 4, RB = 8;
    dim3 grid((Tn + 8 * TPW - 1) / (8 * TPW), (G + E + RB - 1) / RB);
    launch_pdl(router_logits_f32_kernel<TPW, RB>, grid, dim3(256), 0, st, (const float*)x, (const float*)wg, bg,
               (const float*)we, logits, Tn, d, G, E);
  }
  prof_mark("router_logits", st);
  return cudaGetLastError();
}

cudaError_t launch_route(const LayerArgs& a, const void* x, const void* wg, const float* bg,
                         const void* we, float2* wpair, float* logits, int32_t* gidx, int32_t* eidx, float* gate,
                         cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  cudaError_t err = launch_logits(a.bf16, x, wg, bg, we, wpair, logits, a.T, a.d, a.G, a.E, st);
  if (err != cudaSuccess) return err;
  launch_pdl(router_select_kernel, dim3((a.T + 127) / 128), dim3(128), 0, st, (const float*)logits, a.tab, a.T, a.kg,
             a.ke, gidx, eidx, gate);
  prof_mark("router_select", st);
  return cudaGetLastError();
}

}  // namespace moe
