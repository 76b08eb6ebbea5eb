// Router: group and expert logits in the canonical FP32 order, then two-level top-k and gates.
//
// "Breaking the MoE LLM Trilemma" (paper notes), key design 3: a first router picks the group,
// a second one picks experts inside the chosen group.  "混合专家模型的路由机制与工程落地"
// section 3.1: the router runs in FP32.  "MoE架构演进白皮书" chapter 1: top-k of the logits,
// then softmax over the selected logits.
#include "common.cuh"
#include "kernels.h"
#include "route_dev.cuh"

namespace moe {

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

// BF16 router logits with the operands staged in shared memory.  A CTA of 4 x RG warps computes
// 32 tokens x 8 RG router rows (warp (tg, rg): tokens 8 tg.., rows 8 rg..); d streams through a
// three-stage cp.async pipeline in chunks of 256 elements.  Canonical order as above: lane l adds
// the products of its elements 128*j + 4*l + u in ascending index (one rounding per product --
// exact for BF16 x BF16 -- and per add), then the xor butterfly 16, 8, 4, 2, 1.  With L > 0 the
// CTA holds every router row of its tokens (G + E <= 8 RG): the logits stay in shared memory and
// the CTA's warps make the selection itself (L lanes per token, as router_select_kernel<L>).
constexpr int kRtTok = 32, kRtDC = 256, kRtStages = 3;

// The xor butterfly 16, 8, 4, 2, 1 of 32 per-lane values v[0..31] at once: at the step of
// distance k a lane keeps the half of its values whose index bit matches its own lane bit, adds
// the partner's copy of each (own + partner, the butterfly's add for that lane), and hands the
// other half over.  Lane l returns the butterfly total of value l, bit for bit.
__device__ __forceinline__ float butterfly_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) {
    const bool hi = (lane & k) != 0;
#pragma unroll
    for (int j = 0; j < k; ++j) {
      const float keep = hi ? v[j + k] : v[j], send = hi ? v[j] : v[j + k];
      v[j] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, k));
    }
  }
  return v[0];
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// BF16 -> FP32 (exact: the 16 bits move to the top) of element u (0..3) of a 4-element piece.
__device__ __forceinline__ float bf16_elem(const uint2& v, int u) {
  const uint32_t w = u < 2 ? v.x : v.y;
  return __uint_as_float((u & 1) ? (w & 0xffff0000u) : (w << 16));
}

// acc[i][q] += x_i[u] * w_q[u] for u = 0..3 in order (8 x 8 sums, each element rounded once per
// FMA), with the operands converted once and the FMAs paired over (q, q+1): the same rounding
// sequence as 256 scalar FMAs.
__device__ __forceinline__ void fma_tile8x8(const uint2 (&xr)[8], const uint2 (&wr)[8], float2 (&acc)[8][4]) {
  float2 wp[4][4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int qp = 0; qp < 4; ++qp) wp[u][qp] = make_float2(bf16_elem(wr[2 * qp], u), bf16_elem(wr[2 * qp + 1], u));
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float xv = bf16_elem(xr[i], u);
      const float2 a = make_float2(xv, xv);
#pragma unroll
      for (int qp = 0; qp < 4; ++qp) acc[i][qp] = fma2(a, wp[u][qp], acc[i][qp]);
    }
}

template <int RG, int L>
__global__ void __launch_bounds__(128 * RG, RG <= 2 ? 2 : 1) router_logits_smem_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ wg, const float* __restrict__ bg,
    const __nv_bfloat16* __restrict__ we, float* __restrict__ logits, int Tn, int d, int G, int E, GroupTable tab,
    int kg, int ke, int32_t* __restrict__ gidx, int32_t* __restrict__ eidx, float* __restrict__ gate) {
  pdl_wait();
  pdl_trigger();
  constexpr int kRtRows = 8 * RG;
  extern __shared__ __align__(16) uint8_t rt_smem[];   // [stages][32][256] x, then [stages][8 RG][256] w
  __shared__ float s_logit[L > 0 ? kRtTok * kRtRows : 1];
  auto xs = reinterpret_cast<__nv_bfloat16 (*)[kRtTok][kRtDC]>(rt_smem);
  auto ws = reinterpret_cast<__nv_bfloat16 (*)[kRtRows][kRtDC]>(rt_smem + sizeof(__nv_bfloat16) * kRtStages * kRtTok * kRtDC);
  const int R = G + E;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tg = warp & 3, rg = warp >> 2;
  const int t_base = blockIdx.x * kRtTok, r_base = blockIdx.y * kRtRows;
  const int nchunk = (d + kRtDC - 1) / kRtDC;
  // loader: 16-byte pieces; rows past the batch or the router repeat the last one (results unused)
  auto load_chunk = [&](int c, int st) {
    const int cb = c * kRtDC, width = min(kRtDC, d - cb), pieces = width / 8;
    for (int w = threadIdx.x; w < kRtTok * pieces; w += blockDim.x) {
      const int rr = w / pieces, pc = (w % pieces) * 8;
      const int t = min(t_base + rr, Tn - 1);
      cp_async16(&xs[st][rr][pc], x + (size_t)t * d + cb + pc);
    }
    for (int w = threadIdx.x; w < kRtRows * pieces; w += blockDim.x) {
      const int rr = w / pieces, pc = (w % pieces) * 8;
      const int r = min(r_base + rr, R - 1);
      const __nv_bfloat16* src = r < G ? wg + (size_t)r * d : we + (size_t)(r - G) * d;
      cp_async16(&ws[st][rr][pc], src + cb + pc);
    }
  };
  float acc[8][8];                                   // [token][row]
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[i][q] = 0.f;
#pragma unroll
  for (int c = 0; c < kRtStages - 1; ++c) {
    if (c < nchunk) load_chunk(c, c);
    cp_async_commit();
  }
  for (int c = 0; c < nchunk; ++c) {
    cp_async_wait<kRtStages - 2>();
    __syncthreads();
    const int st = c % kRtStages;
    const int nj = min(kRtDC, d - c * kRtDC) / 128;
    for (int jj = 0; jj < nj; ++jj) {
      uint2 xr[8], wr[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) xr[i] = *reinterpret_cast<const uint2*>(&xs[st][tg * 8 + i][jj * 128 + 4 * lane]);
#pragma unroll
      for (int q = 0; q < 8; ++q) wr[q] = *reinterpret_cast<const uint2*>(&ws[st][rg * 8 + q][jj * 128 + 4 * lane]);
      // element u of the lane's 4-element chunk: the mixed-precision FMA takes the BF16 halves
      // as they are (BF16 x BF16 is exact in FP32, so it rounds once, like mul + add)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t a = u < 2 ? xr[i].x : xr[i].y;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t w = u < 2 ? wr[q].x : wr[q].y;
            acc[i][q] = (u & 1) ? fma_bf16_hi(a, w, acc[i][q]) : fma_bf16_lo(a, w, acc[i][q]);
          }
        }
      }
    }
    // refill the stage computed in the previous iteration (every warp has passed the barrier above)
    const int cn = c + kRtStages - 1;
    if (cn < nchunk) load_chunk(cn, cn % kRtStages);
    cp_async_commit();
  }
  // the butterfly of each of the 64 sums, as two reduce-scatters of 32 sums each: lane l ends with
  // sum l of each half (tokens 0..3 / 4..7) and every add is the butterfly's own add
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    float v[32];
#pragma unroll
    for (int o = 0; o < 32; ++o) v[o] = acc[4 * hf + (o >> 3)][o & 7];
    const float s = butterfly_scatter32(v, lane);
    const int i = 4 * hf + (lane >> 3), q = lane & 7;
    const int t = t_base + tg * 8 + i, rr = r_base + rg * 8 + q;
    float out = s;
    if (rr < G && bg != nullptr) out = __fadd_rn(out, bg[rr]);
    if constexpr (L > 0) {
      s_logit[(tg * 8 + i) * kRtRows + rg * 8 + q] = out;
    } else if (t < Tn && rr < R) {
      logits[(size_t)t * R + rr] = out;
    }
  }
  if constexpr (L > 0) {
    // selection of the CTA's 32 tokens: L lanes per token, 32 / L tokens per warp
    __syncthreads();
    constexpr int kPerWarp = 32 / L;
    const int li = lane & (L - 1);
    for (int tt0 = warp * kPerWarp; tt0 < kRtTok; tt0 += 4 * RG * kPerWarp) {
      const int tt = tt0 + lane / L, t = t_base + tt;
      const bool valid = t < Tn;
      select_token<L>(s_logit + tt * kRtRows, tab, valid ? t : Tn - 1, valid, kg, ke, li, gidx, eidx, gate);
    }
  }
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

// Selection over logits rows 0 .. n-1 (n = Tn, or *list_n with list: row p belongs to token
// list[p]); L lanes per row, grid-stride.
template <int L>
__global__ void __launch_bounds__(256) router_select_kernel(const float* __restrict__ logits, GroupTable tab,
                                                            int Tn, const int32_t* __restrict__ list,
                                                            const int* list_n, int kg, int ke,
                                                            int32_t* __restrict__ gidx, int32_t* __restrict__ eidx,
                                                            float* __restrict__ gate) {
  pdl_wait();
  pdl_trigger();
  const int n = list ? *(volatile const int*)list_n : Tn;
  const int li = threadIdx.x & (L - 1);
  for (int base = blockIdx.x * blockDim.x;; base += gridDim.x * blockDim.x) {
    if ((base + (int)(threadIdx.x & ~31u)) / L >= n) break;   // the whole warp is past the rows
    const int p_raw = (base + (int)threadIdx.x) / L;
    const bool valid = p_raw < n;
    const int p = valid ? p_raw : n - 1;
    const int t = list ? list[p] : p;
    select_token<L>(logits + (size_t)p * (tab.G + tab.E), tab, t, valid, kg, ke, li, gidx, eidx, gate);
  }
}

template <int L>
static void launch_select(const LayerArgs& a, const float* logits, const int32_t* list, const int* list_n,
                          int32_t* gidx, int32_t* eidx, float* gate, cudaStream_t st) {
  const int per_block = 256 / L;
  int blocks = (a.T + per_block - 1) / per_block;
  if (list && blocks > 148) blocks = 148;      // rows known on the device only: grid-stride
  launch_pdl(router_select_kernel<L>, dim3(blocks), dim3(256), 0, st, logits, a.tab, a.T, list, list_n, a.kg, a.ke,
             gidx, eidx, gate);
}

static void launch_select_any(const LayerArgs& a, const float* logits, const int32_t* list, const int* list_n,
                              int32_t* gidx, int32_t* eidx, float* gate, cudaStream_t st) {
  const int need = a.G > a.K ? a.G : a.K;
  if (need <= 4) launch_select<4>(a, logits, list, list_n, gidx, eidx, gate, st);
  else if (need <= 8) launch_select<8>(a, logits, list, list_n, gidx, eidx, gate, st);
  else if (need <= 16) launch_select<16>(a, logits, list, list_n, gidx, eidx, gate, st);
  else launch_select<32>(a, logits, list, list_n, gidx, eidx, gate, st);
}

// The across-groups reading of level 2: among a token's k = k_g k_e candidate slots (each chosen
// group's top-k_e members, which hold every member of the union's top k_e), the k_e best by
// canonical expert logit (ties to the lower id) get gate = softmax over their logits (in pick
// order, as the within-group gates), every other slot gate 0.  One thread per token.
__device__ __forceinline__ void across_token(const float* __restrict__ se, int t, int k, int ke,
                                             const int32_t* __restrict__ eidx, float* __restrict__ gate) {
  // every array index below is a compile-time constant (unrolled loops), so all stays in registers
  int id[kMaxK];
  float v[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) {
    id[s] = s < k ? eidx[(size_t)t * k + s] : 0;
    v[s] = s < k ? se[id[s]] : 0.f;
  }
  uint32_t picked = 0;
  float q[kMaxK];
  uint32_t pick_mask[kMaxK];
  float den = 0.f, v0 = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    q[j] = 0.f;
    pick_mask[j] = 0u;
    if (j < ke) {
      float bv = 0.f;
      int bid = 0;
      uint32_t bmask = 0u;
#pragma unroll
      for (int s = 0; s < kMaxK; ++s) {
        const bool cand = s < k && !((picked >> s) & 1u);
        if (cand && (bmask == 0u || v[s] > bv || (v[s] == bv && id[s] < bid))) { bv = v[s]; bid = id[s]; bmask = 1u << s; }
      }
      picked |= bmask;
      pick_mask[j] = bmask;
      if (j == 0) v0 = bv;
      q[j] = expf(bv - v0);
      den += q[j];
    }
  }
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) {
    if (s >= k) break;
    float g = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if ((pick_mask[j] >> s) & 1u) g = q[j] / den;
    gate[(size_t)t * k + s] = g;
  }
}

// With a list (the tokens the tensor-core router left over), logits row p belongs to token
// list[p], p < *list_n, grid-stride; without one, row p is token p.
__global__ void __launch_bounds__(256) router_across_kernel(const float* __restrict__ logits, int Tn, int G, int E,
                                                            int k, int ke, const int32_t* __restrict__ eidx,
                                                            float* __restrict__ gate, const int32_t* __restrict__ list,
                                                            const int* list_n) {
  pdl_wait();
  pdl_trigger();
  const int n = list ? *(volatile const int*)list_n : Tn;
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n; p += gridDim.x * blockDim.x)
    across_token(logits + (size_t)p * (G + E) + G, list ? list[p] : p, k, ke, eidx, gate);
}

// Canonical-order BF16 logits of the listed tokens (the ones the tensor-core router could not
// verify), grid-stride; logits row p belongs to token list[p].  Lane l adds the products of its
// elements 128 j + 4 l + u in ascending index, then the xor butterfly 16, 8, 4, 2, 1 (as a
// reduce-scatter for the 8 x 8 tiles), as the other canonical kernels.  Few tokens: one warp per
// (token, 8 router rows), so that they spread over every SM; many: one warp per (8 tokens,
// 8 router rows), which reads each row once for 8 tokens.
__global__ void __launch_bounds__(256, 1) router_exact_list_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ wg, const float* __restrict__ bg,
    const __nv_bfloat16* __restrict__ we, const int32_t* __restrict__ list, const int* list_n, int d, int G, int E,
    float* __restrict__ logits) {
  pdl_wait();
  pdl_trigger();
  const int n = *(volatile const int*)list_n;
  const int R = G + E, nrb = (R + 7) / 8, ntb = (n + 7) / 8;
  const int lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  if (n * nrb <= 2 * nw) {
    for (int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < n * nrb; item += nw) {
      const int p = item / nrb, r0 = (item % nrb) * 8;
      const __nv_bfloat16* xr = x + (size_t)list[p] * d + 4 * lane;
      const __nv_bfloat16* wr[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int rr = min(r0 + q, R - 1);
        wr[q] = (rr < G ? wg + (size_t)rr * d : we + (size_t)(rr - G) * d) + 4 * lane;
      }
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.f;
#pragma unroll 4
      for (int j = 0; j < d; j += 128) {
        const uint2 xv = *reinterpret_cast<const uint2*>(xr + j);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint2 wv = *reinterpret_cast<const uint2*>(wr[q] + j);
          acc[q] = fma_bf16_lo(xv.x, wv.x, acc[q]);
          acc[q] = fma_bf16_hi(xv.x, wv.x, acc[q]);
          acc[q] = fma_bf16_lo(xv.y, wv.y, acc[q]);
          acc[q] = fma_bf16_hi(xv.y, wv.y, acc[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q)
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) acc[q] = __fadd_rn(acc[q], __shfl_xor_sync(0xffffffffu, acc[q], o));
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int rr = r0 + q;
        if (lane == q && rr < R) {
          float v = acc[q];
          if (rr < G && bg != nullptr) v = __fadd_rn(v, bg[rr]);
          logits[(size_t)p * R + rr] = v;
        }
      }
    }
    return;
  }
  for (int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < ntb * nrb; item += nw) {
    const int p0 = (item / nrb) * 8, r0 = (item % nrb) * 8;
    const __nv_bfloat16* xr[8];
    const __nv_bfloat16* wr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      xr[i] = x + (size_t)list[min(p0 + i, n - 1)] * d + 4 * lane;
      const int rr = min(r0 + i, R - 1);
      wr[i] = (rr < G ? wg + (size_t)rr * d : we + (size_t)(rr - G) * d) + 4 * lane;
    }
    float2 acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][q] = make_float2(0.f, 0.f);
#pragma unroll 2
    for (int j = 0; j < d; j += 128) {
      uint2 xv[8], wv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) { xv[i] = *reinterpret_cast<const uint2*>(xr[i] + j); wv[i] = *reinterpret_cast<const uint2*>(wr[i] + j); }
      fma_tile8x8(xv, wv, acc);
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      float v[32];
#pragma unroll
      for (int o = 0; o < 32; ++o) v[o] = (o & 1) ? acc[4 * hf + (o >> 3)][(o & 7) >> 1].y : acc[4 * hf + (o >> 3)][(o & 7) >> 1].x;
      float out = butterfly_scatter32(v, lane);
      const int p = p0 + 4 * hf + (lane >> 3), rr = r0 + (lane & 7);
      if (rr < G && bg != nullptr) out = __fadd_rn(out, bg[rr]);
      if (p < n && rr < R) logits[(size_t)p * R + rr] = out;
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

template <int RG, int L>
static cudaError_t launch_smem_logits(const LayerArgs& a, const void* x, const void* wg, const float* bg,
                                      const void* we, float* logits, int32_t* gidx, int32_t* eidx, float* gate,
                                      cudaStream_t st) {
  constexpr int rows = 8 * RG;
  const int Tn = a.T, d = a.d, G = a.G, E = a.E;
  dim3 grid((Tn + kRtTok - 1) / kRtTok, (G + E + rows - 1) / rows);
  constexpr size_t smem = sizeof(__nv_bfloat16) * kRtStages * (kRtTok + rows) * kRtDC;
  static std::atomic<uint64_t> attr{0};
  if (const cudaError_t e = smem_attr_once(router_logits_smem_kernel<RG, L>, smem, attr); e != cudaSuccess) return e;
  return launch_pdl(router_logits_smem_kernel<RG, L>, grid, dim3(128 * RG), smem, st, (const __nv_bfloat16*)x,
                    (const __nv_bfloat16*)wg, bg, (const __nv_bfloat16*)we, logits, Tn, d, G, E, a.tab, a.kg, a.ke,
                    gidx, eidx, gate);
}

// Router logits and selection in one launch when a CTA can hold every router row of its tokens
// (G + E <= 24, at least 1024 tokens); returns false (nothing launched) otherwise.
static bool fused_route_ok(const LayerArgs& a) {
  const int R = a.G + a.E, need = a.G > a.K ? a.G : a.K;
  return a.bf16 && a.T >= 1024 && R <= 24 && need <= 8;
}

static bool launch_fused_route(const LayerArgs& a, const void* x, const void* wg, const float* bg, const void* we,
                               int32_t* gidx, int32_t* eidx, float* gate, cudaStream_t st, cudaError_t* err) {
  const int R = a.G + a.E, need = a.G > a.K ? a.G : a.K;
  if (!fused_route_ok(a)) return false;
  if (R <= 16)
    *err = need <= 4 ? launch_smem_logits<2, 4>(a, x, wg, bg, we, nullptr, gidx, eidx, gate, st)
                     : launch_smem_logits<2, 8>(a, x, wg, bg, we, nullptr, gidx, eidx, gate, st);
  else
    *err = need <= 4 ? launch_smem_logits<3, 4>(a, x, wg, bg, we, nullptr, gidx, eidx, gate, st)
                     : launch_smem_logits<3, 8>(a, x, wg, bg, we, nullptr, gidx, eidx, gate, st);
  prof_mark("router", st);
  return true;
}

static cudaError_t launch_logits(const LayerArgs& a, bool bf16, const void* x, const void* wg, const float* bg,
                                 const void* we, float* logits, int Tn, int d, int G, int E, cudaStream_t st) {
  if (bf16 && Tn >= 1024) {
    const cudaError_t e = launch_smem_logits<2, 0>(a, x, wg, bg, we, logits, nullptr, nullptr, nullptr, st);
    if (e != cudaSuccess) return e;
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
                         const void* we, float* logits, int32_t* redo, int32_t* gidx, int32_t* eidx,
                         float* gate, DevStatus* status, bool status_zeroed, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  cudaError_t err = cudaSuccess;
  if (a.across && (fused_route_ok(a) || !route_tc_ok(a))) {
    // canonical logits of every token stay in the workspace: the within-group selection gives the
    // candidate slots, then the picks over their union set the gates
    if ((err = launch_logits(a, a.bf16, x, wg, bg, we, logits, a.T, a.d, a.G, a.E, st)) != cudaSuccess) return err;
    launch_select_any(a, logits, nullptr, nullptr, gidx, eidx, gate, st);
    prof_mark("router_select", st);
    launch_pdl(router_across_kernel, dim3((a.T + 255) / 256), dim3(256), 0, st, (const float*)logits, a.T, a.G, a.E,
               a.k, a.ke, (const int32_t*)eidx, gate, (const int32_t*)nullptr, (const int*)nullptr);
    prof_mark("router_across", st);
    return cudaGetLastError();
  }
  if (!fused_route_ok(a) && route_tc_ok(a)) {
    // tensor-core logits with verification, then the canonical order for the unverified tokens
    if (!status_zeroed && (err = cudaMemsetAsync(&status->route_redo, 0, sizeof(int), st)) != cudaSuccess)
      return err;
    if ((err = launch_route_tc(a, x, wg, bg, we, gidx, eidx, gate, redo, status, st)) != cudaSuccess) return err;
    const int* n = &status->route_redo;
    launch_pdl(router_exact_list_kernel, dim3(148), dim3(256), 0, st, (const __nv_bfloat16*)x,
               (const __nv_bfloat16*)wg, bg, (const __nv_bfloat16*)we, (const int32_t*)redo, n, a.d, a.G, a.E, logits);
    prof_mark("router_exact_list", st);
    launch_select_any(a, logits, redo, n, gidx, eidx, gate, st);
    prof_mark("router_select_list", st);
    if (a.across) {
      // the tensor-core router set the verified tokens' gates itself; the listed ones here
      launch_pdl(router_across_kernel, dim3(148), dim3(256), 0, st, (const float*)logits, a.T, a.G, a.E, a.k, a.ke,
                 (const int32_t*)eidx, gate, (const int32_t*)redo, n);
      prof_mark("router_across_list", st);
    }
    return cudaGetLastError();
  }
  if (launch_fused_route(a, x, wg, bg, we, gidx, eidx, gate, st, &err)) return err != cudaSuccess ? err : cudaGetLastError();
  err = launch_logits(a, a.bf16, x, wg, bg, we, logits, a.T, a.d, a.G, a.E, st);
  if (err != cudaSuccess) return err;
  launch_select_any(a, logits, nullptr, nullptr, gidx, eidx, gate, st);
  prof_mark("router_select", st);
  return cudaGetLastError();
}

}  // namespace moe
