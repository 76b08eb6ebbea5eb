// Device-side U = A^T x on the CUDA cores for batches of few rows (decode), shared by the U
// kernel and the fused decode pre-pass.  "Breaking the MoE LLM Trilemma" (paper notes), key
// design 2: the residual is applied as B (A^T x), and A is INT4 (key design 4).
#pragma once
#include "common.cuh"

namespace moe {

// Residual factors and the stacks built from them (the tensor-core path's weight preparation).
struct PrepArgs {
  ResidView A[3], B[3];
  __nv_bfloat16 *Ain, *Adn, *Bdn;
  __half *Bgs, *Bus;
  __half* Adt;          // A_down^T transposed, FP16 dequantised: [G][f][KRP] (NULL: not built)
  int G, K, d, f, r, KRP;
  bool need_ain;        // the U GEMM reads Ain (the CUDA-core U kernel reads the codes itself)
  bool adn_f16;         // Adn holds FP16 dequantised values (else BF16 codes, scaled later)
};

// ------------------------------------------------------------------------------------------
// 3'. U on the CUDA cores, for batches of few rows (decode): block (row i, matrix m) computes
//     (blocks m = 0 also write the gathered row X[i] of step 2)
//     U[i][m*KRP + o] = sum_c x[t(i)][c] A_m,e_j^T[k][c] (o = j*r + k) for the K experts of the
//     row's group straight from the INT4 codes; block z of the row takes 32 of them, warp w four,
//     lanes stride over c in 32-element chunks (one 16-byte load of codes per output and chunk,
//     four chunks' loads in flight together), FP32 accumulation, FP16 out, padding columns zero.
//     Codes become BF16 values without a per-element conversion: a nibble q or'ed into the
//     mantissa of the BF16 number 128 (bits 0x4300) is the BF16 number 128 + q, and subtracting
//     136 leaves q - 8 exactly (the exponent-bias conversion used by weight-only quantised GEMM
//     kernels, e.g. Kim et al., "Who Says Elephants Can't Run", 2022); the mixed-precision FMA
//     then multiplies BF16 x by it exactly and rounds once into the FP32 sum.
// ------------------------------------------------------------------------------------------
template <bool AH, bool BH>
__device__ __forceinline__ float fma_bf16_sel(uint32_t a, uint32_t b, float c) {
  float d;
  if (AH && BH)
    asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
        " fma.rn.f32.bf16 %0, ah, bh, %3;\n}" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  else if (AH)
    asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
        " fma.rn.f32.bf16 %0, ah, bl, %3;\n}" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  else if (BH)
    asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
        " fma.rn.f32.bf16 %0, al, bh, %3;\n}" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  else
    asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
        " fma.rn.f32.bf16 %0, al, bl, %3;\n}" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}

// Two BF16 pairs (q - 8) from two code bytes: for bytes (b_lo, b_hi) of w selected by `sel`,
// P = (hi nibble of b_lo, hi nibble of b_hi), Q = (lo nibble of b_lo, lo nibble of b_hi).
__device__ __forceinline__ void code_pairs(uint32_t w, uint32_t sel, uint32_t& P, uint32_t& Q) {
  const uint32_t r = __byte_perm(w, 0u, sel);               // [b_lo, 0, b_hi, 0]
  const uint32_t p = ((r >> 4) & 0x000F000Fu) | 0x43004300u;
  const uint32_t q = (r & 0x000F000Fu) | 0x43004300u;
  const __nv_bfloat162 off = __floats2bfloat162_rn(136.f, 136.f);
  __nv_bfloat162 pp = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&p), off);
  __nv_bfloat162 qq = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&q), off);
  P = *reinterpret_cast<uint32_t*>(&pp);
  Q = *reinterpret_cast<uint32_t*>(&qq);
}

// sum over 8 elements: x pairs X0 = (x0, x1) .. X3 = (x6, x7), code word w (element 2b = high
// nibble of byte b, element 2b + 1 = low nibble)
__device__ __forceinline__ float dot8_int4(uint32_t w, uint32_t X0, uint32_t X1, uint32_t X2, uint32_t X3, float acc) {
  uint32_t P0, Q0, P1, Q1;
  code_pairs(w, 0x4140u, P0, Q0);                          // (e0, e2), (e1, e3)
  code_pairs(w, 0x4342u, P1, Q1);                          // (e4, e6), (e5, e7)
  acc = fma_bf16_sel<false, false>(X0, P0, acc);
  acc = fma_bf16_sel<true, false>(X0, Q0, acc);
  acc = fma_bf16_sel<false, true>(X1, P0, acc);
  acc = fma_bf16_sel<true, true>(X1, Q0, acc);
  acc = fma_bf16_sel<false, false>(X2, P1, acc);
  acc = fma_bf16_sel<true, false>(X2, Q1, acc);
  acc = fma_bf16_sel<false, true>(X3, P1, acc);
  acc = fma_bf16_sel<true, true>(X3, Q1, acc);
  return acc;
}

constexpr int kUSimtOut = 4;    // outputs per warp
constexpr int kUSimtChunks = 4; // 32-element chunks per lane whose loads are in flight together

// One (row i, matrix m, output block z) item of the CUDA-core U: stages the row's x in `xs` (d
// BF16 values of shared memory; one __syncthreads), then each warp computes its four outputs.
// Called by every thread of the CTA; a warp without outputs returns early after the barrier.
__device__ __forceinline__ void u_simt_item(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ row_asg,
                                            const int32_t* __restrict__ eidx, const PrepArgs& p, const GroupTable& tab,
                                            int kg, int ke, __half* __restrict__ U, __nv_bfloat16* __restrict__ X,
                                            int i, int m, int z, __nv_bfloat16* xs) {
  const int d = p.d, KRP = p.KRP, r = p.r, K = p.K;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int b = row_asg[i], t = b / kg, jg = b % kg;
  const int g = tab.group_of[eidx[(size_t)t * kg * ke + jg * ke]];
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(x + (size_t)t * d + c);
    *reinterpret_cast<uint4*>(xs + c) = v;
    if (m == 0 && z == 0) *reinterpret_cast<uint4*>(X + (size_t)i * d + c) = v;   // the row in (group, token) order
  }
  __syncthreads();
  const ResidView& v = p.A[m];
  const uint8_t* codes = (const uint8_t*)v.vals;
  const int nchunk = d / 32;                                  // 32-element chunks of a rank row
  // block z takes outputs [z * nwarps * 4, ...) of the row's 2 x KRP; warp w four of them
  const int ob = (z * nwarps + warp) * kUSimtOut;
  if (ob >= KRP) return;
  const uint8_t* crow[kUSimtOut];
  const __half* srow[kUSimtOut];
  bool live[kUSimtOut];
#pragma unroll
  for (int q = 0; q < kUSimtOut; ++q) {
    const int o = ob + q, j = o / r, k = o % r;
    live[q] = o < KRP && j < K;
    const size_t row = live[q] ? (size_t)tab.member[g * K + j] * r + k : 0;
    crow[q] = codes + row * (d / 2);
    srow[q] = v.scales + row * (d / kQGroup);
  }
  float acc[kUSimtOut];
#pragma unroll
  for (int q = 0; q < kUSimtOut; ++q) acc[q] = 0.f;
  for (int c0 = lane; c0 < nchunk; c0 += 32 * kUSimtChunks) {
    // every load of this group of chunks first, then the arithmetic
    uint4 cw[kUSimtChunks][kUSimtOut];
    float sc[kUSimtChunks][kUSimtOut];
#pragma unroll
    for (int u = 0; u < kUSimtChunks; ++u) {
      const int c = c0 + 32 * u;
#pragma unroll
      for (int q = 0; q < kUSimtOut; ++q) {
        const bool on = live[q] && c < nchunk;
        cw[u][q] = on ? __ldg(reinterpret_cast<const uint4*>(crow[q] + (size_t)c * 16)) : make_uint4(0, 0, 0, 0);
        sc[u][q] = on ? __half2float(srow[q][c >> 1]) : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kUSimtChunks; ++u) {
      const int c = c0 + 32 * u;
      if (c >= nchunk) break;
      const uint4* xp = reinterpret_cast<const uint4*>(xs + c * 32);
      const uint4 x0 = xp[0], x1 = xp[1], x2 = xp[2], x3 = xp[3];
#pragma unroll
      for (int q = 0; q < kUSimtOut; ++q) {
        float s = 0.f;
        s = dot8_int4(cw[u][q].x, x0.x, x0.y, x0.z, x0.w, s);
        s = dot8_int4(cw[u][q].y, x1.x, x1.y, x1.z, x1.w, s);
        s = dot8_int4(cw[u][q].z, x2.x, x2.y, x2.z, x2.w, s);
        s = dot8_int4(cw[u][q].w, x3.x, x3.y, x3.z, x3.w, s);
        acc[q] = fmaf(s, sc[u][q], acc[q]);
      }
    }
  }
#pragma unroll
  for (int q = 0; q < kUSimtOut; ++q)
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], off);
  if (lane < kUSimtOut && ob + lane < KRP) {
    float val = acc[0];
#pragma unroll
    for (int q = 1; q < kUSimtOut; ++q) val = lane == q ? acc[q] : val;
    U[(size_t)i * 2 * KRP + m * KRP + ob + lane] = __float2half_rn(val);
  }
}

}  // namespace moe
