// Expert computation on CUDA cores (FP32 arithmetic): the path for FP32 layers.
//
// "Breaking the MoE LLM Trilemma" (paper notes), key design 2: W~_i x = W_base^g x + B_i (A_i^T x);
// the base product is formed once per (token, group) row and shared by the row's k_e experts.
// Expert body: SwiGLU FFN W~_down (silu(W~_gate x) * W~_up x) ("混合专家模型的路由机制与工程落地"
// section 1.2), gated sum over the row's experts.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int BM = 64, BN = 64, BK = 32;

// Maps a tile index to (group, first row of the tile) from device row offsets; false if unused.
__device__ __forceinline__ bool tile_of(const int32_t* row_begin, int G, int tile, int& g, int& r0,
                                        int& r1) {
  for (int gg = 0; gg < G; ++gg) {
    const int b = row_begin[gg], e = row_begin[gg + 1];
    const int nt = (e - b + BM - 1) / BM;
    if (tile < nt) {
      g = gg;
      r0 = b + tile * BM;
      r1 = e;
      return true;
    }
    tile -= nt;
  }
  return false;
}
}  // namespace

// U[i][s][m][k] = A_{m,e}^T x_t for m in (gate, up): one warp per (row, slot).
template <typename T>
__global__ void resid_in_kernel(const T* __restrict__ x, ResidView Ag, ResidView Au,
                                const int32_t* __restrict__ eidx, const int32_t* __restrict__ row_asg,
                                int R, int d, int kg, int ke, int r, float* __restrict__ U) {
  pdl_wait();
  pdl_trigger();
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (gw >= R * ke) return;
  const int i = gw / ke, s = gw % ke;
  const int b = row_asg[i], t = b / kg, j = b % kg;
  const int e = eidx[(size_t)t * kg * ke + j * ke + s];
  const T* xt = x + (size_t)t * d;
  for (int m = 0; m < 2; ++m) {
    const ResidView& A = m == 0 ? Ag : Au;
    for (int kk = 0; kk < r; ++kk) {
      float acc = 0.f;
      for (int c = lane; c < d; c += 32) acc += A.at(e, kk, c) * to_f32(xt[c]);
      for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) U[(((size_t)i * ke + s) * 2 + m) * r + kk] = acc;
    }
  }
}

// Gate/up base GEMM per group with the residual + SwiGLU + gating epilogue.
template <typename T>
__global__ void __launch_bounds__(256) ffn_up_kernel(
    const T* __restrict__ x, const T* __restrict__ wg, const T* __restrict__ wu, ResidView Bg,
    ResidView Bu, const float* __restrict__ U, const int32_t* __restrict__ eidx,
    const float* __restrict__ gate, const int32_t* __restrict__ row_asg,
    const int32_t* __restrict__ row_begin, int G, int d, int f, int kg, int ke, int r,
    float* __restrict__ H, float* __restrict__ hsum) {
  pdl_wait();
  pdl_trigger();
  __shared__ float Xs[BM][BK + 1];
  __shared__ float Gs[BN][BK + 1];
  __shared__ float Us[BN][BK + 1];
  __shared__ int tok[BM];
  int g, r0, r1;
  if (!tile_of(row_begin, G, blockIdx.y, g, r0, r1)) return;
  const int c0 = blockIdx.x * BN;
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  if (tid < BM) tok[tid] = (r0 + tid < r1) ? row_asg[r0 + tid] / kg : -1;
  __syncthreads();
  const T* Wg = wg + (size_t)g * f * d;
  const T* Wu = wu + (size_t)g * f * d;
  float ag[4][4] = {}, au[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += BK) {
    for (int idx = tid; idx < BM * BK; idx += 256) {
      const int rr = idx / BK, kk = idx % BK;
      const int t = tok[rr];
      Xs[rr][kk] = t >= 0 ? to_f32(x[(size_t)t * d + k0 + kk]) : 0.f;
      const int c = c0 + rr;
      Gs[rr][kk] = c < f ? to_f32(Wg[(size_t)c * d + k0 + kk]) : 0.f;
      Us[rr][kk] = c < f ? to_f32(Wu[(size_t)c * d + k0 + kk]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float xv[4], gv[4], uv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) xv[a] = Xs[ty * 4 + a][kk];
#pragma unroll
      for (int b = 0; b < 4; ++b) { gv[b] = Gs[tx * 4 + b][kk]; uv[b] = Us[tx * 4 + b][kk]; }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) { ag[a][b] += xv[a] * gv[b]; au[a][b] += xv[a] * uv[b]; }
    }
    __syncthreads();
  }
  const int k = kg * ke;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = r0 + ty * 4 + a;
    if (i >= r1) continue;
    const int bsg = row_asg[i], t = bsg / kg, j = bsg % kg;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int c = c0 + tx * 4 + b;
      if (c >= f) continue;
      float hs = 0.f;
      for (int s = 0; s < ke; ++s) {
        const int e = eidx[(size_t)t * k + j * ke + s];
        const float gt = gate[(size_t)t * k + j * ke + s];
        const float* u = U + ((size_t)i * ke + s) * 2 * r;
        float av = ag[a][b], bv = au[a][b];
        for (int kk = 0; kk < r; ++kk) {
          av += u[kk] * Bg.at(e, kk, c);
          bv += u[r + kk] * Bu.at(e, kk, c);
        }
        const float h = silu_f(av) * bv;
        H[((size_t)i * ke + s) * f + c] = h;
        hs += gt * h;
      }
      hsum[(size_t)i * f + c] = hs;
    }
  }
}

// V[i][s][k] = A_{down,e}^T h_s: one warp per (row, slot).
__global__ void resid_out_kernel(const float* __restrict__ H, ResidView Ad,
                                 const int32_t* __restrict__ eidx, const int32_t* __restrict__ row_asg,
                                 int R, int f, int kg, int ke, int r, float* __restrict__ V) {
  pdl_wait();
  pdl_trigger();
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (gw >= R * ke) return;
  const int i = gw / ke, s = gw % ke;
  const int b = row_asg[i], t = b / kg, j = b % kg;
  const int e = eidx[(size_t)t * kg * ke + j * ke + s];
  const float* h = H + ((size_t)i * ke + s) * f;
  for (int kk = 0; kk < r; ++kk) {
    float acc = 0.f;
    for (int c = lane; c < f; c += 32) acc += Ad.at(e, kk, c) * h[c];
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) V[((size_t)i * ke + s) * r + kk] = acc;
  }
}

// Down base GEMM per group + gated down residual; rows scattered to token order y_rows[t][j].
template <typename T>
__global__ void __launch_bounds__(256) ffn_down_kernel(
    const float* __restrict__ hsum, const T* __restrict__ wd, ResidView Bd, const float* __restrict__ V,
    const int32_t* __restrict__ eidx, const float* __restrict__ gate,
    const int32_t* __restrict__ row_asg, const int32_t* __restrict__ row_begin, int G, int d, int f,
    int kg, int ke, int r, T* __restrict__ y_rows) {
  pdl_wait();
  pdl_trigger();
  __shared__ float Hs[BM][BK + 1];
  __shared__ float Ws[BN][BK + 1];
  int g, r0, r1;
  if (!tile_of(row_begin, G, blockIdx.y, g, r0, r1)) return;
  const int c0 = blockIdx.x * BN;
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  const T* Wd = wd + (size_t)g * d * f;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < f; k0 += BK) {
    for (int idx = tid; idx < BM * BK; idx += 256) {
      const int rr = idx / BK, kk = idx % BK;
      const int i = r0 + rr;
      Hs[rr][kk] = i < r1 ? hsum[(size_t)i * f + k0 + kk] : 0.f;
      const int c = c0 + rr;
      Ws[rr][kk] = c < d ? to_f32(Wd[(size_t)c * f + k0 + kk]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float hv[4], wv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) hv[a] = Hs[ty * 4 + a][kk];
#pragma unroll
      for (int b = 0; b < 4; ++b) wv[b] = Ws[tx * 4 + b][kk];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] += hv[a] * wv[b];
    }
    __syncthreads();
  }
  const int k = kg * ke;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = r0 + ty * 4 + a;
    if (i >= r1) continue;
    const int bsg = row_asg[i], t = bsg / kg, j = bsg % kg;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int c = c0 + tx * 4 + b;
      if (c >= d) continue;
      float v = acc[a][b];
      for (int s = 0; s < ke; ++s) {
        const int e = eidx[(size_t)t * k + j * ke + s];
        const float gt = gate[(size_t)t * k + j * ke + s];
        const float* vv = V + ((size_t)i * ke + s) * r;
        float rs = 0.f;
        for (int kk = 0; kk < r; ++kk) rs += vv[kk] * Bd.at(e, kk, c);
        v += gt * rs;
      }
      y_rows[((size_t)t * kg + j) * d + c] = from_f32<T>(v);
    }
  }
}

template <typename T>
static cudaError_t run(const LayerArgs& a, const void* x, const void* wg, const void* wu,
                       const void* wd, const ResidPtrs& rp, const int32_t* eidx, const float* gate,
                       const int32_t* row_asg, const int32_t* row_begin, void* y_rows,
                       const FfnBufs& b, cudaStream_t st) {
  const int R = a.R, r = a.r;
  const int tiles = (R + BM - 1) / BM + a.G;
  if (r > 0) {
    const int warps = R * a.ke;
    launch_pdl(resid_in_kernel<T>, dim3((warps * 32 + 255) / 256), dim3(256), 0, st, (const T*)x, rp.A[0], rp.A[1],
               eidx, row_asg, R, a.d, a.kg, a.ke, r, b.U);
  prof_mark("resid_in", st);
  }
  launch_pdl(ffn_up_kernel<T>, dim3((a.f + BN - 1) / BN, tiles), dim3(256), 0, st, (const T*)x, (const T*)wg,
             (const T*)wu, rp.B[0], rp.B[1], (const float*)b.U, eidx, gate, row_asg, row_begin, a.G, a.d, a.f, a.kg,
             a.ke, r, b.H, b.hsum);
  prof_mark("ffn_up_simt", st);
  if (r > 0) {
    const int warps = R * a.ke;
    launch_pdl(resid_out_kernel, dim3((warps * 32 + 255) / 256), dim3(256), 0, st, (const float*)b.H, rp.A[2], eidx,
               row_asg, R, a.f, a.kg, a.ke, r, b.V);
  prof_mark("resid_out", st);
  }
  launch_pdl(ffn_down_kernel<T>, dim3((a.d + BN - 1) / BN, tiles), dim3(256), 0, st, (const float*)b.hsum,
             (const T*)wd, rp.B[2], (const float*)b.V, eidx, gate, row_asg, row_begin, a.G, a.d, a.f, a.kg, a.ke, r,
             (T*)y_rows);
  prof_mark("ffn_down_simt", st);
  return cudaGetLastError();
}

cudaError_t launch_ffn_simt(const LayerArgs& a, const void* x, const void* wg, const void* wu,
                            const void* wd, const ResidPtrs& rp, const int32_t* eidx,
                            const float* gate, const int32_t* row_asg, const int32_t* row_begin,
                            void* y_rows, const FfnBufs& b, cudaStream_t st) {
  if (a.R == 0) return cudaSuccess;
  return a.bf16 ? run<__nv_bfloat16>(a, x, wg, wu, wd, rp, eidx, gate, row_asg, row_begin, y_rows, b, st)
                : run<float>(a, x, wg, wu, wd, rp, eidx, gate, row_asg, row_begin, y_rows, b, st);
}

// y[t] = sum_j y_rows[t][j], FP32 sum in slot order.
template <typename T>
__global__ void combine_kernel(const T* __restrict__ yr, T* __restrict__ y, int Tn, int d, int kg) {
  pdl_wait();
  pdl_trigger();
  const size_t n = (size_t)Tn * d;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < n; idx += (size_t)gridDim.x * blockDim.x) {
    const size_t t = idx / d, c = idx % d;
    float acc = 0.f;
    for (int j = 0; j < kg; ++j) acc += to_f32(yr[(t * kg + j) * d + c]);
    y[idx] = from_f32<T>(acc);
  }
}

// BF16, 8 columns per thread.
__global__ void combine_bf16x8_kernel(const __nv_bfloat16* __restrict__ yr, __nv_bfloat16* __restrict__ y, int Tn,
                                      int d, int kg) {
  pdl_wait();
  pdl_trigger();
  const size_t n8 = (size_t)Tn * d / 8;
  for (size_t w = blockIdx.x * (size_t)blockDim.x + threadIdx.x; w < n8; w += (size_t)gridDim.x * blockDim.x) {
    const size_t t = w / (d / 8), c = (w % (d / 8)) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < kg; ++j) {
      const uint4 v = *reinterpret_cast<const uint4*>(yr + (t * kg + j) * d + c);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += __uint_as_float(u[q] << 16);
        acc[2 * q + 1] += __uint_as_float(u[q] & 0xFFFF0000u);
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      o[q] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(y + t * d + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_combine(const LayerArgs& a, const void* y_rows, void* y, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  if (a.kg == 1) {
    if (y_rows == y) return cudaSuccess;
    return cudaMemcpyAsync(y, y_rows, (size_t)a.T * a.d * (a.bf16 ? 2 : 4), cudaMemcpyDeviceToDevice, st);
  }
  const size_t n = (size_t)a.T * a.d;
  const int blocks = (int)((n + 255) / 256 < 148 * 16 ? (n + 255) / 256 : 148 * 16);
  if (a.bf16)
    launch_pdl(combine_bf16x8_kernel, dim3(blocks), dim3(256), 0, st, (const __nv_bfloat16*)y_rows, (__nv_bfloat16*)y,
               a.T, a.d, a.kg);
  else
    launch_pdl(combine_kernel<float>, dim3(blocks), dim3(256), 0, st, (const float*)y_rows, (float*)y, a.T, a.d,
               a.kg);
  prof_mark("combine", st);
  return cudaGetLastError();
}

}  // namespace moe
