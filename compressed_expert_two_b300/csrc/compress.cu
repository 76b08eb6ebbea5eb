// The compression step that produces the layer's weights, on the GPU.
//
// "Breaking the MoE LLM Trilemma" (paper notes), key design 2: each group's base is the mean of its
// experts' weights, each expert keeps a rank-r residual initialised by a truncated SVD of
// (W_i - W_base^g), quality is the Frobenius reconstruction error; key design 4: the base stays
// 16-bit (BF16 here), the residual factors go to INT4.
//
// Per matrix kind (gate, up or down) and for every expert at once:
//   1. base[g] = bf16(fl32(sum of the members' W, ascending id) / K)           (cmp_mean_kernel)
//   2. truncated SVD of R_i = W_i - base[g(i)] by a randomised range finder with subspace
//      iteration (Halko, Martinsson, Tropp, "Finding structure with randomness", 2011, algorithms
//      4.4 and 5.1): Y = R Omega, then q times (Z = R^T Q, Y = R orth(Z)), every product followed by
//      an orthonormalisation Q = Y V D^{-1/2} from the eigen-decomposition Y^T Y = V D V^T; then
//      Z = R^T Q, Z^T Z = U S^2 U^T, and R ~ (Q U) S (Z U S^{-1})^T, so that
//      B = Q U_r S_r^{1/2}, A = Z U_r S_r^{-1/2}.  R is never stored: every product forms it on
//      the fly from the BF16 W and base (cmp_tsmm_kernel, FP32 on the CUDA cores; the products are
//      tall and skinny, l <= 64 columns, and the two BF16 streams bound them).
//   3. INT4 group-64 codes and FP16 scales of the rank-major rows A^T, B^T (cmp_quant_kernel).
//   4. ||W_i - (base + B_dq A_dq^T)||_F / ||W_i||_F from the stored codes (cmp_err_kernel).
// The small eigenproblems (64 x 64, FP32 from FP64 Grams) run as cyclic Jacobi sweeps in one CTA
// per expert.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kCL = 64;          // sketch columns held (l <= 64; unused columns stay zero)

struct CmpTable {                // members of each group, ascending id; group of each expert
  int E, G, K;
  uint8_t member[kMaxE];
  uint8_t group_of[kMaxE];
};

// ------------------------------------------------------------------------------------------
// 1. group mean
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cmp_mean_kernel(const __nv_bfloat16* __restrict__ W, CmpTable tab, size_t n,
                                                       __nv_bfloat16* __restrict__ base) {
  pdl_wait();
  pdl_trigger();
  const size_t n8 = n / 8;
  const float Kf = (float)tab.K;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < (size_t)tab.G * n8;
       i += (size_t)gridDim.x * blockDim.x) {
    const int g = (int)(i / n8);
    const size_t c8 = i % n8;
    float s[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) s[u] = 0.f;
    for (int m = 0; m < tab.K; ++m) {
      const int e = tab.member[g * tab.K + m];
      const uint4 v = *reinterpret_cast<const uint4*>(W + (size_t)e * n + c8 * 8);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        s[2 * u] = __fadd_rn(s[2 * u], __uint_as_float(w[u] << 16));
        s[2 * u + 1] = __fadd_rn(s[2 * u + 1], __uint_as_float(w[u] & 0xffff0000u));
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(__fdiv_rn(s[2 * u], Kf), __fdiv_rn(s[2 * u + 1], Kf));
      o[u] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(base + (size_t)g * n + c8 * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ------------------------------------------------------------------------------------------
// 2a. tall-skinny products with R = W_e - base_g formed on the fly (FP32)
//   ROW (COL = false): out[e][o][j] = sum_c R[o][c] X[c][j]   (M = d_out rows, K = d_in)
//   COL (COL = true):  out[e][c][j] = sum_o R[o][c] X[o][j]   (M = d_in rows,  K = d_out)
// X is [K][64] per expert (x_stride floats apart; 0: one X for every expert).  A CTA of 128
// threads computes 128 rows x 64 columns, each thread an 8 x 8 block; K runs in chunks of 32
// staged in shared memory (R as As[k][m], X as Bs[k][j]) with the next chunk's global loads held
// in registers meanwhile.
// ------------------------------------------------------------------------------------------
constexpr int kTsM = 128, kTsK = 32, kTsPad = 4;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    f[2 * u] = __uint_as_float(w[u] << 16);
    f[2 * u + 1] = __uint_as_float(w[u] & 0xffff0000u);
  }
}

template <bool COL>
__global__ void __launch_bounds__(128) cmp_tsmm_kernel(const __nv_bfloat16* __restrict__ W,
                                                       const __nv_bfloat16* __restrict__ base, CmpTable tab,
                                                       int d_out, int d_in, const float* __restrict__ X,
                                                       size_t x_stride, float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  __shared__ __align__(16) float As[kTsK][kTsM + kTsPad];
  __shared__ __align__(16) float Bs[kTsK][kCL];
  const int e = blockIdx.y, g = tab.group_of[e];
  const int tid = threadIdx.x;
  const int M = COL ? d_in : d_out, K = COL ? d_out : d_in;
  const int m0 = blockIdx.x * kTsM;
  const __nv_bfloat16* We = W + (size_t)e * d_out * d_in;
  const __nv_bfloat16* Bg = base + (size_t)g * d_out * d_in;
  const float* Xe = X + (size_t)e * x_stride;

  // global -> registers for chunk k0 (4 pieces of 8 R values, 4 float4 of X)
  uint4 rw[4], rb[4];
  float4 rx[4];
  auto load = [&](int k0) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      size_t off;
      if (COL) {
        const int idx = p * 128 + tid;                   // 32 rows o x 16 pieces of 8 columns c
        off = (size_t)(k0 + idx / 16) * d_in + m0 + (idx % 16) * 8;
      } else {
        off = (size_t)(m0 + tid) * d_in + k0 + p * 8;    // row o = m0 + tid, 4 pieces of 8 columns
      }
      rw[p] = *reinterpret_cast<const uint4*>(We + off);
      rb[p] = *reinterpret_cast<const uint4*>(Bg + off);
      const int xi = p * 128 + tid;                      // 32 rows x 16 float4
      rx[p] = *reinterpret_cast<const float4*>(Xe + (size_t)(k0 + xi / 16) * kCL + (xi % 16) * 4);
    }
  };
  auto store = [&]() {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      float fw[8], fb[8];
      bf16x8_to_f32(rw[p], fw);
      bf16x8_to_f32(rb[p], fb);
      if (COL) {
        const int idx = p * 128 + tid, k = idx / 16, m = (idx % 16) * 8;
        float4* d = reinterpret_cast<float4*>(&As[k][m]);
        d[0] = make_float4(__fsub_rn(fw[0], fb[0]), __fsub_rn(fw[1], fb[1]), __fsub_rn(fw[2], fb[2]),
                           __fsub_rn(fw[3], fb[3]));
        d[1] = make_float4(__fsub_rn(fw[4], fb[4]), __fsub_rn(fw[5], fb[5]), __fsub_rn(fw[6], fb[6]),
                           __fsub_rn(fw[7], fb[7]));
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) As[p * 8 + u][tid] = __fsub_rn(fw[u], fb[u]);
      }
      const int xi = p * 128 + tid;
      *reinterpret_cast<float4*>(&Bs[xi / 16][(xi % 16) * 4]) = rx[p];
    }
  };

  const int tm = tid & 15, tj = tid >> 4;                // rows tm*8.., columns tj*8..
  float2 acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.f, 0.f);

  load(0);
  for (int k0 = 0; k0 < K; k0 += kTsK) {
    __syncthreads();
    store();
    __syncthreads();
    if (k0 + kTsK < K) load(k0 + kTsK);
#pragma unroll 4
    for (int k = 0; k < kTsK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[k][tm * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[k][tm * 8 + 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[k][tj * 8]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[k][tj * 8 + 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float2 b[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                           make_float2(b1.z, b1.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fma2(make_float2(a[i], a[i]), b[j], acc[i][j]);
    }
  }
  float* oe = out + (size_t)e * M * kCL;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float4* d = reinterpret_cast<float4*>(oe + (size_t)(m0 + tm * 8 + i) * kCL + tj * 8);
    d[0] = make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y);
    d[1] = make_float4(acc[i][2].x, acc[i][2].y, acc[i][3].x, acc[i][3].y);
  }
}

// ------------------------------------------------------------------------------------------
// 2b. Gram matrices  gram[e] += Y_e^T Y_e  (FP64 accumulators, zeroed before the launch).
// grid (row splits, E); each thread a 4 x 4 block of the 64 x 64 result over 64-row chunks.
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cmp_gram_kernel(const float* __restrict__ Y, int rows, int rows_per_cta,
                                                       double* __restrict__ gram) {
  pdl_wait();
  pdl_trigger();
  __shared__ __align__(16) float Ys[64][kCL];
  const int e = blockIdx.y, tid = threadIdx.x;
  const int bi = (tid & 15) * 4, bj = (tid >> 4) * 4;
  const float* Ye = Y + (size_t)e * rows * kCL;
  float acc[4][4] = {};
  const int r_begin = blockIdx.x * rows_per_cta, r_end = min(rows, r_begin + rows_per_cta);
  for (int r0 = r_begin; r0 < r_end; r0 += 64) {
    __syncthreads();
    for (int i = tid; i < 64 * 16; i += 256) {
      const int rr = i / 16, c4 = (i % 16) * 4;
      *reinterpret_cast<float4*>(&Ys[rr][c4]) =
          r0 + rr < r_end ? *reinterpret_cast<const float4*>(Ye + (size_t)(r0 + rr) * kCL + c4)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
#pragma unroll 8
    for (int rr = 0; rr < 64; ++rr) {
      const float4 a = *reinterpret_cast<const float4*>(&Ys[rr][bi]);
      const float4 b = *reinterpret_cast<const float4*>(&Ys[rr][bj]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
  }
  double* ge = gram + (size_t)e * kCL * kCL;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) atomicAdd(ge + (bi + i) * kCL + bj + j, (double)acc[i][j]);
}

// ------------------------------------------------------------------------------------------
// 2c. Symmetric 64 x 64 eigenproblem (cyclic Jacobi in FP32 -- the FP64 units of this part run at
// a small fraction of the FP32 rate -- one CTA of 256 threads per expert; the Gram comes in FP64
// and is rounded once).  Rotations of 32 disjoint index pairs (round-robin order) per step, 63
// steps per sweep, until the off-diagonal mass is below 1e-13 of the total (at most 20 sweeps).
// Then, by mode:
//   ORTH: M = V D^{-1/2}, the transform that orthonormalises Y: Q = Y M (directions whose
//         eigenvalue is below 1e-6 of the largest, which FP32 cannot resolve, are dropped: their
//         columns of M are zero; the next orthonormalisation pass sees a clean basis);
//   SVD:  eigenvalues descending, sigma_k = sqrt(lambda_k) for k < r, and the r-column transforms
//         P_B = U_r S^{1/2} and P_A = U_r S^{-1/2}, each column's sign fixed so that its largest
//         component is positive.
// Transforms are written FP32 [64][64] (P_B in columns 0..r-1, P_A in columns 32..32+r-1).
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cmp_eig_kernel(const double* __restrict__ gram, int mode, int r,
                                                      float* __restrict__ xform, float* __restrict__ sigma) {
  pdl_wait();
  pdl_trigger();
  constexpr int N = kCL;
  __shared__ float A[N][N + 1];
  __shared__ float V[N][N + 1];
  __shared__ float cs[N / 2][2];
  __shared__ int pr[N / 2][2];
  __shared__ float red[2][256];
  __shared__ int order[N];
  __shared__ float lam[N];
  const int e = blockIdx.x, tid = threadIdx.x;
  const double* ge = gram + (size_t)e * N * N;
  for (int i = tid; i < N * N; i += 256) {
    const int a = i / N, b = i % N;
    A[a][b] = (float)(0.5 * (ge[a * N + b] + ge[b * N + a]));   // exact symmetry
    V[a][b] = a == b ? 1.f : 0.f;
  }
  __syncthreads();
  for (int sweep = 0; sweep < 20; ++sweep) {
    float off = 0.f, tot = 0.f;
    for (int i = tid; i < N * N; i += 256) {
      const float v = A[i / N][i % N] * A[i / N][i % N];
      tot += v;
      if (i / N != i % N) off += v;
    }
    red[0][tid] = off;
    red[1][tid] = tot;
    __syncthreads();
    for (int s = 128; s > 0; s >>= 1) {
      if (tid < s) { red[0][tid] += red[0][tid + s]; red[1][tid] += red[1][tid + s]; }
      __syncthreads();
    }
    const float off_all = red[0][0], tot_all = red[1][0];
    __syncthreads();
    if (off_all <= 1e-13f * tot_all || tot_all == 0.f) break;
    for (int step = 0; step < N - 1; ++step) {
      if (tid < N / 2) {
        int p, q;
        if (tid == 0) { p = step; q = N - 1; }
        else { p = (step + tid) % (N - 1); q = (step - tid + (N - 1)) % (N - 1); }
        if (p > q) { const int t = p; p = q; q = t; }
        const float apq = A[p][q], app = A[p][p], aqq = A[q][q];
        float c = 1.f, s = 0.f;
        if (apq != 0.f) {
          const float tau = (aqq - app) / (2.f * apq);
          const float t = (tau >= 0.f ? 1.f : -1.f) / (fabsf(tau) + sqrtf(1.f + tau * tau));
          c = rsqrtf(1.f + t * t);
          s = t * c;
        }
        pr[tid][0] = p; pr[tid][1] = q; cs[tid][0] = c; cs[tid][1] = s;
      }
      __syncthreads();
      // rows: A <- J^T A
      for (int i = tid; i < (N / 2) * N; i += 256) {
        const int k = i / N, col = i % N, p = pr[k][0], q = pr[k][1];
        const float c = cs[k][0], s = cs[k][1], ap = A[p][col], aq = A[q][col];
        A[p][col] = c * ap - s * aq;
        A[q][col] = s * ap + c * aq;
      }
      __syncthreads();
      // columns: A <- A J, V <- V J
      for (int i = tid; i < (N / 2) * N; i += 256) {
        const int k = i / N, row = i % N, p = pr[k][0], q = pr[k][1];
        const float c = cs[k][0], s = cs[k][1];
        const float ap = A[row][p], aq = A[row][q];
        A[row][p] = c * ap - s * aq;
        A[row][q] = s * ap + c * aq;
        const float vp = V[row][p], vq = V[row][q];
        V[row][p] = c * vp - s * vq;
        V[row][q] = s * vp + c * vq;
      }
      __syncthreads();
    }
  }
  if (tid < N) lam[tid] = A[tid][tid];
  __syncthreads();
  if (tid < N) {            // rank of eigenvalue tid in descending order (ties: lower index first)
    int rank = 0;
    for (int j = 0; j < N; ++j) rank += (lam[j] > lam[tid]) || (lam[j] == lam[tid] && j < tid);
    order[rank] = tid;
  }
  __syncthreads();
  float* xe = xform + (size_t)e * N * N;
  const float lmax = fmaxf(lam[order[0]], 0.f);
  if (mode == 0) {
    for (int i = tid; i < N * N; i += 256) {
      const int row = i / N, col = i % N;
      const float l = lam[col];
      xe[i] = l > 1e-6f * lmax && l > 0.f ? V[row][col] * rsqrtf(l) : 0.f;
    }
  } else {
    for (int i = tid; i < N * N; i += 256) xe[i] = 0.f;
    __syncthreads();
    if (tid < r) {
      const int col = order[tid];
      const float sg = sqrtf(fmaxf(lam[col], 0.f));
      int big = 0;
      for (int row = 1; row < N; ++row)
        if (fabsf(V[row][col]) > fabsf(V[big][col])) big = row;
      const float sgn = V[big][col] < 0.f ? -1.f : 1.f;
      const float rb = sqrtf(sg), ra = sg > 0.f ? rsqrtf(sg) : 0.f;
      for (int row = 0; row < N; ++row) {
        xe[row * N + tid] = sgn * V[row][col] * rb;
        xe[row * N + 32 + tid] = sgn * V[row][col] * ra;
      }
      sigma[(size_t)e * r + tid] = sg;
    }
  }
}

// ------------------------------------------------------------------------------------------
// 2d. out = in M: in [E][rows][64], M [E][64][64] (columns c0 .. c0+ncols-1 used).
// transposed = 0: out [E][rows][64] (columns >= ncols zero); 1: out [E][ncols][rows] (rank-major).
// One warp per row; lane j holds in[row][j] and in[row][j+32], sums over shuffles.
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cmp_apply_kernel(const float* __restrict__ in, int rows,
                                                        const float* __restrict__ M, int c0, int ncols,
                                                        int transposed, float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  __shared__ float Ms[kCL][kCL + 1];
  const int e = blockIdx.y, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* Me = M + (size_t)e * kCL * kCL;
  for (int i = threadIdx.x; i < kCL * kCL; i += blockDim.x) Ms[i / kCL][i % kCL] = Me[i];
  __syncthreads();
  const float* ie = in + (size_t)e * rows * kCL;
  for (int row = blockIdx.x * 8 + warp; row < rows; row += gridDim.x * 8) {
    const float v0 = ie[(size_t)row * kCL + lane], v1 = ie[(size_t)row * kCL + 32 + lane];
    float o0 = 0.f, o1 = 0.f;       // output columns lane and lane + 32
#pragma unroll 8
    for (int j = 0; j < 32; ++j) {
      const float a = __shfl_sync(0xffffffffu, v0, j), b = __shfl_sync(0xffffffffu, v1, j);
      o0 = fmaf(a, Ms[j][c0 + lane], o0);
      o0 = fmaf(b, Ms[j + 32][c0 + lane], o0);
      if (c0 + lane + 32 < kCL) {
        o1 = fmaf(a, Ms[j][c0 + lane + 32], o1);
        o1 = fmaf(b, Ms[j + 32][c0 + lane + 32], o1);
      }
    }
    if (transposed) {
      float* oe = out + (size_t)e * ncols * rows;
      if (lane < ncols) oe[(size_t)lane * rows + row] = o0;
      if (lane + 32 < ncols) oe[(size_t)(lane + 32) * rows + row] = o1;
    } else {
      float* oe = out + (size_t)e * rows * kCL;
      oe[(size_t)row * kCL + lane] = lane < ncols ? o0 : 0.f;
      oe[(size_t)row * kCL + 32 + lane] = lane + 32 < ncols ? o1 : 0.f;
    }
  }
}

// ------------------------------------------------------------------------------------------
// 3. INT4 group-64 quantisation of FP32 rows [rows][n]: one warp per 64-element group, lane j
//    holding elements 2j (high nibble) and 2j + 1 (low nibble) of byte j.
//    scale = fp16_rn(absmax / 7), q = clamp(rint(w / scale), -7, 7) (FP32 division, 0 if scale 0)
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cmp_quant_kernel(const float* __restrict__ v, size_t groups,
                                                        uint8_t* __restrict__ codes, __half* __restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  for (size_t gi = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) / 32; gi < groups;
       gi += (size_t)gridDim.x * blockDim.x / 32) {
    const float2 w = *reinterpret_cast<const float2*>(v + gi * 64 + 2 * lane);
    float amax = fmaxf(fabsf(w.x), fabsf(w.y));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const __half s16 = __float2half_rn(__fdiv_rn(amax, 7.0f));
    const float s = __half2float(s16);
    auto code = [&](float x) {
      if (!(s > 0.f)) return 8;
      const float q = fminf(fmaxf(rintf(__fdiv_rn(x, s)), -7.f), 7.f);
      return (int)q + 8;
    };
    codes[gi * 32 + lane] = (uint8_t)((code(w.x) << 4) | code(w.y));
    if (lane == 0) scales[gi] = s16;
  }
}

// ------------------------------------------------------------------------------------------
// 4. Reconstruction error: acc[e] += (sum over the expert's elements of (W - base - B A^T)^2,
//    sum of W^2) with A, B dequantised from their codes; FP64 accumulators zeroed before.
//    CTA (column tile of 128, expert, row split): A^T's 128 columns of every rank, dequantised once
//    into shared memory; each warp then takes rows of the split, lane j holding 4 consecutive
//    columns, the row's r values of B dequantised by lanes 0..r-1 and shared by shuffles.
// ------------------------------------------------------------------------------------------
constexpr int kErrCols = 128;

__device__ __forceinline__ float dq4(const uint8_t* codes, const __half* scales, size_t row, int n, int c) {
  const uint8_t b = codes[row * (n / 2) + (c >> 1)];
  const int u = (c & 1) ? (b & 0xF) : (b >> 4);
  return (float)(u - 8) * __half2float(scales[row * (n / 64) + c / 64]);
}

__global__ void __launch_bounds__(256) cmp_err_kernel(const __nv_bfloat16* __restrict__ W,
                                                      const __nv_bfloat16* __restrict__ base, CmpTable tab,
                                                      int d_out, int d_in, int r, const uint8_t* __restrict__ Aq,
                                                      const __half* __restrict__ As, const uint8_t* __restrict__ Bq,
                                                      const __half* __restrict__ Bs, double* __restrict__ acc) {
  pdl_wait();
  pdl_trigger();
  __shared__ __align__(16) float Asm[32][kErrCols];
  __shared__ double red[2][8];
  const int e = blockIdx.y, g = tab.group_of[e];
  const int c_tile = blockIdx.x * kErrCols;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < r * kErrCols; i += blockDim.x) {
    const int k = i / kErrCols, c = i % kErrCols;
    Asm[k][c] = dq4(Aq, As, (size_t)e * r + k, d_in, c_tile + c);
  }
  __syncthreads();
  const int rows_per = (d_out + gridDim.z - 1) / gridDim.z;
  const int o_begin = blockIdx.z * rows_per, o_end = min(d_out, o_begin + rows_per);
  const int c0 = c_tile + lane * 4;
  double num = 0.0, den = 0.0;
  for (int o = o_begin + warp; o < o_end; o += 8) {
    const float bk_lane = lane < r ? dq4(Bq, Bs, (size_t)e * r + lane, d_out, o) : 0.f;
    const uint2 wv = *reinterpret_cast<const uint2*>(W + ((size_t)e * d_out + o) * d_in + c0);
    const uint2 bv = *reinterpret_cast<const uint2*>(base + ((size_t)g * d_out + o) * d_in + c0);
    const float w[4] = {__uint_as_float(wv.x << 16), __uint_as_float(wv.x & 0xffff0000u),
                        __uint_as_float(wv.y << 16), __uint_as_float(wv.y & 0xffff0000u)};
    const float b[4] = {__uint_as_float(bv.x << 16), __uint_as_float(bv.x & 0xffff0000u),
                        __uint_as_float(bv.y << 16), __uint_as_float(bv.y & 0xffff0000u)};
    float pred[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < r; ++k) {
      const float bk = __shfl_sync(0xffffffffu, bk_lane, k);
      const float4 a0 = *reinterpret_cast<const float4*>(&Asm[k][lane * 4]);
      pred[0] = fmaf(bk, a0.x, pred[0]); pred[1] = fmaf(bk, a0.y, pred[1]);
      pred[2] = fmaf(bk, a0.z, pred[2]); pred[3] = fmaf(bk, a0.w, pred[3]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const double dlt = (double)w[u] - (double)b[u] - (double)pred[u];
      num += dlt * dlt;
      den += (double)w[u] * (double)w[u];
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    num += __shfl_xor_sync(0xffffffffu, num, o);
    den += __shfl_xor_sync(0xffffffffu, den, o);
  }
  if (lane == 0) { red[0][warp] = num; red[1][warp] = den; }
  __syncthreads();
  if (threadIdx.x == 0) {
    double a = 0.0, b2 = 0.0;
    for (int w8 = 0; w8 < 8; ++w8) { a += red[0][w8]; b2 += red[1][w8]; }
    atomicAdd(acc + 2 * e, a);
    atomicAdd(acc + 2 * e + 1, b2);
  }
}

__global__ void cmp_err_final_kernel(const double* __restrict__ acc, int E, double* __restrict__ err) {
  pdl_wait();
  pdl_trigger();
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < E) err[e] = acc[2 * e + 1] > 0.0 ? sqrt(acc[2 * e] / acc[2 * e + 1]) : 0.0;
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
struct CmpPlan {
  size_t Om, Y, Q, Z, Zq, gram, xform, At, Bt, acc, total;
};

static size_t cmp_align(size_t v) { return (v + 255) & ~size_t(255); }

static CmpPlan cmp_plan(const CmpArgs& c) {
  CmpPlan p{};
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o = cmp_align(o + bytes); return at; };
  const size_t E = c.E;
  p.Om = take((size_t)c.d_in * kCL * 4);
  p.Y = take(E * c.d_out * kCL * 4);
  p.Q = take(E * c.d_out * kCL * 4);
  p.Z = take(E * c.d_in * kCL * 4);
  p.Zq = take(E * c.d_in * kCL * 4);
  p.gram = take(E * kCL * kCL * 8);
  p.xform = take(E * kCL * kCL * 4);
  p.At = take(E * c.r * c.d_in * 4);
  p.Bt = take(E * c.r * c.d_out * 4);
  p.acc = take(E * 2 * 8);
  p.total = o;
  return p;
}

size_t cmp_workspace_bytes(const CmpArgs& c) { return cmp_plan(c).total; }

static CmpTable cmp_table(const CmpArgs& c) {
  CmpTable t{};
  t.E = c.E; t.G = c.G; t.K = c.E / c.G;
  for (int i = 0; i < kMaxE; ++i) { t.member[i] = c.member[i]; t.group_of[i] = c.group_of[i]; }
  return t;
}

cudaError_t launch_quant_int4(const float* v, size_t rows, int n, uint8_t* codes, __half* scales, cudaStream_t st) {
  const size_t groups = rows * (size_t)(n / 64);
  if (groups == 0) return cudaSuccess;
  size_t blocks = (groups * 32 + 255) / 256;
  if (blocks > 148 * 16) blocks = 148 * 16;
  launch_pdl(cmp_quant_kernel, dim3((unsigned)blocks), dim3(256), 0, st, v, groups, codes, scales);
  prof_mark("cmp_quant", st);
  return cudaGetLastError();
}

cudaError_t launch_compress(const CmpArgs& c, const void* W, const float* omega, void* base_out, uint8_t* Aq,
                            __half* As, uint8_t* Bq, __half* Bs, float* sigma, double* err, float* At_out,
                            float* Bt_out, void* ws, cudaStream_t st) {
  const CmpPlan p = cmp_plan(c);
  const CmpTable tab = cmp_table(c);
  char* w = (char*)ws;
  float *Y = (float*)(w + p.Y), *Q = (float*)(w + p.Q), *Z = (float*)(w + p.Z), *Zq = (float*)(w + p.Zq);
  double* gram = (double*)(w + p.gram);
  float* xf = (float*)(w + p.xform);
  float* At = At_out ? At_out : (float*)(w + p.At);
  float* Bt = Bt_out ? Bt_out : (float*)(w + p.Bt);
  double* acc = (double*)(w + p.acc);
  const __nv_bfloat16* Wb = (const __nv_bfloat16*)W;
  __nv_bfloat16* base = (__nv_bfloat16*)base_out;
  const int E = c.E, d_out = c.d_out, d_in = c.d_in, r = c.r;
  cudaError_t e;

  // 1. base
  const size_t n = (size_t)d_out * d_in;
  {
    size_t blocks = ((size_t)c.G * (n / 8) + 255) / 256;
    if (blocks > 148 * 32) blocks = 148 * 32;
    launch_pdl(cmp_mean_kernel, dim3((unsigned)blocks), dim3(256), 0, st, Wb, tab, n, base);
    prof_mark("cmp_mean", st);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  auto rmul = [&](const float* X, size_t x_stride, float* out) {     // out = R X
    launch_pdl(cmp_tsmm_kernel<false>, dim3(d_out / kTsM, E), dim3(128), 0, st, Wb, (const __nv_bfloat16*)base, tab,
               d_out, d_in, X, x_stride, out);
    prof_mark("cmp_tsmm_row", st);
    return cudaGetLastError();
  };
  auto rtmul = [&](const float* X, float* out) {                     // out = R^T X
    launch_pdl(cmp_tsmm_kernel<true>, dim3(d_in / kTsM, E), dim3(128), 0, st, Wb, (const __nv_bfloat16*)base, tab,
               d_out, d_in, X, (size_t)d_out * kCL, out);
    prof_mark("cmp_tsmm_col", st);
    return cudaGetLastError();
  };
  auto gram_of = [&](const float* Y_, int rows) {
    cudaError_t er = cudaMemsetAsync(gram, 0, (size_t)E * kCL * kCL * 8, st);
    if (er != cudaSuccess) return er;
    const int per = 1024;
    launch_pdl(cmp_gram_kernel, dim3((rows + per - 1) / per, E), dim3(256), 0, st, Y_, rows, per, gram);
    prof_mark("cmp_gram", st);
    return cudaGetLastError();
  };
  auto eig = [&](int mode) {
    launch_pdl(cmp_eig_kernel, dim3(E), dim3(256), 0, st, (const double*)gram, mode, r, xf, sigma);
    prof_mark("cmp_eig", st);
    return cudaGetLastError();
  };
  auto apply = [&](const float* in, int rows, int c0, int ncols, int transposed, float* out) {
    launch_pdl(cmp_apply_kernel, dim3((rows + 7) / 8 < 4096 ? (rows + 7) / 8 : 4096, E), dim3(256), 0, st, in, rows,
               (const float*)xf, c0, ncols, transposed, out);
    prof_mark("cmp_apply", st);
    return cudaGetLastError();
  };
  auto orth = [&](float* Y_, int rows, float* out) {                 // out = Y V D^{-1/2}
    cudaError_t er;
    if ((er = gram_of(Y_, rows)) != cudaSuccess) return er;
    if ((er = eig(0)) != cudaSuccess) return er;
    return apply(Y_, rows, 0, kCL, 0, out);
  };

  // 2. randomised range finder with subspace iteration (the test matrix padded to 64 columns)
  float* Om = (float*)(w + p.Om);
  if ((e = cudaMemsetAsync(Om, 0, (size_t)d_in * kCL * 4, st)) != cudaSuccess) return e;
  if ((e = cudaMemcpy2DAsync(Om, kCL * 4, omega, (size_t)c.l * 4, (size_t)c.l * 4, d_in, cudaMemcpyDeviceToDevice,
                             st)) != cudaSuccess)
    return e;
  if ((e = rmul(Om, 0, Y)) != cudaSuccess) return e;
  if ((e = orth(Y, d_out, Q)) != cudaSuccess) return e;
  for (int it = 0; it < c.power_iters; ++it) {
    if ((e = rtmul(Q, Z)) != cudaSuccess) return e;
    if ((e = orth(Z, d_in, Zq)) != cudaSuccess) return e;
    if ((e = rmul(Zq, (size_t)d_in * kCL, Y)) != cudaSuccess) return e;
    if ((e = orth(Y, d_out, Q)) != cudaSuccess) return e;
  }
  // a second orthonormalisation pass (the first leaves errors of the Gram's conditioning)
  if ((e = orth(Q, d_out, Y)) != cudaSuccess) return e;
  if ((e = rtmul(Y, Z)) != cudaSuccess) return e;           // Z = R^T Q
  if ((e = gram_of(Z, d_in)) != cudaSuccess) return e;
  if ((e = eig(1)) != cudaSuccess) return e;
  if ((e = apply(Y, d_out, 0, r, 1, Bt)) != cudaSuccess) return e;    // B^T = (Q P_B)^T
  if ((e = apply(Z, d_in, 32, r, 1, At)) != cudaSuccess) return e;    // A^T = (Z P_A)^T
  // 3. INT4 codes
  if ((e = launch_quant_int4(At, (size_t)E * r, d_in, Aq, As, st)) != cudaSuccess) return e;
  if ((e = launch_quant_int4(Bt, (size_t)E * r, d_out, Bq, Bs, st)) != cudaSuccess) return e;
  // 4. reconstruction error
  if (err) {
    if ((e = cudaMemsetAsync(acc, 0, (size_t)E * 2 * 8, st)) != cudaSuccess) return e;
    const int ctiles = d_in / kErrCols;
    int splits = (148 * 4 + ctiles * E - 1) / (ctiles * E);
    if (splits > d_out / 8) splits = d_out / 8;
    if (splits < 1) splits = 1;
    launch_pdl(cmp_err_kernel, dim3(ctiles, E, splits), dim3(256), 0, st, Wb,
               (const __nv_bfloat16*)base, tab, d_out, d_in, r, (const uint8_t*)Aq, (const __half*)As,
               (const uint8_t*)Bq, (const __half*)Bs, acc);
    prof_mark("cmp_err", st);
    launch_pdl(cmp_err_final_kernel, dim3((E + 127) / 128), dim3(128), 0, st, (const double*)acc, E, err);
    prof_mark("cmp_err_final", st);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
