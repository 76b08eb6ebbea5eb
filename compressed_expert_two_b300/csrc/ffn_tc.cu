// Expert computation on the tcgen05 tensor cores (BF16 layers, INT4 group-64 residual).
//
// "Breaking the MoE LLM Trilemma: Dynamic Expert Clustering with Structured Compression"
// (paper notes), key design 2: W~_i = W_base^g + B_i A_i^T and W~_i x = W_base^g x + B_i (A_i^T x),
// the base product computed once for all of a group's experts on the same tokens.  Key design 4:
// BF16/FP16 base, INT4 residual.  Expert body: SwiGLU ("混合专家模型的路由机制与工程落地" 1.2).
//
// Rows are (token, group) pairs in (group, token) order; each row carries k_e experts.
//   1. resid_prep   stacks of the group's K experts, KRP = K*r padded to 64: A_gate^T/A_up^T
//                   as hi+lo BF16 pairs holding the dequantised values exactly (Ain
//                   [G][2][2*KRP][d]); B_gate/B_up dequantised to FP16 (Bgs/Bus [G][f][KRP],
//                   relative rounding <= 2^-11); A_down^T as its integer codes (Adn [G][KRP][f];
//                   the FP16 scale, constant over a 64-column tile, is applied to the product);
//                   B_down as a hi|lo BF16 pair along K (Bdn [G][d][2*KRP]).
//   2. gather_rows  X[i] = x[token(i)] (BF16 rows in (group, token) order).
//   3. U GEMM       U[i] = X[i] (Ain_hi + Ain_lo)_g^T, FP32 accumulation, stored as FP16:
//                   A^T x for every expert of the group.
//   4. ffn_up       per 128-row x 64-column tile of group g: base [Hg|Hu] = X [Wg|Wu]^T once;
//                   per expert slot s: R_s = U~_s [Bgs|Bus]^T (FP16 MMA; U~_s = the row's slot-s
//                   block of U, other blocks zero), h_s = silu(Hg + R_gate) *
//                   (Hu + R_up), hsum += gate_s h_s, and v_s += A_down,e_s^T h_s via
//                   V = h_s Adn_g^T times the tile's A_down scales (tcgen05).
//   5. v_reduce     sums the v partials of the column chunks into V~ [R][2*KRP] (gate-scaled,
//                   block of each slot's expert, repeated for the hi and lo halves of Bdn).
//   6. down GEMM    Y[i] = [hsum | V~][i] [Wd_g | Bdn_g]^T, written to the row's token slot.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "u_dev.cuh"

namespace moe {

namespace {

constexpr int kTile = 128;      // rows per tile (MMA M)
constexpr int kUSimtMaxRows = 1024;   // up to this many rows U is computed on the CUDA cores
constexpr int kNf = 64;         // d_ff columns per gate/up tile

// Tile index -> (group, first row, end of the group's rows); false if the index is unused.
__device__ __forceinline__ bool tile_of(const int32_t* row_begin, int G, int tile, int& g, int& r0, int& r1) {
  for (int gg = 0; gg < G; ++gg) {
    const int b = row_begin[gg], e = row_begin[gg + 1];
    const int nt = (e - b + kTile - 1) / kTile;
    if (tile < nt) {
      g = gg;
      r0 = b + tile * kTile;
      r1 = e;
      return true;
    }
    tile -= nt;
  }
  return false;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return (uint8_t*)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}


}  // namespace

// ------------------------------------------------------------------------------------------
// 1. INT4 -> BF16 residual stacks
// ------------------------------------------------------------------------------------------

// Eight consecutive elements c8..c8+7 of rank row k of expert e: their codes (u - 8) and the
// FP16 scale of their 64-element group (INT4 group-64 format, high nibble first).
__device__ __forceinline__ void codes8(const ResidView& v, int e, int k, int c8, float (&q)[8], float& sc) {
  const size_t row = (size_t)e * v.r + k;
  const uint32_t w = *reinterpret_cast<const uint32_t*>((const uint8_t*)v.vals + row * (v.n / 2) + c8 / 2);
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t byte = (w >> (8 * b)) & 0xFFu;
    q[2 * b] = (float)((int)(byte >> 4) - 8);
    q[2 * b + 1] = (float)((int)(byte & 0xFu) - 8);
  }
  sc = __half2float(v.scales[row * (v.n / kQGroup) + c8 / kQGroup]);
}

// Row-major stacks (Ain hi/lo, Adn): 8 consecutive elements per work item, grid-stride.
__global__ void resid_prep_rows_kernel(PrepArgs p, GroupTable tab) {
  pdl_wait();
  pdl_trigger();
  const int G = p.G, K = p.K, r = p.r, KRP = p.KRP, d = p.d, f = p.f;
  const size_t nAin = p.need_ain ? (size_t)G * 2 * KRP * (d / 8) : 0;   // hi/lo pairs written together
  const size_t nAdn = (size_t)G * KRP * (f / 8);
  for (size_t w = blockIdx.x * (size_t)blockDim.x + threadIdx.x; w < nAin + nAdn; w += (size_t)gridDim.x * blockDim.x) {
    if (w < nAin) {
      // Ain[g][0][m*KRP + j*r + k][c] = hi, Ain[g][1][...] = lo of A_m,e_j^T[k][c]
      const int c8 = (int)(w % (d / 8)) * 8;
      const size_t rowg = w / (d / 8);
      const int g = (int)(rowg / (2 * KRP)), row = (int)(rowg % (2 * KRP));
      const int m = row / KRP, jk = row % KRP, j = jk / r, k = jk % r;
      uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
      if (j < K) {
        const int e = tab.member[g * K + j];
        float cq[8], sc;
        codes8(p.A[m], e, k, c8, cq, sc);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float v0 = cq[2 * q] * sc, v1 = cq[2 * q + 1] * sc;
          const __nv_bfloat16 h0 = __float2bfloat16_rn(v0), h1 = __float2bfloat16_rn(v1);
          hi[q] = tc::pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
          lo[q] = tc::pack_bf16(v0 - __bfloat162float(h0), v1 - __bfloat162float(h1));
        }
      }
      __nv_bfloat16* dst = p.Ain + ((size_t)g * 2 * (2 * KRP) + row) * d + c8;
      *reinterpret_cast<uint4*>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(dst + (size_t)2 * KRP * d) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    } else {
      // Adn[g][j*r + k][c] = code of A_down,e_j^T[k][c]
      const size_t idx = w - nAin;
      const int c8 = (int)(idx % (f / 8)) * 8;
      const size_t rowg = idx / (f / 8);
      const int g = (int)(rowg / KRP), jk = (int)(rowg % KRP), j = jk / r, k = jk % r;
      uint32_t out[4] = {0u, 0u, 0u, 0u};
      if (j < K) {
        const int e = tab.member[g * K + j];
        float cq[8], sc;
        codes8(p.A[2], e, k, c8, cq, sc);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (p.adn_f16) {
            __half2 h2 = __floats2half2_rn(cq[2 * q] * sc, cq[2 * q + 1] * sc);
            out[q] = *reinterpret_cast<uint32_t*>(&h2);
          } else {
            out[q] = tc::pack_bf16(cq[2 * q], cq[2 * q + 1]);
          }
        }
      }
      *reinterpret_cast<uint4*>(p.Adn + rowg * f + c8) = make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
}

// Transposed stacks: block (m, g, 64-column chunk) reads the KRP rank rows of the chunk
// (coalesced), transposes through shared memory and writes 64 rows of KRP (or 2*KRP) values.
//   m = 0, 1: Bgs/Bus[g][n][j*r + k] = fp16(dequantised B_m,e_j^T[k][n])
//   m = 2:    Bdn[g][n][j*r + k] = hi, Bdn[g][n][KRP + j*r + k] = lo of B_down,e_j^T[k][n]
//   m = 3:    Adt[g][n][j*r + k] = fp16(dequantised A_down,e_j^T[k][n]) (when Adt is set)
__global__ void __launch_bounds__(256) resid_prep_t_kernel(PrepArgs p, GroupTable tab) {
  pdl_wait();
  pdl_trigger();
  constexpr int CW = 64;                   // columns per block
  __shared__ float tile[CW][128 + 1];      // [column][jk], KRP <= 128
  const int G = p.G, K = p.K, r = p.r, KRP = p.KRP, d = p.d, f = p.f;
  const int nf = f / CW, nd = d / CW;
  int blk = blockIdx.x, m;
  if (blk < G * nf) m = 0;
  else if ((blk -= G * nf) < G * nf) m = 1;
  else if ((blk -= G * nf) < G * nd) m = 2;
  else { blk -= G * nd; m = 3; }
  const int n = m == 2 ? d : f, nchunk = m == 2 ? nd : nf;
  const int g = blk / nchunk, c0 = (blk % nchunk) * CW;
  const ResidView& v = m == 3 ? p.A[2] : p.B[m];
  // load: a work item is 8 consecutive columns (4 bytes of codes) of one rank row
  for (int it = threadIdx.x; it < KRP * (CW / 8); it += blockDim.x) {
    const int jk = it / (CW / 8), c8 = (it % (CW / 8)) * 8, j = jk / r, k = jk % r;
    float vals[8];
    if (j < K) {
      const int e = tab.member[g * K + j];
      const size_t rowi = (size_t)e * r + k;
      const uint32_t bytes = *reinterpret_cast<const uint32_t*>((const uint8_t*)v.vals + rowi * (n / 2) + (c0 + c8) / 2);
      const float sc = __half2float(v.scales[rowi * (n / 64) + (c0 + c8) / 64]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t b8 = (bytes >> (8 * q)) & 0xFFu;
        vals[2 * q] = (float)((int)(b8 >> 4) - 8) * sc;
        vals[2 * q + 1] = (float)((int)(b8 & 0xF) - 8) * sc;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) vals[q] = 0.f;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) tile[c8 + q][jk] = vals[q];
  }
  __syncthreads();
  const int width = m == 2 ? 2 * KRP : KRP;
  void* base = m == 0 ? (void*)p.Bgs : m == 1 ? (void*)p.Bus : m == 2 ? (void*)p.Bdn : (void*)p.Adt;
  for (int it = threadIdx.x; it < CW * (KRP / 8); it += blockDim.x) {
    const int c = it / (KRP / 8), jk0 = (it % (KRP / 8)) * 8;
    uint16_t* dst = (uint16_t*)base + ((size_t)g * n + c0 + c) * width + jk0;
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float a0 = tile[c][jk0 + 2 * q], a1 = tile[c][jk0 + 2 * q + 1];
      if (m == 2) {
        const float h0 = __bfloat162float(__float2bfloat16_rn(a0)), h1 = __bfloat162float(__float2bfloat16_rn(a1));
        hi[q] = tc::pack_bf16(h0, h1);
        lo[q] = tc::pack_bf16(a0 - h0, a1 - h1);
      } else {
        __half2 h2 = __floats2half2_rn(a0, a1);
        hi[q] = *reinterpret_cast<uint32_t*>(&h2);
        lo[q] = 0u;
      }
    }
    *reinterpret_cast<uint4*>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    if (m == 2) *reinterpret_cast<uint4*>(dst + KRP) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// ------------------------------------------------------------------------------------------
// 2. X rows in (group, token) order
// ------------------------------------------------------------------------------------------
// One warp per row (grid-stride over rows): the row's token is looked up once, then each lane
// moves four 16-byte pieces per round with all four loads in flight before the stores.
__global__ void gather_rows_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ row_asg,
                                   int R, int d, int kg, __nv_bfloat16* __restrict__ X) {
  pdl_wait();
  pdl_trigger();
  const int per_row = d / 8;                       // 16-byte pieces per row (d % 128 == 0)
  const int lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < R; i += nw) {
    const int t = row_asg[i] / kg;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    uint4* dst = reinterpret_cast<uint4*>(X + (size_t)i * d);
    for (int c = lane; c < per_row; c += 128) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c + 32 * u < per_row) v[u] = src[c + 32 * u];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c + 32 * u < per_row) dst[c + 32 * u] = v[u];
    }
  }
}

__global__ void __launch_bounds__(256, 2) u_simt_kernel(const __nv_bfloat16* __restrict__ x,
                                                     const int32_t* __restrict__ row_asg,
                                                     const int32_t* __restrict__ eidx, PrepArgs p, GroupTable tab,
                                                     int kg, int ke, __half* __restrict__ U,
                                                     __nv_bfloat16* __restrict__ X) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) __nv_bfloat16 xs[];      // the row's x (d values)
  u_simt_item(x, row_asg, eidx, p, tab, kg, ke, U, X, blockIdx.x, blockIdx.y, blockIdx.z, xs);
}

// ------------------------------------------------------------------------------------------
// 3/6. Generic grouped GEMM: out[row] = [A0 | A1][i] [B0_g | B1_g]^T (BF16 in, FP32 acc, BF16,
//      FP32 or FP16 out).  Group g's B rows start at g*b_stride in B0 and at g*b_stride + b1_off in B1.
enum OutKind { kOutBf16 = 0, kOutF32 = 1, kOutF16 = 2 };
// Slot of group g's rows in B0 (g itself unless B0 is a cache of offloaded group bases).
struct SlotMap {
  uint8_t s[kMaxE];
};
static SlotMap identity_slots() {
  SlotMap m;
  for (int i = 0; i < kMaxE; ++i) m.s[i] = (uint8_t)i;
  return m;
}
// ------------------------------------------------------------------------------------------
template <int BN, int STAGES, int OUT>
__global__ void __launch_bounds__(192, 1) tc_gemm_kernel(
    const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
    const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1, int nk0, int nk1,
    const int32_t* __restrict__ row_begin, int G, int b_stride, int b1_off, void* __restrict__ out, int out_ld,
    const int32_t* __restrict__ scatter, DevStatus* status, SlotMap b0s) {
  pdl_wait();
  pdl_trigger();
  constexpr uint32_t A_BYTES = kTile * 128, B_BYTES = BN * 128;
  constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[STAGES], empty[STAGES], acc_full, fin;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  int g, r0, r1;
  if (!tile_of(row_begin, G, blockIdx.y, g, r0, r1)) return;
  const int n0 = blockIdx.x * BN;
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tc::Abort ab{&abort_flag, status};

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { tc::bar_init(&full[s], 1); tc::bar_init(&empty[s], 1); }
    tc::bar_init(&acc_full, 1);
    tc::bar_init(&fin, 1);
    abort_flag = 0;
    tc::bar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, TMEM_COLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_base;
  const int nk = nk0 + nk1;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    tc::prefetch_map(&mA0); tc::prefetch_map(&mB0);
    if (nk1) { tc::prefetch_map(&mA1); tc::prefetch_map(&mB1); }
    int kb = 0;
    for (; kb < nk; ++kb) {
      const int s = kb % STAGES, it = kb / STAGES;
      if (kb >= STAGES && !tc::bar_wait(&empty[s], (it - 1) & 1, ab, 1)) break;
      tc::bar_expect_tx(&full[s], A_BYTES + B_BYTES);
      const bool first = kb < nk0;
      const int kx = (first ? kb : kb - nk0) * 64;
      tc::tma_load_2d(sA + s * A_BYTES, first ? &mA0 : &mA1, &full[s], kx, r0);
      tc::tma_load_2d(sB + s * B_BYTES, first ? &mB0 : &mB1, &full[s], kx,
                      (first ? (int)b0s.s[g] : g) * b_stride + (first ? 0 : b1_off) + n0);
    }
    if (abort_flag) tc::drain_copies();
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc = tc::idesc_bf16(kTile, BN);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % STAGES, it = kb / STAGES;
      if (!tc::bar_wait(&full[s], it & 1, ab, 2)) break;
      tc::fence_after();
      const uint32_t a0 = tc::smem_u32(sA + s * A_BYTES), b0 = tc::smem_u32(sB + s * B_BYTES);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc::mma_bf16(tmem, tc::sdesc(a0 + 32 * k), tc::sdesc(b0 + 32 * k), idesc, (kb | k) != 0);
      tc::mma_commit(&empty[s]);
    }
    tc::mma_commit(&acc_full);
    tc::mma_commit(&fin);
    const uint64_t t0 = tc::now_ns();
    while (!tc::bar_test(&fin, 0) && tc::now_ns() - t0 < tc::kWaitNs) {}
  } else if (warp >= 2) {
    // ---------------- epilogue: TMEM -> BF16 rows
    const int q = warp & 3, row = q * 32 + lane, i = r0 + row;
    if (tc::bar_wait(&acc_full, 0, ab, 3) && !abort_flag) {
      tc::fence_after();
      const bool valid = i < r1;
      const size_t orow = valid ? (size_t)(scatter ? scatter[i] : i) : 0;
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        uint32_t v[16];
        tc::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c, v);
        tc::tmem_ld_wait();
        if (valid) {
          if constexpr (OUT == kOutF32) {
            uint4* d4 = reinterpret_cast<uint4*>((float*)out + orow * out_ld + n0 + c);
#pragma unroll
            for (int e = 0; e < 4; ++e) d4[e] = make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
          } else if constexpr (OUT == kOutF16) {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              __half2 h2 = __floats2half2_rn(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
              pk[e] = *reinterpret_cast<uint32_t*>(&h2);
            }
            uint4* d4 = reinterpret_cast<uint4*>((__half*)out + orow * out_ld + n0 + c);
            d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          } else {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[e] = tc::pack_bf16(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
            uint4* d4 = reinterpret_cast<uint4*>((__nv_bfloat16*)out + orow * out_ld + n0 + c);
            d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------------------
// 3/6 (persistent).  The same grouped GEMM for grids of many waves: one CTA per SM walks the work
// items w = blockIdx.x + k * gridDim.x (item = row tile * n_tiles + N tile; unused row tiles are
// skipped by every role alike), the stage ring runs on across items, and TMEM holds two
// accumulators (2 x BN columns) so that the epilogue of one item overlaps the K loop of the next.
// ------------------------------------------------------------------------------------------
template <int BN, int STAGES, int OUT>
__global__ void __launch_bounds__(192, 1) tc_gemm_persist_kernel(
    const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
    const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1, int nk0, int nk1,
    const int32_t* __restrict__ row_begin, int G, int b_stride, int b1_off, int tiles, int n_tiles,
    void* __restrict__ out, int out_ld, const int32_t* __restrict__ scatter, DevStatus* status, SlotMap b0s) {
  pdl_wait();
  pdl_trigger();
  constexpr uint32_t A_BYTES = kTile * 128, B_BYTES = BN * 128;
  static_assert(2 * BN <= 512, "two accumulators in TMEM");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], fin;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tc::Abort ab{&abort_flag, status};
  const int items = tiles * n_tiles;
  const int nk = nk0 + nk1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { tc::bar_init(&full[s], 1); tc::bar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { tc::bar_init(&acc_full[b], 1); tc::bar_init(&acc_empty[b], 4); }
    tc::bar_init(&fin, 1);
    abort_flag = 0;
    tc::bar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, 2 * BN);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer: the stage ring runs on across items
    tc::prefetch_map(&mA0); tc::prefetch_map(&mB0);
    if (nk1) { tc::prefetch_map(&mA1); tc::prefetch_map(&mB1); }
    int kc = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < items && ok; w += gridDim.x) {
      int g, r0, r1;
      if (!tile_of(row_begin, G, w / n_tiles, g, r0, r1)) continue;
      const int n0 = (w % n_tiles) * BN;
      for (int kb = 0; kb < nk; ++kb, ++kc) {
        const int s = kc % STAGES, it = kc / STAGES;
        if (kc >= STAGES && !tc::bar_wait(&empty[s], (it - 1) & 1, ab, 151)) { ok = false; break; }
        tc::bar_expect_tx(&full[s], A_BYTES + B_BYTES);
        const bool first = kb < nk0;
        const int kx = (first ? kb : kb - nk0) * 64;
        tc::tma_load_2d(sA + s * A_BYTES, first ? &mA0 : &mA1, &full[s], kx, r0);
        tc::tma_load_2d(sB + s * B_BYTES, first ? &mB0 : &mB1, &full[s], kx,
                        (first ? (int)b0s.s[g] : g) * b_stride + (first ? 0 : b1_off) + n0);
      }
    }
    if (abort_flag) tc::drain_copies();
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer: item li into acc[li & 1]
    constexpr uint32_t idesc = tc::idesc_bf16(kTile, BN);
    int kc = 0, li = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < items && ok; w += gridDim.x) {
      int g, r0, r1;
      if (!tile_of(row_begin, G, w / n_tiles, g, r0, r1)) continue;
      const int b = li & 1;
      if (li >= 2 && !tc::bar_wait(&acc_empty[b], ((li >> 1) - 1) & 1, ab, 152)) break;
      tc::fence_after();
      const uint32_t dcol = tmem + b * BN;
      for (int kb = 0; kb < nk; ++kb, ++kc) {
        const int s = kc % STAGES, it = kc / STAGES;
        if (!tc::bar_wait(&full[s], it & 1, ab, 153)) { ok = false; break; }
        tc::fence_after();
        const uint32_t a0 = tc::smem_u32(sA + s * A_BYTES), b0 = tc::smem_u32(sB + s * B_BYTES);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_bf16(dcol, tc::sdesc(a0 + 32 * k), tc::sdesc(b0 + 32 * k), idesc, (kb | k) != 0);
        tc::mma_commit(&empty[s]);
      }
      if (!ok) break;
      tc::mma_commit(&acc_full[b]);
      ++li;
    }
    tc::mma_commit(&fin);
    const uint64_t t0 = tc::now_ns();
    while (!tc::bar_test(&fin, 0) && tc::now_ns() - t0 < tc::kWaitNs) {}
  } else if (warp >= 2) {
    // ---------------- epilogue: TMEM -> rows, item li from acc[li & 1]
    const int q = warp & 3, row = q * 32 + lane;
    int li = 0;
    for (int w = blockIdx.x; w < items; w += gridDim.x) {
      int g, r0, r1;
      if (!tile_of(row_begin, G, w / n_tiles, g, r0, r1)) continue;
      const int b = li & 1, n0 = (w % n_tiles) * BN;
      const bool got = tc::bar_wait(&acc_full[b], (li >> 1) & 1, ab, 154);
      if (!__all_sync(0xffffffffu, got) || abort_flag) break;
      tc::fence_after();
      const int i = r0 + row;
      const bool valid = i < r1;
      const size_t orow = valid ? (size_t)(scatter ? scatter[i] : i) : 0;
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t v[32];
        tc::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + b * BN + c, *reinterpret_cast<uint32_t(*)[16]>(v));
        tc::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + b * BN + c + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
        tc::tmem_ld_wait();
        if (c + 32 >= BN) {
          // this warp has read the whole accumulator: the MMA of item li + 2 may overwrite it
          tc::fence_before();
          __syncwarp();
          if (lane == 0) tc::bar_arrive(&acc_empty[b]);
        }
        if (valid) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint32_t* vv = v + 16 * hh;
            const int cc = c + 16 * hh;
            if constexpr (OUT == kOutF32) {
              uint4* d4 = reinterpret_cast<uint4*>((float*)out + orow * out_ld + n0 + cc);
#pragma unroll
              for (int e = 0; e < 4; ++e) d4[e] = make_uint4(vv[4 * e], vv[4 * e + 1], vv[4 * e + 2], vv[4 * e + 3]);
            } else if constexpr (OUT == kOutF16) {
              uint32_t pk[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                __half2 h2 = __floats2half2_rn(__uint_as_float(vv[2 * e]), __uint_as_float(vv[2 * e + 1]));
                pk[e] = *reinterpret_cast<uint32_t*>(&h2);
              }
              uint4* d4 = reinterpret_cast<uint4*>((__half*)out + orow * out_ld + n0 + cc);
              d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            } else {
              uint32_t pk[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) pk[e] = tc::pack_bf16(__uint_as_float(vv[2 * e]), __uint_as_float(vv[2 * e + 1]));
              uint4* d4 = reinterpret_cast<uint4*>((__nv_bfloat16*)out + orow * out_ld + n0 + cc);
              d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
          }
        }
      }
      ++li;
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 2 * BN);
  }
}

// ------------------------------------------------------------------------------------------
// 3/6 (pairs). The same grouped GEMM on CTA pairs: the two CTAs of a cluster take two 128-row
//      tiles of one group (pair P covers the group's tiles 2P and 2P + 1; the second may lie past
//      the group's end and then only feeds the pair) and one MMA of M = 256 x N = BN, issued by
//      rank 0, reads each CTA's A rows and B half (BN/2 rows) from its own shared memory.  Both
//      CTAs' TMA loads complete on rank 0's stage barrier; rank 0's commits arrive on both CTAs'
//      barriers.  Per SM a K step lands 16 KB of A and BN/2 x 128 B of B.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ bool pair_tile_of(const int32_t* row_begin, int G, int P, int m, int& g, int& r0, int& r1) {
  for (int gg = 0; gg < G; ++gg) {
    const int b = row_begin[gg], e = row_begin[gg + 1];
    const int np = ((e - b + kTile - 1) / kTile + 1) / 2;
    if (P < np) {
      g = gg;
      r0 = b + (2 * P + m) * kTile;
      r1 = e;
      return true;
    }
    P -= np;
  }
  return false;
}

template <int BN, int STAGES, int OUT>
__global__ void __launch_bounds__(192, 1) tc_gemm_pair_kernel(
    const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
    const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1, int nk0, int nk1,
    const int32_t* __restrict__ row_begin, int G, int b_stride, int b1_off, void* __restrict__ out, int out_ld,
    const int32_t* __restrict__ scatter, DevStatus* status, int dense_rows, SlotMap b0s, int band) {
  constexpr int BH = BN / 2;                                  // B rows held by each CTA
  constexpr uint32_t A_BYTES = kTile * 128, B_BYTES = BH * 128, STAGE_BYTES = A_BYTES + B_BYTES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[STAGES], empty[STAGES], acc_full;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  pdl_wait();
  pdl_trigger();

  const uint32_t rank = tc::cluster_rank();
  int g, r0, r1;
  // tile of this cluster: (pair tile P, N tile nt).  With band > 0 the clusters, numbered in
  // launch order, take bands of `band` pair tiles across every N tile, so that the clusters
  // resident at once share a few row slabs of A and N tiles of B in L2 instead of streaming all
  // rows for one N tile at a time
  int P = blockIdx.x >> 1, nt = blockIdx.y;
  if (band > 0) {
    const int np = gridDim.x >> 1, ntn = gridDim.y;
    const int c = blockIdx.y * np + P, per = band * ntn, b = c / per, in = c % per;
    const int rows = min(band, np - b * band);
    P = b * band + in % rows;
    nt = in / rows;
  }
  // dense_rows > 0: rows [0, dense_rows) of A against every group's B (N tile nt = group nt, its
  // BN rows), output columns nt * BN ..; else rows of each group against that group's B
  if (dense_rows > 0) {
    if (P * 2 * kTile >= dense_rows) return;                                      // same for both CTAs
    g = nt;
    r0 = (2 * P + (int)rank) * kTile;
    r1 = dense_rows;
  } else if (!pair_tile_of(row_begin, G, P, (int)rank, g, r0, r1)) {
    return;                                                                        // same for both CTAs
  }
  const int n0 = dense_rows > 0 ? 0 : nt * BN;                 // B rows of the N tile inside group g
  const int oc0 = nt * BN;                                     // output columns
  uint8_t* smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tc::Abort ab{&abort_flag, status};

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { tc::bar_init(&full[s], 1); tc::bar_init(&empty[s], 1); }
    tc::bar_init(&acc_full, 1);
    abort_flag = 0;
    tc::bar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc_pair(&tmem_base, BN);
  tc::fence_before();
  // both CTAs' barriers are initialised before either CTA signals the other's
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  tc::fence_after();
  const uint32_t tmem = tmem_base;
  const int nk = nk0 + nk1;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs): own A rows and own half of B, counted on rank 0
    tc::prefetch_map(&mA0); tc::prefetch_map(&mB0);
    if (nk1) { tc::prefetch_map(&mA1); tc::prefetch_map(&mB1); }
    const uint32_t full0 = tc::map_shared(tc::smem_u32(&full[0]), 0);
    bool ok = true;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % STAGES, it = kb / STAGES;
      if (kb >= STAGES && !tc::bar_wait_cluster(&empty[s], (it - 1) & 1, ab, 41)) { ok = false; break; }
      if (rank == 0) tc::bar_expect_tx(&full[s], 2 * STAGE_BYTES);
      const bool first = kb < nk0;
      const int kx = (first ? kb : kb - nk0) * 64;
      uint8_t* st = smem + s * STAGE_BYTES;
      tc::tma_load_2d_pair(st, first ? &mA0 : &mA1, full0 + 8 * s, kx, r0);
      tc::tma_load_2d_pair(st + A_BYTES, first ? &mB0 : &mB1, full0 + 8 * s, kx,
                           (first ? (int)b0s.s[g] : g) * b_stride + (first ? 0 : b1_off) + n0 + (int)rank * BH);
    }
    // every commit rank 0 sends to this CTA's stage barriers has landed before the CTA exits
    if (ok) {
      for (int s = 0; s < STAGES && s < nk; ++s)
        if (!tc::bar_wait_cluster(&empty[s], ((nk - 1 - s) / STAGES) & 1, ab, 42)) break;
    }
    if (abort_flag) tc::drain_copies();
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer (rank 0)
    constexpr uint32_t idesc = tc::idesc_bf16(2 * kTile, BN);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % STAGES, it = kb / STAGES;
      if (!tc::bar_wait_cluster(&full[s], it & 1, ab, 43)) break;
      tc::fence_after();
      const uint32_t a0 = tc::smem_u32(smem + s * STAGE_BYTES), b0 = a0 + A_BYTES;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc::mma_bf16_pair(tmem, tc::sdesc(a0 + 32 * k), tc::sdesc(b0 + 32 * k), idesc, (kb | k) != 0);
      tc::mma_commit_pair(&empty[s], 3);
    }
    tc::mma_commit_pair(&acc_full, 3);
  } else if (warp >= 2) {
    // ---------------- epilogue (both CTAs): this CTA's 128 rows, all BN columns
    const int q = warp & 3, row = q * 32 + lane, i = r0 + row;
    if (tc::bar_wait_cluster(&acc_full, 0, ab, 44) && !abort_flag) {
      tc::fence_after();
      const bool valid = i < r1;
      const size_t orow = valid ? (size_t)(scatter ? scatter[i] : i) : 0;
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        uint32_t v[16];
        tc::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c, v);
        tc::tmem_ld_wait();
        if (valid) {
          if constexpr (OUT == kOutF32) {
            uint4* d4 = reinterpret_cast<uint4*>((float*)out + orow * out_ld + oc0 + c);
#pragma unroll
            for (int e = 0; e < 4; ++e) d4[e] = make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
          } else if constexpr (OUT == kOutF16) {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              __half2 h2 = __floats2half2_rn(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
              pk[e] = *reinterpret_cast<uint32_t*>(&h2);
            }
            uint4* d4 = reinterpret_cast<uint4*>((__half*)out + orow * out_ld + oc0 + c);
            d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          } else {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[e] = tc::pack_bf16(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
            uint4* d4 = reinterpret_cast<uint4*>((__nv_bfloat16*)out + orow * out_ld + oc0 + c);
            d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc_pair(tmem, BN);
  }
}

// ------------------------------------------------------------------------------------------
// 4. Fused gate/up tile: base once, per-slot residual, SwiGLU, gated sum, down-residual partials
//
// A work item is a 128-row tile of one group and a chunk of 64-column d_ff tiles; one CTA per SM
// walks the items w = blockIdx.x, blockIdx.x + gridDim.x, ... (persistent: the stage ring, the
// double-buffered accumulator and the slot phases run on across items, so the next item's K loop
// overlaps this item's slots, and small items balance the SMs).  Warp roles
// (12 warps): 0 TMA producer of the base stages (X, W_gate, W_up); 1 base MMA issuer (owns TMEM);
// 2 residual/V MMA issuer; 3 TMA producer of the residual tiles (B_gate, B_up, A_down^T codes);
// 4..11 epilogue, two warps per TMEM lane quarter, warp group h in {0,1} handling the tile's d_ff
// columns [32h, 32h+32) (group 0 also builds the gate half of U~ and reads V out, group 1 the up
// half of U~).
//
// TMEM columns: two accumulators acc[b] = [gate 64 | up 64] (double buffered so that the next
// tile's K-loop overlaps this tile's slots) and V (KRP).  The residual is added INTO the
// accumulator: for slot s of a tile the residual MMA adds D_s [B_gate | B_up]^T, where
// D_0 = U~_0 and D_s = U~_s - U~_{s-1}, so that after it acc = base + R_s exactly up to FP32
// rounding (the blocks of U~_s and U~_{s-1} are disjoint: a row's experts are distinct).  The
// epilogue reads acc once per slot (no separate residual buffer), forms h_s = silu(a) * b, adds
// gate_s h_s into the tile's hsum, and stores h_s (BF16) for the V MMA V = h_s A_down^T, which
// runs one slot behind so that it leaves the slot chain.
// ------------------------------------------------------------------------------------------
constexpr int kMaxKe = 4;
constexpr int kRank = 16;      // residual rank handled by this kernel
constexpr int kUpWarps = 12;
constexpr int kUpEpi = 256;    // epilogue threads
constexpr int kUpEpiWarp0 = 4;

struct UpArgs {
  const int32_t* row_begin;
  const int32_t* row_asg;
  const int32_t* eidx;
  const float* gate;
  const __half* U;          // [R][2*KRP] FP16: A_gate^T x | A_up^T x of the group's experts
                            // (u_by_token: [T][G*2*KRP], token t's block of every group)
  int u_by_token;
  const __half* sAd;        // FP16 scales [E][16][f/64] of A_down^T
  __nv_bfloat16* hsum;      // [R][f]
  float* Vpart;             // [nchunks][R][ke][16]
  DevStatus* status;
  GroupTable tab;
  int G, d, f, kg, ke, R, n_ftiles, ftiles_per_chunk;
  int n_row_tiles, n_chunks;   // work items of the 128-column kernel: row tile x chunk
};

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}

template <int KRP, int STAGES, int KE, int RBUF>
__global__ void __launch_bounds__(kUpWarps * 32, 1) ffn_up_tc_kernel(
    const __grid_constant__ CUtensorMap mX, const __grid_constant__ CUtensorMap mWg,
    const __grid_constant__ CUtensorMap mWu, const __grid_constant__ CUtensorMap mBg,
    const __grid_constant__ CUtensorMap mBu, const __grid_constant__ CUtensorMap mAd, const UpArgs p) {
  pdl_wait();
  pdl_trigger();
  constexpr uint32_t X_BYTES = kTile * 128, W_BYTES = 2 * kNf * 128, STAGE_BYTES = X_BYTES + W_BYTES;
  constexpr uint32_t BRES_BYTES = KRP * kNf * 2;          // one of Bg / Bu tiles (64 rows x KRP)
  constexpr uint32_t AD_BYTES = KRP * 128;                 // KRP rows x 64 columns
  constexpr uint32_t RES_BYTES = 2 * BRES_BYTES + AD_BYTES;
  constexpr uint32_t UT_BYTES = kTile * KRP * 2;           // 128 rows x KRP
  constexpr int KATOM = KRP / 64;
  constexpr uint32_t COL_V = 4 * kNf;
  static_assert(COL_V + KRP <= 512, "TMEM budget");
  static_assert(KE >= 1 && KE <= kMaxKe, "slots");

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[STAGES], empty[STAGES];
  __shared__ uint64_t base_full[2], acc_empty[2];
  __shared__ uint64_t rb_full[RBUF], rb_empty[RBUF], ad_full[RBUF], ad_empty[RBUF];
  __shared__ uint64_t acc_full, acc_read, u_ready, h_ready, v_full, v_empty, fin1, fin2;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  // work items w = row tile * n_chunks + chunk, taken w = blockIdx.x, blockIdx.x + gridDim.x, ...
  // (one CTA per item, or one per SM walking several); every role walks the same items and skips
  // the unused ones alike, and the stage ring, accumulator parity and slot phases run on across
  // items (glt: tiles, sig: slots, counted over the CTA's items)
  const int n_items = p.n_row_tiles * p.n_chunks;
  auto item = [&](int w, int& g, int& r0, int& r1, int& ft0, int& nft) -> bool {
    if (!tile_of(p.row_begin, p.G, w / p.n_chunks, g, r0, r1)) return false;
    ft0 = (w % p.n_chunks) * p.ftiles_per_chunk;
    nft = min(ft0 + p.ftiles_per_chunk, p.n_ftiles) - ft0;
    return nft > 0;
  };
  const int nkb = p.d / 64;
  const int f = p.f, fg = f / 64;

  uint8_t* smem = align1024(smem_raw);
  uint8_t* sStage = smem;
  uint8_t* sRes = sStage + STAGES * STAGE_BYTES;     // RBUF x [Bg | Bu | Ad]
  uint8_t* sUg = sRes + RBUF * RES_BYTES;
  uint8_t* sUu = sUg + UT_BYTES;
  uint8_t* sH = sUu + UT_BYTES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tc::Abort ab{&abort_flag, p.status};
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { tc::bar_init(&full[s], 1); tc::bar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { tc::bar_init(&base_full[b], 1); tc::bar_init(&acc_empty[b], kUpEpi); }
    for (int b = 0; b < RBUF; ++b) {
      tc::bar_init(&rb_full[b], 1); tc::bar_init(&rb_empty[b], 1);
      tc::bar_init(&ad_full[b], 1); tc::bar_init(&ad_empty[b], 1);
    }
    tc::bar_init(&acc_full, 1);
    tc::bar_init(&acc_read, kUpEpi);
    tc::bar_init(&u_ready, kUpEpi);
    tc::bar_init(&h_ready, kUpEpi);
    tc::bar_init(&v_full, 1);
    tc::bar_init(&v_empty, kUpEpi);
    tc::bar_init(&fin1, 1);
    tc::bar_init(&fin2, 1);
    abort_flag = 0;
    tc::bar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, 512);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer of the base stages
      tc::prefetch_map(&mX); tc::prefetch_map(&mWg); tc::prefetch_map(&mWu);
      int kc = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      int g, r0, r1, ft0, nft;
      if (!item(w, g, r0, r1, ft0, nft)) continue;
      for (int lt = 0; lt < nft && ok; ++lt) {
        const int n0 = (ft0 + lt) * kNf;
        for (int kb = 0; kb < nkb; ++kb, ++kc) {
          const int s = kc % STAGES, it = kc / STAGES;
          if (kc >= STAGES && !tc::bar_wait(&empty[s], (it - 1) & 1, ab, 11)) { ok = false; break; }
          uint8_t* st = sStage + s * STAGE_BYTES;
          tc::bar_expect_tx(&full[s], STAGE_BYTES);
          tc::tma_load_2d(st, &mX, &full[s], kb * 64, r0);
          tc::tma_load_2d(st + X_BYTES, &mWg, &full[s], kb * 64, (int)p.tab.wslot[g] * f + n0);
          tc::tma_load_2d(st + X_BYTES + kNf * 128, &mWu, &full[s], kb * 64, (int)p.tab.wslot[g] * f + n0);
        }
      }
      }
      if (abort_flag) tc::drain_copies();
    }
  } else if (warp == 3) {
    if (lane == 0) {
      // ---------------- TMA producer of the residual tiles (one set per d_ff tile)
      tc::prefetch_map(&mBg); tc::prefetch_map(&mBu); tc::prefetch_map(&mAd);
      int glt = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      int g, r0, r1, ft0, nft;
      if (!item(w, g, r0, r1, ft0, nft)) continue;
      for (int lt = 0; lt < nft; ++lt, ++glt) {
        const int n0 = (ft0 + lt) * kNf, rb = glt % RBUF, use = glt / RBUF;
        uint8_t* sr = sRes + rb * RES_BYTES;
        if (use > 0 && !tc::bar_wait(&rb_empty[rb], (use - 1) & 1, ab, 13)) { ok = false; break; }
        tc::bar_expect_tx(&rb_full[rb], 2 * BRES_BYTES);
#pragma unroll
        for (int a = 0; a < KATOM; ++a) {
          tc::tma_load_2d(sr + a * kNf * 128, &mBg, &rb_full[rb], a * 64, g * f + n0);
          tc::tma_load_2d(sr + BRES_BYTES + a * kNf * 128, &mBu, &rb_full[rb], a * 64, g * f + n0);
        }
        if (use > 0 && !tc::bar_wait(&ad_empty[rb], (use - 1) & 1, ab, 14)) { ok = false; break; }
        tc::bar_expect_tx(&ad_full[rb], AD_BYTES);
        tc::tma_load_2d(sr + 2 * BRES_BYTES, &mAd, &ad_full[rb], n0, g * KRP);
      }
      }
      if (abort_flag) tc::drain_copies();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- base MMA issuer: [Hg | Hu] = X [Wg | Wu]^T into acc[lt & 1]
      constexpr uint32_t id_base = tc::idesc_bf16(kTile, 2 * kNf);
      int kc = 0, glt = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      int g, r0, r1, ft0, nft;
      if (!item(w, g, r0, r1, ft0, nft)) continue;
      for (int lt = 0; lt < nft && ok; ++lt, ++glt) {
        const int b = glt & 1;
        if (glt >= 2 && !tc::bar_wait(&acc_empty[b], ((glt >> 1) - 1) & 1, ab, 21)) { ok = false; break; }
        tc::fence_after();
        const uint32_t dcol = tmem + b * 2 * kNf;
        for (int kb = 0; kb < nkb; ++kb, ++kc) {
          const int s = kc % STAGES, it = kc / STAGES;
          if (!tc::bar_wait(&full[s], it & 1, ab, 22)) { ok = false; break; }
          tc::fence_after();
          const uint32_t a0 = tc::smem_u32(sStage + s * STAGE_BYTES);
          const uint32_t b0 = a0 + X_BYTES;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_bf16(dcol, tc::sdesc(a0 + 32 * k), tc::sdesc(b0 + 32 * k), id_base, (kb | k) != 0);
          tc::mma_commit(&empty[s]);
        }
        if (!ok) break;
        tc::mma_commit(&base_full[b]);
      }
      }
      tc::mma_commit(&fin1);
      const uint64_t t0 = tc::now_ns();
      while (!tc::bar_test(&fin1, 0) && tc::now_ns() - t0 < tc::kWaitNs) {}
    }
  } else if (warp == 2) {
    if (lane == 0) {
      // ---------------- residual issuer: acc[b] += D_s [Bg | Bu]^T, then (one slot behind)
      //                  V = h_s Adn^T
      constexpr uint32_t id_res = tc::idesc_f16(kTile, kNf);     // FP16 U~ x FP16 B
      constexpr uint32_t id_v = tc::idesc_bf16(kTile, KRP);
      const uint32_t ug = tc::smem_u32(sUg), uu = tc::smem_u32(sUu), hh = tc::smem_u32(sH);
      // V MMA of slot index tau (CTA-wide tile tau / KE, slot tau % KE)
      auto issue_v = [&](int tau) -> bool {
        const int glt = tau / KE, s = tau % KE, rb = glt % RBUF, use = glt / RBUF;
        if (s == 0 && !tc::bar_wait(&ad_full[rb], use & 1, ab, 26)) return false;
        if (!tc::bar_wait(&h_ready, tau & 1, ab, 27)) return false;
        if (tau >= 1 && !tc::bar_wait(&v_empty, (tau - 1) & 1, ab, 28)) return false;
        tc::fence_after();
        const uint32_t ad = tc::smem_u32(sRes + rb * RES_BYTES + 2 * BRES_BYTES);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tmem + COL_V, tc::sdesc(hh + 32 * kk), tc::sdesc(ad + 32 * kk), id_v, kk != 0);
        tc::mma_commit(&v_full);
        if (s == KE - 1) tc::mma_commit(&ad_empty[rb]);
        return true;
      };
      bool ok = true;
      int sig = 0;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      int g, r0, r1, ft0, nft;
      if (!item(w, g, r0, r1, ft0, nft)) continue;
      for (int ls = 0; ls < nft * KE && ok; ++ls, ++sig) {
        const int glt = sig / KE, s = sig % KE, b = glt & 1, rb = glt % RBUF, use = glt / RBUF;
        if (sig >= 1 && !issue_v(sig - 1)) { ok = false; break; }
        if (s == 0) {
          if (!tc::bar_wait(&base_full[b], (glt >> 1) & 1, ab, 23)) { ok = false; break; }
          if (!tc::bar_wait(&rb_full[rb], use & 1, ab, 24)) { ok = false; break; }
        }
        if (!tc::bar_wait(&u_ready, sig & 1, ab, 25)) { ok = false; break; }
        if (s > 0 && !tc::bar_wait(&acc_read, (sig - 1) & 1, ab, 29)) { ok = false; break; }
        tc::fence_after();
        const uint32_t bg = tc::smem_u32(sRes + rb * RES_BYTES), bu = bg + BRES_BYTES;
        const uint32_t dcol = tmem + b * 2 * kNf;
#pragma unroll
        for (int kk = 0; kk < KRP / 16; ++kk) {
          const uint32_t off_u = (kk >> 2) * (kTile * 128) + (kk & 3) * 32;
          const uint32_t off_b = (kk >> 2) * (kNf * 128) + (kk & 3) * 32;
          tc::mma_bf16(dcol, tc::sdesc(ug + off_u), tc::sdesc(bg + off_b), id_res, 1u);
          tc::mma_bf16(dcol + kNf, tc::sdesc(uu + off_u), tc::sdesc(bu + off_b), id_res, 1u);
        }
        tc::mma_commit(&acc_full);
        if (s == KE - 1) tc::mma_commit(&rb_empty[rb]);
      }
      }
      if (ok && sig > 0) issue_v(sig - 1);
      tc::mma_commit(&fin2);
      const uint64_t t0 = tc::now_ns();
      while (!tc::bar_test(&fin2, 0) && tc::now_ns() - t0 < tc::kWaitNs) {}
    }
  } else {
    // ---------------- epilogue: one thread per (tile row, column half)
    const int q = warp & 3, half = (warp - kUpEpiWarp0) >> 2, row = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int c_half = half * 32;                    // this group's first column of the tile
    uint8_t* sU = half == 0 ? sUg : sUu;             // U~ half this group writes
    // this row of this half's U~ starts at zero (later items find the previous item's last delta
    // there, which the first delta of the item clears)
#pragma unroll
    for (int a = 0; a < KATOM; ++a) {
      uint4* z = reinterpret_cast<uint4*>(sU + a * kTile * 128 + (row >> 3) * 1024 + (row & 7) * 128);
#pragma unroll
      for (int c = 0; c < 8; ++c) z[c] = make_uint4(0, 0, 0, 0);
    }
    // U~ holds the last delta: +values in block nz_pos, -values in block nz_neg (or none).
    int nz_pos = -1, nz_neg = -1;
    uint32_t unext[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) unext[c] = 0u;
    __half2 sc_ad[kRank / 2];                        // A_down scales of the slot V is pending for
    bool ok = true;
    int sig = 0, glt = 0;
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
    int g, r0, r1, ft0, nft;
    if (!item(w, g, r0, r1, ft0, nft)) continue;
    const int i = r0 + row, chunk = w % p.n_chunks;
    const bool valid = i < r1;
    int le[KE], eid[KE];
    float gt[KE];
#pragma unroll
    for (int s = 0; s < KE; ++s) { le[s] = 0; eid[s] = 0; gt[s] = 0.f; }
    const __half* urow = p.U;
    if (valid) {
      const int b = p.row_asg[i], t = b / p.kg, j = b % p.kg, k = p.kg * KE;
#pragma unroll
      for (int s = 0; s < KE; ++s) {
        const int e = p.eidx[(size_t)t * k + j * KE + s];
        le[s] = p.tab.local_of[e];
        eid[s] = e;
        gt[s] = p.gate[(size_t)t * k + j * KE + s];
      }
      urow = p.U + (p.u_by_token ? (size_t)t * p.G * 2 * KRP + (size_t)g * 2 * KRP : (size_t)i * 2 * KRP) +
             half * KRP;
    }
    // V accumulators: half h keeps the slots s with s % 2 == h (vacc[s / 2])
    constexpr int KV = (KE + 1) / 2;
    float vacc[KV][kRank];
#pragma unroll
    for (int s = 0; s < KV; ++s)
#pragma unroll
      for (int k = 0; k < kRank; ++k) vacc[s][k] = 0.f;

    // U~ values of slot s for this row (FP16, the same for every d_ff tile)
    auto load_u = [&](int lt, int s, uint32_t (&pk)[8]) {
      (void)lt;
      if (!valid) return;
      const uint4* u4 = reinterpret_cast<const uint4*>(urow + le[s] * kRank);
      const uint4 a = u4[0], b = u4[1];
      pk[0] = a.x; pk[1] = a.y; pk[2] = a.z; pk[3] = a.w;
      pk[4] = b.x; pk[5] = b.y; pk[6] = b.z; pk[7] = b.w;
    };
    auto put_block = [&](int blk, const uint32_t (&pk)[8], uint32_t flip) {
      *reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, blk * kRank, kTile)) =
          make_uint4(pk[0] ^ flip, pk[1] ^ flip, pk[2] ^ flip, pk[3] ^ flip);
      *reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, blk * kRank + 8, kTile)) =
          make_uint4(pk[4] ^ flip, pk[5] ^ flip, pk[6] ^ flip, pk[7] ^ flip);
    };
    auto zero_block = [&](int blk) {
      const uint4 z = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, blk * kRank, kTile)) = z;
      *reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, blk * kRank + 8, kTile)) = z;
    };
    // Writes the delta of slot s (first slot of a tile: no subtraction) from unext.
    auto build_delta = [&](int s) {
      if (!valid) return;
      const int pos = le[s], neg = s > 0 ? le[s - 1] : -1;
      if (neg >= 0) {
        // the previous slot's values are still in block neg (= the last nz_pos): negate in place
        uint4* b0 = reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, neg * kRank, kTile));
        uint4* b1 = reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, neg * kRank + 8, kTile));
        const uint4 v0 = *b0, v1 = *b1;
        constexpr uint32_t F = 0x80008000u;          // exact FP16 negation
        *b0 = make_uint4(v0.x ^ F, v0.y ^ F, v0.z ^ F, v0.w ^ F);
        *b1 = make_uint4(v1.x ^ F, v1.y ^ F, v1.z ^ F, v1.w ^ F);
      }
      if (nz_neg >= 0 && nz_neg != pos && nz_neg != neg) zero_block(nz_neg);
      if (nz_pos >= 0 && nz_pos != pos && nz_pos != neg) zero_block(nz_pos);
      put_block(pos, unext, 0u);
      nz_pos = pos; nz_neg = neg;
    };

    load_u(0, 0, unext);
    build_delta(0);
    tc::fence_async_smem();
    tc::bar_arrive(&u_ready);
    if (KE > 1) load_u(0, KE > 1 ? 1 : 0, unext);
    else if (nft > 1) load_u(1, 0, unext);

    for (int lt = 0; lt < nft && ok; ++lt, ++glt) {
      const int bsel = glt & 1;
      const uint32_t acc_col = bsel * 2 * kNf;
      float hs[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) hs[c] = 0.f;
#pragma unroll
      for (int s = 0; s < KE; ++s, ++sig) {
        // (A) V of the previous slot of this item: wait (this also frees sH), read the row's
        // block, scale (the previous item's last V was read at that item's end)
        if (lt * KE + s >= 1) {
          if (!tc::bar_wait(&v_full, (sig - 1) & 1, ab, 30)) { ok = false; break; }
          tc::fence_after();
          const int ps = s > 0 ? s - 1 : KE - 1;
          if (half == (ps & 1)) {
#pragma unroll 1
            for (int jb = 0; jb < KRP / 16; ++jb) {
              uint32_t vv[16];
              tc::tmem_ld16(tmem + lane_off + COL_V + jb * 16, vv);
              tc::tmem_ld_wait();
              if (valid && jb == le[ps]) {
#pragma unroll
                for (int k = 0; k < kRank; k += 2) {
                  const float2 sf = __half22float2(sc_ad[k / 2]);
                  vacc[ps / 2][k] += __uint_as_float(vv[k]) * sf.x;
                  vacc[ps / 2][k + 1] += __uint_as_float(vv[k + 1]) * sf.y;
                }
              }
            }
          }
          tc::fence_before();
          tc::bar_arrive(&v_empty);
        }
        // (B) acc = base + R_s
        if (!tc::bar_wait(&acc_full, sig & 1, ab, 31)) { ok = false; break; }
        tc::fence_after();
        // (C) h_s = silu(a) * b for this half's 32 columns; hsum; h_s -> sH
#pragma unroll
        for (int c = 0; c < 32; c += 8) {
          uint32_t av[8], bv[8];
          tmem_ld8(tmem + lane_off + acc_col + c_half + c, av);
          tmem_ld8(tmem + lane_off + acc_col + kNf + c_half + c, bv);
          tc::tmem_ld_wait();
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            float h2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              h2[u] = silu_fast(__uint_as_float(av[e + u])) * __uint_as_float(bv[e + u]);
              hs[c + e + u] += gt[s] * h2[u];
            }
            pk[e / 2] = tc::pack_bf16(h2[0], h2[1]);
          }
          *reinterpret_cast<uint4*>(sH + tc::sw128_offset(row, c_half + c, kTile)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        // (D) acc read
        tc::fence_before();
        tc::bar_arrive(&acc_read);
        if (s == KE - 1) tc::bar_arrive(&acc_empty[bsel]);
        // (E) h_s ready for the V MMA
        tc::fence_async_smem();
        tc::bar_arrive(&h_ready);
        if (half == (s & 1) && valid) {
          const __half* sc = p.sAd + (size_t)eid[s] * kRank * fg + ft0 + lt;
#pragma unroll
          for (int k = 0; k < kRank; k += 2) sc_ad[k / 2] = __halves2half2(sc[(size_t)k * fg], sc[(size_t)(k + 1) * fg]);
        }
        // (F) delta for the next slot (U~ is free: the residual MMA of this slot has completed)
        const bool more = s + 1 < KE || lt + 1 < nft;
        if (more) {
          build_delta(s + 1 < KE ? s + 1 : 0);
          tc::fence_async_smem();
          tc::bar_arrive(&u_ready);
          // prefetch the slot after that
          const int s2 = (s + 2) % KE;
          const int lt2 = lt + (s + 2) / KE;
          if (lt2 < nft) load_u(lt2, s2, unext);
        }
      }
      if (!ok) break;
      // (G) hsum of this tile
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(p.hsum + (size_t)i * f + (ft0 + lt) * kNf + c_half);
#pragma unroll
        for (int c = 0; c < 32; c += 8)
          dst[c / 8] = make_uint4(tc::pack_bf16(hs[c], hs[c + 1]), tc::pack_bf16(hs[c + 2], hs[c + 3]),
                                  tc::pack_bf16(hs[c + 4], hs[c + 5]), tc::pack_bf16(hs[c + 6], hs[c + 7]));
      }
    }
    if (!ok) break;
    // V of the item's last slot; then V is free for the next item's first V MMA
    {
      if (!tc::bar_wait(&v_full, (sig - 1) & 1, ab, 33)) ok = false;
      tc::fence_after();
      constexpr int ps = KE - 1;
      if (ok && half == (ps & 1)) {
#pragma unroll 1
        for (int jb = 0; jb < KRP / 16; ++jb) {
          uint32_t vv[16];
          tc::tmem_ld16(tmem + lane_off + COL_V + jb * 16, vv);
          tc::tmem_ld_wait();
          if (valid && jb == le[ps]) {
#pragma unroll
            for (int k = 0; k < kRank; k += 2) {
              const float2 sf = __half22float2(sc_ad[k / 2]);
              vacc[ps / 2][k] += __uint_as_float(vv[k]) * sf.x;
              vacc[ps / 2][k + 1] += __uint_as_float(vv[k + 1]) * sf.y;
            }
          }
        }
      }
    }
    tc::fence_before();
    tc::bar_arrive(&v_empty);
    if (ok && valid) {
      float* vp = p.Vpart + ((size_t)chunk * p.R + i) * KE * kRank;
#pragma unroll
      for (int s = 0; s < KE; ++s)
        if (half == (s & 1)) {
#pragma unroll
          for (int k = 0; k < kRank; k += 4)
            *reinterpret_cast<float4*>(vp + s * kRank + k) =
                make_float4(gt[s] * vacc[s / 2][k], gt[s] * vacc[s / 2][k + 1], gt[s] * vacc[s / 2][k + 2],
                            gt[s] * vacc[s / 2][k + 3]);
        }
    }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------------
// 4b. Fused gate/up on 256-column MMAs (one CTA per 128-row tile and chunk of 128-column d_ff
//     tiles; for K r = 64 (KRP = 64) and at most two expert slots per row).
//
// The accumulator acc = [gate 128 | up 128] of one d_ff tile fills half of TMEM; V_s (the
// A_down^T h_s of slot s, all K experts' blocks) has KRP columns per slot and accumulates over
// every tile of the chunk; h_s goes to TMEM as FP16 (two per column, 64 columns, double
// buffered) where the V MMA reads it as its A operand, with B = A_down^T dequantised to FP16,
// so no scale is applied afterwards.  acc is single-buffered: the next tile's K loop starts when
// the epilogue has read acc for the tile's last slot.  Residual deltas as in 4: acc += D_s
// [B_gate | B_up]^T with D_0 = U~_0, D_s = U~_s - U~_{s-1}.
// ------------------------------------------------------------------------------------------
constexpr int kNf3 = 128;                 // d_ff columns per tile
constexpr int kStages3 = 3;
constexpr int kUp3EpiWarps = 16;          // four warps per TMEM lane quarter, 32 d_ff columns each
constexpr int kUp3Warps = kUpEpiWarp0 + kUp3EpiWarps;

template <int KE>
__global__ void __launch_bounds__(kUp3Warps * 32, 1) ffn_up3_kernel(
    const __grid_constant__ CUtensorMap mX, const __grid_constant__ CUtensorMap mWg,
    const __grid_constant__ CUtensorMap mWu, const __grid_constant__ CUtensorMap mBg,
    const __grid_constant__ CUtensorMap mBu, const __grid_constant__ CUtensorMap mAd, const UpArgs p) {
  pdl_wait();
  pdl_trigger();
  constexpr int KRP = 64, NF = kNf3, STAGES = kStages3;
  constexpr uint32_t X_BYTES = kTile * 128, W_BYTES = 2 * NF * 128, STAGE_BYTES = X_BYTES + W_BYTES;
  constexpr uint32_t BRES_BYTES = NF * KRP * 2;            // B_gate or B_up tile: 128 rows x KRP
  constexpr uint32_t AD_BYTES = KRP * NF * 2;              // A_down^T tile: KRP rows x 128 (two 64-column atoms)
  constexpr uint32_t UT_BYTES = kTile * KRP * 2;
  constexpr uint32_t COL_V = 2 * NF;                       // V_s at COL_V + s * KRP
  constexpr uint32_t COL_H = COL_V + KE * KRP;             // h buffers at COL_H + 64 b
  static_assert(KE >= 1 && KE <= 2 && COL_H + 128 <= 512, "TMEM budget");

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[STAGES], empty[STAGES];
  __shared__ uint64_t acc_empty, rb_full, rb_empty, ad_full, ad_empty;
  __shared__ uint64_t acc_full, acc_read, u_ready, h_ready[2], v_done[2], fin1, fin2;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  int g, r0, r1;
  if (!tile_of(p.row_begin, p.G, blockIdx.y, g, r0, r1)) return;
  const int chunk = blockIdx.x;
  const int ft0 = chunk * p.ftiles_per_chunk;
  const int ft1 = min(ft0 + p.ftiles_per_chunk, p.n_ftiles);
  if (ft0 >= ft1) return;
  const int nft = ft1 - ft0;
  const int nkb = p.d / 64;
  const int f = p.f;

  uint8_t* smem = align1024(smem_raw);
  uint8_t* sStage = smem;
  uint8_t* sBg = sStage + STAGES * STAGE_BYTES;
  uint8_t* sBu = sBg + BRES_BYTES;
  uint8_t* sAd = sBu + BRES_BYTES;
  uint8_t* sUg = sAd + AD_BYTES;
  uint8_t* sUu = sUg + UT_BYTES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tc::Abort ab{&abort_flag, p.status};
  constexpr int kEpiArrive = kUp3EpiWarps;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { tc::bar_init(&full[s], 1); tc::bar_init(&empty[s], 1); }
    tc::bar_init(&acc_empty, kEpiArrive);
    tc::bar_init(&rb_full, 1); tc::bar_init(&rb_empty, 1); tc::bar_init(&ad_full, 1); tc::bar_init(&ad_empty, 1);
    tc::bar_init(&acc_full, 1);
    tc::bar_init(&acc_read, kEpiArrive);
    tc::bar_init(&u_ready, kEpiArrive);
    tc::bar_init(&h_ready[0], kEpiArrive); tc::bar_init(&h_ready[1], kEpiArrive);
    tc::bar_init(&v_done[0], 1); tc::bar_init(&v_done[1], 1);
    tc::bar_init(&fin1, 1); tc::bar_init(&fin2, 1);
    abort_flag = 0;
    tc::bar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, 512);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_base;
  auto warp_arrive = [&](uint64_t* b) {
    __syncwarp();
    if (lane == 0) tc::bar_arrive(b);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer of the base stages (X, W_gate, W_up of one 128-column tile)
      tc::prefetch_map(&mX); tc::prefetch_map(&mWg); tc::prefetch_map(&mWu);
      int kc = 0;
      bool ok = true;
      for (int lt = 0; lt < nft && ok; ++lt) {
        const int n0 = (ft0 + lt) * NF;
        for (int kb = 0; kb < nkb; ++kb, ++kc) {
          const int s = kc % STAGES, it = kc / STAGES;
          if (kc >= STAGES && !tc::bar_wait(&empty[s], (it - 1) & 1, ab, 51)) { ok = false; break; }
          uint8_t* st = sStage + s * STAGE_BYTES;
          tc::bar_expect_tx(&full[s], STAGE_BYTES);
          tc::tma_load_2d(st, &mX, &full[s], kb * 64, r0);
          tc::tma_load_2d(st + X_BYTES, &mWg, &full[s], kb * 64, (int)p.tab.wslot[g] * f + n0);
          tc::tma_load_2d(st + X_BYTES + NF * 128, &mWu, &full[s], kb * 64, (int)p.tab.wslot[g] * f + n0);
        }
      }
      if (abort_flag) tc::drain_copies();
    }
  } else if (warp == 3) {
    if (lane == 0) {
      // ---------------- TMA producer of the residual tiles of each d_ff tile
      tc::prefetch_map(&mBg); tc::prefetch_map(&mBu); tc::prefetch_map(&mAd);
      for (int lt = 0; lt < nft; ++lt) {
        const int n0 = (ft0 + lt) * NF;
        if (lt > 0 && !tc::bar_wait(&rb_empty, (lt - 1) & 1, ab, 52)) break;
        tc::bar_expect_tx(&rb_full, 2 * BRES_BYTES);
        tc::tma_load_2d(sBg, &mBg, &rb_full, 0, g * f + n0);
        tc::tma_load_2d(sBu, &mBu, &rb_full, 0, g * f + n0);
        if (lt > 0 && !tc::bar_wait(&ad_empty, (lt - 1) & 1, ab, 53)) break;
        tc::bar_expect_tx(&ad_full, AD_BYTES);
        tc::tma_load_2d(sAd, &mAd, &ad_full, n0, g * KRP);
        tc::tma_load_2d(sAd + KRP * 128, &mAd, &ad_full, n0 + 64, g * KRP);
      }
      if (abort_flag) tc::drain_copies();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- base MMA issuer: acc = X [Wg | Wu]^T, N = 256, then slot 0's residual
      //                  acc += D_0 [Bg | Bu]^T right behind the K loop
      constexpr uint32_t id_base = tc::idesc_bf16(kTile, 2 * NF);
      constexpr uint32_t id_res = tc::idesc_f16(kTile, NF);
      const uint32_t ug = tc::smem_u32(sUg), uu = tc::smem_u32(sUu);
      const uint32_t bg = tc::smem_u32(sBg), bu = tc::smem_u32(sBu);
      int kc = 0;
      bool ok = true;
      for (int lt = 0; lt < nft && ok; ++lt) {
        if (lt >= 1 && !tc::bar_wait(&acc_empty, (lt - 1) & 1, ab, 54)) break;
        tc::fence_after();
        for (int kb = 0; kb < nkb; ++kb, ++kc) {
          const int s = kc % STAGES, it = kc / STAGES;
          if (!tc::bar_wait(&full[s], it & 1, ab, 55)) { ok = false; break; }
          tc::fence_after();
          const uint32_t a0 = tc::smem_u32(sStage + s * STAGE_BYTES);
          const uint32_t b0 = a0 + X_BYTES;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_bf16(tmem, tc::sdesc(a0 + 32 * k), tc::sdesc(b0 + 32 * k), id_base, (kb | k) != 0);
          tc::mma_commit(&empty[s]);
        }
        if (!ok) break;
        if (!tc::bar_wait(&rb_full, lt & 1, ab, 58)) break;
        if (!tc::bar_wait(&u_ready, (lt * KE) & 1, ab, 60)) break;
        tc::fence_after();
#pragma unroll
        for (int kk = 0; kk < KRP / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;
          tc::mma_bf16(tmem, tc::sdesc(ug + off), tc::sdesc(bg + off), id_res, 1u);
          tc::mma_bf16(tmem + NF, tc::sdesc(uu + off), tc::sdesc(bu + off), id_res, 1u);
        }
        tc::mma_commit(&acc_full);
        if (KE == 1) tc::mma_commit(&rb_empty);
      }
      tc::mma_commit(&fin1);
      const uint64_t t0 = tc::now_ns();
      while (!tc::bar_test(&fin1, 0) && tc::now_ns() - t0 < tc::kWaitNs) {}
    }
  } else if (warp == 2) {
    if (lane == 0) {
      // ---------------- residual issuer: acc += D_s [Bg | Bu]^T for slots s >= 1; V_s += h_s Adn^T
      //                  (one slot behind)
      constexpr uint32_t id_res = tc::idesc_f16(kTile, NF);
      constexpr uint32_t id_v = tc::idesc_f16(kTile, KRP);
      const uint32_t ug = tc::smem_u32(sUg), uu = tc::smem_u32(sUu);
      const uint32_t bg = tc::smem_u32(sBg), bu = tc::smem_u32(sBu), ad = tc::smem_u32(sAd);
      const int n_slots = nft * KE;
      auto issue_v = [&](int tau) -> bool {
        const int lt = tau / KE, s = tau % KE;
        if (s == 0 && !tc::bar_wait(&ad_full, lt & 1, ab, 56)) return false;
        if (!tc::bar_wait(&h_ready[tau & 1], (tau >> 1) & 1, ab, 57)) return false;
        tc::fence_after();
        const uint32_t hcol = tmem + COL_H + 64 * (tau & 1);
#pragma unroll
        for (int kk = 0; kk < NF / 16; ++kk)
          tc::mma_f16_tmem_a(tmem + COL_V + s * KRP, hcol + 8 * kk,
                             tc::sdesc(ad + (kk >> 2) * (KRP * 128) + (kk & 3) * 32), id_v, (lt | kk) != 0);
        tc::mma_commit(&v_done[tau & 1]);
        if (s == KE - 1) tc::mma_commit(&ad_empty);
        return true;
      };
      bool ok = true;
      for (int sig = 0; sig < n_slots && ok; ++sig) {
        const int lt = sig / KE, s = sig % KE;
        // slot 0's residual is the base issuer's; the V of the previous tile's last slot goes
        // here (the new tile's base K loop is long); inside a tile, V of slot s - 1 follows R_s
        // so that R_s does not wait for h_{s-1}
        (void)lt;
        if (s == 0) {
          if (sig >= 1 && !issue_v(sig - 1)) { ok = false; break; }
          continue;
        }
        if (!tc::bar_wait(&u_ready, sig & 1, ab, 60)) { ok = false; break; }
        if (!tc::bar_wait(&acc_read, (sig - 1) & 1, ab, 61)) { ok = false; break; }
        tc::fence_after();
#pragma unroll
        for (int kk = 0; kk < KRP / 16; ++kk) {
          const uint32_t off_u = (kk & 3) * 32, off_b = (kk & 3) * 32;
          tc::mma_bf16(tmem, tc::sdesc(ug + off_u), tc::sdesc(bg + off_b), id_res, 1u);
          tc::mma_bf16(tmem + NF, tc::sdesc(uu + off_u), tc::sdesc(bu + off_b), id_res, 1u);
        }
        tc::mma_commit(&acc_full);
        if (s == KE - 1) tc::mma_commit(&rb_empty);
        if (!issue_v(sig - 1)) { ok = false; break; }
      }
      if (ok && n_slots > 0) issue_v(n_slots - 1);
      tc::mma_commit(&fin2);
      const uint64_t t0 = tc::now_ns();
      while (!tc::bar_test(&fin2, 0) && tc::now_ns() - t0 < tc::kWaitNs) {}
    }
  } else {
    // ---------------- epilogue: one thread per (tile row, quarter of 32 d_ff columns)
    const int q = warp & 3, part = (warp - kUpEpiWarp0) >> 2, row = q * 32 + lane, i = r0 + row;
    auto ewait = [&](uint64_t* b, uint32_t par, int where) -> bool {
      const bool r = tc::bar_wait(b, par, ab, where);
      return __all_sync(0xffffffffu, r);
    };
    const bool valid = i < r1;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int c0 = part * 32;
    // parts 0 and 1 keep this row's U~ blocks (gate, up); parts 2 and 3 only compute
    const bool builds = part < 2;
    uint8_t* sU = part == 0 ? sUg : sUu;
    int le[KE], eid[KE];
    float gt[KE];
#pragma unroll
    for (int s = 0; s < KE; ++s) { le[s] = 0; eid[s] = 0; gt[s] = 0.f; }
    const __half* urow = p.U;
    if (valid) {
      const int b = p.row_asg[i], t = b / p.kg, j = b % p.kg, k = p.kg * KE;
#pragma unroll
      for (int s = 0; s < KE; ++s) {
        const int e = p.eidx[(size_t)t * k + j * KE + s];
        le[s] = p.tab.local_of[e];
        eid[s] = e;
        gt[s] = p.gate[(size_t)t * k + j * KE + s];
      }
      urow = p.U + (p.u_by_token ? (size_t)t * p.G * 2 * KRP + (size_t)g * 2 * KRP : (size_t)i * 2 * KRP) +
             (part & 1) * KRP;
    }
    if (builds) {
      uint4* z = reinterpret_cast<uint4*>(sU + (row >> 3) * 1024 + (row & 7) * 128);
#pragma unroll
      for (int c = 0; c < 8; ++c) z[c] = make_uint4(0, 0, 0, 0);
    }
    auto load_u = [&](int s, uint32_t (&pk)[8]) {
      if (!valid || !builds) return;
      const uint4* u4 = reinterpret_cast<const uint4*>(urow + le[s] * kRank);
      const uint4 a = u4[0], b = u4[1];
      pk[0] = a.x; pk[1] = a.y; pk[2] = a.z; pk[3] = a.w;
      pk[4] = b.x; pk[5] = b.y; pk[6] = b.z; pk[7] = b.w;
    };
    auto zero_block = [&](int blk) {
      const uint4 z = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, blk * kRank, kTile)) = z;
      *reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, blk * kRank + 8, kTile)) = z;
    };
    int nz_pos = -1, nz_neg = -1;
    uint32_t unext[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) unext[c] = 0u;
    auto build_delta = [&](int s) {
      if (!valid || !builds) return;
      const int pos = le[s], neg = s > 0 ? le[s - 1] : -1;
      if (neg >= 0) {
        uint4* b0 = reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, neg * kRank, kTile));
        uint4* b1 = reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, neg * kRank + 8, kTile));
        const uint4 v0 = *b0, v1 = *b1;
        constexpr uint32_t F = 0x80008000u;          // exact FP16 negation
        *b0 = make_uint4(v0.x ^ F, v0.y ^ F, v0.z ^ F, v0.w ^ F);
        *b1 = make_uint4(v1.x ^ F, v1.y ^ F, v1.z ^ F, v1.w ^ F);
      }
      if (nz_neg >= 0 && nz_neg != pos && nz_neg != neg) zero_block(nz_neg);
      if (nz_pos >= 0 && nz_pos != pos && nz_pos != neg) zero_block(nz_pos);
      *reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, pos * kRank, kTile)) =
          make_uint4(unext[0], unext[1], unext[2], unext[3]);
      *reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, pos * kRank + 8, kTile)) =
          make_uint4(unext[4], unext[5], unext[6], unext[7]);
      nz_pos = pos; nz_neg = neg;
    };

    load_u(0, unext);
    build_delta(0);
    tc::fence_async_smem();
    warp_arrive(&u_ready);
    if (KE > 1) load_u(KE > 1 ? 1 : 0, unext);
    else if (nft > 1) load_u(0, unext);

    bool ok = true;
    int sig = 0;
    for (int lt = 0; lt < nft && ok; ++lt) {
      float hs[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) hs[c] = 0.f;
#pragma unroll
      for (int s = 0; s < KE; ++s, ++sig) {
        if (!ewait(&acc_full, sig & 1, 62)) { ok = false; break; }
        // R_s has finished reading the U~ tile.  Inside a tile the next delta is built now, so
        // that the next residual MMA waits only for acc to be read; the next tile's first delta
        // is built after acc is released (its MMA follows the next base K loop)
        auto next_delta = [&]() {
          build_delta(s + 1 < KE ? s + 1 : 0);
          tc::fence_async_smem();
          warp_arrive(&u_ready);
          const int s2 = (s + 2) % KE;
          const int lt2 = lt + (s + 2) / KE;
          if (lt2 < nft) load_u(s2, unext);
        };
        if (s + 1 < KE) next_delta();
        // the h buffer of this slot is free once the V MMA of slot sig - 2 has completed
        if (sig >= 2 && !ewait(&v_done[sig & 1], ((sig - 2) >> 1) & 1, 63)) { ok = false; break; }
        tc::fence_after();
        const uint32_t hbuf = tmem + lane_off + COL_H + 64 * (sig & 1) + c0 / 2;
        // two batches of 16 columns, one TMEM round trip each; acc is released as soon as the
        // second batch has been read, so the next slot's residual MMA overlaps the arithmetic
#pragma unroll
        for (int bt = 0; bt < 2; ++bt) {
          uint32_t av[16], bv[16];
          tc::tmem_ld16(tmem + lane_off + c0 + 16 * bt, av);
          tc::tmem_ld16(tmem + lane_off + NF + c0 + 16 * bt, bv);
          tc::tmem_ld_wait();
          if (bt == 1) {
            tc::fence_before();
            warp_arrive(&acc_read);
            if (s == KE - 1) {
              warp_arrive(&acc_empty);
              if (lt + 1 < nft) next_delta();
            }
          }
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float h2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              h2[u] = silu_fast(__uint_as_float(av[e + u])) * __uint_as_float(bv[e + u]);
              hs[16 * bt + e + u] += gt[s] * h2[u];
            }
            __half2 hh = __floats2half2_rn(h2[0], h2[1]);
            pk[e / 2] = *reinterpret_cast<uint32_t*>(&hh);
          }
          tc::tmem_st4(hbuf + 8 * bt, pk[0], pk[1], pk[2], pk[3]);
          tc::tmem_st4(hbuf + 8 * bt + 4, pk[4], pk[5], pk[6], pk[7]);
        }
        tc::tmem_st_wait();
        tc::fence_before();
        warp_arrive(&h_ready[sig & 1]);
      }
      if (!ok) break;
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(p.hsum + (size_t)i * f + (ft0 + lt) * NF + c0);
#pragma unroll
        for (int c = 0; c < 32; c += 8)
          dst[c / 8] = make_uint4(tc::pack_bf16(hs[c], hs[c + 1]), tc::pack_bf16(hs[c + 2], hs[c + 3]),
                                  tc::pack_bf16(hs[c + 4], hs[c + 5]), tc::pack_bf16(hs[c + 6], hs[c + 7]));
      }
    }
    // every V MMA has completed: the last two commits of v_done
    if (ok && sig >= 1) ok = ewait(&v_done[(sig - 1) & 1], ((sig - 1) >> 1) & 1, 64);
    if (ok && sig >= 2) ok = ewait(&v_done[(sig - 2) & 1], ((sig - 2) >> 1) & 1, 65);
    if (ok) {
      tc::fence_after();
      // V_s of slot s is read by part s; the row's expert block le[s] of the KRP columns
#pragma unroll
      for (int s = 0; s < KE; ++s) {
        if (part != s) continue;
        float v[kRank];
#pragma unroll
        for (int k = 0; k < kRank; ++k) v[k] = 0.f;
#pragma unroll
        for (int jb = 0; jb < KRP / 16; ++jb) {
          uint32_t vv[16];
          tc::tmem_ld16(tmem + lane_off + COL_V + s * KRP + jb * 16, vv);
          tc::tmem_ld_wait();
          if (jb == le[s]) {
#pragma unroll
            for (int k = 0; k < kRank; ++k) v[k] = __uint_as_float(vv[k]);
          }
        }
        if (valid) {
          float* vp = p.Vpart + ((size_t)chunk * p.R + i) * KE * kRank + s * kRank;
#pragma unroll
          for (int k = 0; k < kRank; k += 4)
            *reinterpret_cast<float4*>(vp + k) =
                make_float4(gt[s] * v[k], gt[s] * v[k + 1], gt[s] * v[k + 2], gt[s] * v[k + 3]);
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------------
// 4c. Fused gate/up on 256-column MMAs with a double-buffered accumulator, on CTA pairs (K r = 64
//     columns, at most two slots per row).
//
// As 4b, but TMEM holds two accumulators acc[b] = [gate 128 | up 128] (512 columns) so that the
// next tile's K loop runs during this tile's slots, and V_s = A_down^T h_s is accumulated on the
// CUDA cores: each epilogue thread keeps, for its row and its 64 d_ff columns, the 16 partial
// sums of each slot, reading the row's expert block of A_down^T from a transposed FP16 tile in
// shared memory.  12 warps: base TMA, base MMA, residual MMA, residual TMA, 8 epilogue warps
// (two per TMEM lane quarter, 64 d_ff columns each).
//
// The two CTAs of a cluster take two 128-row tiles of one group (pair tiles as in the pair GEMM)
// and the same chunk of d_ff tiles; rank 0 issues every MMA with M = 256 (cta_group::2).  For the
// base product rank 0 holds the W_gate tile and rank 1 the W_up tile of B (N = 256 = gate | up),
// so a K step lands 16 KB of X and 16 KB of W per SM instead of 16 + 32 KB: the shared-memory
// fill rate, not the tensor pipe, bounds a single CTA here.  The residual MMAs (N = 128 each)
// split B_gate / B_up by rows (64 per CTA); each CTA keeps its own U~ tiles, A_down^T tile and
// epilogue.  Both CTAs' loads of a stage complete on rank 0's barrier; rank 0's commits arrive on
// the barriers of the CTAs that wait on them; the epilogues of both CTAs arrive on rank 0's
// barriers.
// ------------------------------------------------------------------------------------------
constexpr int kUp4EpiWarps = 8;
constexpr int kStages4p = 5;
// registers per thread: at launch (the __launch_bounds__ limit for 384 threads, one CTA per SM),
// and after the split between warpgroup 0 (producers, issuers) and the two epilogue warpgroups
// (the counts at which neither side spills, per number of slots)
constexpr int kUp4RegsLaunch = 168;
template <int KE> constexpr int kUp4RegsLow = KE == 1 ? 88 : 120;
template <int KE> constexpr int kUp4RegsHigh = KE == 1 ? 208 : 192;
static_assert(kUpWarps == 12 && kUpEpiWarp0 == 4 && kUp4EpiWarps == 8, "one producer warpgroup, two epilogue");
static_assert(4 * kUp4RegsLow<1> + 8 * kUp4RegsHigh<1> <= 12 * kUp4RegsLaunch &&
                  4 * kUp4RegsLow<2> + 8 * kUp4RegsHigh<2> <= 12 * kUp4RegsLaunch,
              "the split must not exceed the launch's registers");

template <int KE>
__global__ void __launch_bounds__(kUpWarps * 32, 1) ffn_up4p_kernel(
    const __grid_constant__ CUtensorMap mX, const __grid_constant__ CUtensorMap mWg,
    const __grid_constant__ CUtensorMap mWu, const __grid_constant__ CUtensorMap mBg,
    const __grid_constant__ CUtensorMap mBu, const __grid_constant__ CUtensorMap mAdt, const UpArgs p) {
  pdl_wait();
  pdl_trigger();
  constexpr int KRP = 64, NF = kNf3, STAGES = kStages4p;
  constexpr uint32_t X_BYTES = kTile * 128, W_BYTES = NF * 128, STAGE_BYTES = X_BYTES + W_BYTES;   // per CTA
  constexpr uint32_t BRES_BYTES = (NF / 2) * KRP * 2;      // this CTA's half of B_gate or B_up: 64 rows x KRP
  constexpr uint32_t ADT_BYTES = NF * KRP * 2;             // A_down^T transposed: 128 d_ff columns x KRP (FP16)
  constexpr uint32_t UT_BYTES = kTile * KRP * 2;
  static_assert(KE >= 1 && KE <= 2, "slots");

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[STAGES], empty[STAGES];
  __shared__ uint64_t base_full[2], acc_empty[2];
  __shared__ uint64_t rb_full, rb_empty, ad_full, ad_empty;
  __shared__ uint64_t acc_full, acc_read, u_ready, fin1, fin2;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const uint32_t rank = tc::cluster_rank();
  // work items w = pair tile * n_chunks + chunk, taken by cluster c as c, c + clusters, ...: the
  // clusters running at once cover a band of consecutive pair tiles across every chunk, so the
  // band's X rows stay in L2 while they are re-read for each d_ff tile, and each W tile is read
  // from DRAM about once per round of items.  Both CTAs of a cluster walk the same items (a pair
  // tile is empty for both or for neither), every role skips the empty ones alike, and the stage
  // ring, accumulator parity and slot phases run on across items (glt: tiles, sig: slots over the
  // cluster's items).
  const int cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;
  const int n_items = p.n_row_tiles * p.n_chunks;
  auto item = [&](int w, int& g, int& r0, int& r1, int& ft0, int& nft) -> bool {
    if (!pair_tile_of(p.row_begin, p.G, w / p.n_chunks, (int)rank, g, r0, r1)) return false;
    ft0 = (w % p.n_chunks) * p.ftiles_per_chunk;
    nft = min(ft0 + p.ftiles_per_chunk, p.n_ftiles) - ft0;
    return nft > 0;
  };
  const int nkb = p.d / 64;
  const int f = p.f;

  uint8_t* smem = align1024(smem_raw);
  uint8_t* sStage = smem;
  uint8_t* sBg = sStage + STAGES * STAGE_BYTES;
  uint8_t* sBu = sBg + BRES_BYTES;
  uint8_t* sAdt = sBu + BRES_BYTES;
  uint8_t* sUg = sAdt + ADT_BYTES;
  uint8_t* sUu = sUg + UT_BYTES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tc::Abort ab{&abort_flag, p.status};
  constexpr int kEpiArrive = 2 * kUp4EpiWarps;             // epilogue warps of both CTAs (rank 0's barriers)
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { tc::bar_init(&full[s], 1); tc::bar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { tc::bar_init(&base_full[b], 1); tc::bar_init(&acc_empty[b], kEpiArrive); }
    tc::bar_init(&rb_full, 1); tc::bar_init(&rb_empty, 1);
    tc::bar_init(&ad_full, 1); tc::bar_init(&ad_empty, kUp4EpiWarps);
    tc::bar_init(&acc_full, 1);
    tc::bar_init(&acc_read, kEpiArrive);
    tc::bar_init(&u_ready, kEpiArrive);
    tc::bar_init(&fin1, 1); tc::bar_init(&fin2, 1);
    abort_flag = 0;
    tc::bar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc_pair(&tmem_base, 512);
  tc::fence_before();
  // both CTAs' barriers are initialised before either CTA signals the other's
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  tc::fence_after();
  const uint32_t tmem = tmem_base;
  // epilogue arrivals go to rank 0's barrier at the same offset
  auto warp_arrive0 = [&](uint64_t* b) {
    __syncwarp();
    if (lane == 0) tc::bar_arrive_cluster(tc::map_shared(tc::smem_u32(b), 0));
  };
  auto warp_arrive = [&](uint64_t* b) {
    __syncwarp();
    if (lane == 0) tc::bar_arrive(b);
  };
  // the single-lane producer and issuer roles (warpgroup 0) hand registers to the epilogue
  // warpgroups, whose per-thread V partials, gated h sums and TMEM reads do not fit in the
  // launch's even share: 4 x 32 x low + 8 x 32 x high <= 384 x kUp4RegsLaunch
  if (warp < kUpEpiWarp0) {
    tc::setmaxnreg_dec<kUp4RegsLow<KE>>();
    if (warp == 0) {
      if (lane == 0) {
        // ---------------- TMA producer (both CTAs): own X rows and own W tile (rank 0 gate, rank 1 up)
        tc::prefetch_map(&mX); tc::prefetch_map(rank == 0 ? &mWg : &mWu);
        const uint32_t full0 = tc::map_shared(tc::smem_u32(&full[0]), 0);
        int kc = 0;
        bool ok = true;
        for (int w = cluster; w < n_items && ok; w += clusters) {
          int g, r0, r1, ft0, nft;
          if (!item(w, g, r0, r1, ft0, nft)) continue;
          for (int lt = 0; lt < nft && ok; ++lt) {
            const int n0 = (ft0 + lt) * NF;
            for (int kb = 0; kb < nkb; ++kb, ++kc) {
              const int s = kc % STAGES, it = kc / STAGES;
              if (kc >= STAGES && !tc::bar_wait_cluster(&empty[s], (it - 1) & 1, ab, 91)) { ok = false; break; }
              uint8_t* st = sStage + s * STAGE_BYTES;
              if (rank == 0) tc::bar_expect_tx(&full[s], 2 * STAGE_BYTES);
              tc::tma_load_2d_pair(st, &mX, full0 + 8 * s, kb * 64, r0);
              tc::tma_load_2d_pair(st + X_BYTES, rank == 0 ? &mWg : &mWu, full0 + 8 * s, kb * 64,
                                   (int)p.tab.wslot[g] * f + n0);
            }
          }
        }
        // every commit rank 0 sends to this CTA's stage barriers has landed before the CTA exits
        if (ok) {
          for (int s = 0; s < STAGES && s < kc; ++s)
            if (!tc::bar_wait_cluster(&empty[s], ((kc - 1 - s) / STAGES) & 1, ab, 92)) break;
        }
        if (abort_flag) tc::drain_copies();
      }
    } else if (warp == 3) {
      if (lane == 0) {
        // ---------------- TMA producer of the residual tiles: this CTA's halves of B_gate / B_up
        //                  (pair loads, counted on rank 0) and the whole A_down^T tile (local)
        tc::prefetch_map(&mBg); tc::prefetch_map(&mBu); tc::prefetch_map(&mAdt);
        const uint32_t rb0 = tc::map_shared(tc::smem_u32(&rb_full), 0);
        bool ok = true;
        int glt = 0;
        for (int w = cluster; w < n_items && ok; w += clusters) {
          int g, r0, r1, ft0, nft;
          if (!item(w, g, r0, r1, ft0, nft)) continue;
          for (int lt = 0; lt < nft; ++lt, ++glt) {
            const int n0 = (ft0 + lt) * NF;
            if (glt > 0 && !tc::bar_wait_cluster(&rb_empty, (glt - 1) & 1, ab, 93)) { ok = false; break; }
            if (rank == 0) tc::bar_expect_tx(&rb_full, 4 * BRES_BYTES);
            tc::tma_load_2d_pair(sBg, &mBg, rb0, 0, g * f + n0 + (int)rank * (NF / 2));
            tc::tma_load_2d_pair(sBu, &mBu, rb0, 0, g * f + n0 + (int)rank * (NF / 2));
            if (glt > 0 && !tc::bar_wait(&ad_empty, (glt - 1) & 1, ab, 94)) { ok = false; break; }
            tc::bar_expect_tx(&ad_full, ADT_BYTES);
            tc::tma_load_2d(sAdt, &mAdt, &ad_full, 0, g * f + n0);
          }
        }
        // rank 0's last release of the residual tiles has landed before the CTA exits
        if (ok && glt > 0) tc::bar_wait_cluster(&rb_empty, (glt - 1) & 1, ab, 95);
        if (abort_flag) tc::drain_copies();
      }
    } else if (warp == 1) {
      if (lane == 0 && rank == 0) {
        // ---------------- base MMA issuer (rank 0): acc[lt & 1] = X [Wg | Wu]^T, M = 256, N = 256
        constexpr uint32_t id_base = tc::idesc_bf16(2 * kTile, 2 * NF);
        int kc = 0, glt = 0;
        bool ok = true;
        for (int w = cluster; w < n_items && ok; w += clusters) {
          int g, r0, r1, ft0, nft;
          if (!item(w, g, r0, r1, ft0, nft)) continue;
          for (int lt = 0; lt < nft && ok; ++lt, ++glt) {
            const int b = glt & 1;
            if (glt >= 2 && !tc::bar_wait_cluster(&acc_empty[b], ((glt >> 1) - 1) & 1, ab, 96)) { ok = false; break; }
            tc::fence_after();
            const uint32_t dcol = tmem + b * 2 * NF;
            for (int kb = 0; kb < nkb; ++kb, ++kc) {
              const int s = kc % STAGES, it = kc / STAGES;
              if (!tc::bar_wait_cluster(&full[s], it & 1, ab, 97)) { ok = false; break; }
              tc::fence_after();
              const uint32_t a0 = tc::smem_u32(sStage + s * STAGE_BYTES);
              const uint32_t b0 = a0 + X_BYTES;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                tc::mma_bf16_pair(dcol, tc::sdesc(a0 + 32 * k), tc::sdesc(b0 + 32 * k), id_base, (kb | k) != 0);
              tc::mma_commit_pair(&empty[s], 3);
            }
            if (!ok) break;
            tc::mma_commit_pair(&base_full[b], 1);
          }
        }
        tc::mma_commit_pair(&fin1, 1);
        const uint64_t t0 = tc::now_ns();
        while (!tc::bar_test(&fin1, 0) && tc::now_ns() - t0 < tc::kWaitNs) {}
      }
    } else if (warp == 2) {
      if (lane == 0 && rank == 0) {
        // ---------------- residual issuer (rank 0): acc[b] += D_s [Bg | Bu]^T, M = 256, two N = 128
        constexpr uint32_t id_res = tc::idesc_f16(2 * kTile, NF);
        const uint32_t ug = tc::smem_u32(sUg), uu = tc::smem_u32(sUu);
        const uint32_t bg = tc::smem_u32(sBg), bu = tc::smem_u32(sBu);
        bool ok = true;
        int sig = 0;
        for (int w = cluster; w < n_items && ok; w += clusters) {
          int g, r0, r1, ft0, nft;
          if (!item(w, g, r0, r1, ft0, nft)) continue;
          for (int ls = 0; ls < nft * KE && ok; ++ls, ++sig) {
            const int glt = sig / KE, s = sig % KE, b = glt & 1;
            if (s == 0) {
              if (!tc::bar_wait(&base_full[b], (glt >> 1) & 1, ab, 98)) { ok = false; break; }
              if (!tc::bar_wait_cluster(&rb_full, glt & 1, ab, 99)) { ok = false; break; }
            }
            if (!tc::bar_wait_cluster(&u_ready, sig & 1, ab, 100)) { ok = false; break; }
            if (s > 0 && !tc::bar_wait_cluster(&acc_read, (sig - 1) & 1, ab, 101)) { ok = false; break; }
            tc::fence_after();
            const uint32_t dcol = tmem + b * 2 * NF;
#pragma unroll
            for (int kk = 0; kk < KRP / 16; ++kk) {
              const uint32_t off = (kk & 3) * 32;
              tc::mma_bf16_pair(dcol, tc::sdesc(ug + off), tc::sdesc(bg + off), id_res, 1u);
              tc::mma_bf16_pair(dcol + NF, tc::sdesc(uu + off), tc::sdesc(bu + off), id_res, 1u);
            }
            tc::mma_commit_pair(&acc_full, 3);
            if (s == KE - 1) tc::mma_commit_pair(&rb_empty, 3);
          }
        }
        tc::mma_commit_pair(&fin2, 1);
        const uint64_t t0 = tc::now_ns();
        while (!tc::bar_test(&fin2, 0) && tc::now_ns() - t0 < tc::kWaitNs) {}
      }
    }
  } else {
    tc::setmaxnreg_inc<kUp4RegsHigh<KE>>();
    // ---------------- epilogue (both CTAs): one thread per (tile row, half of 64 d_ff columns)
    const int q = warp & 3, half = (warp - kUpEpiWarp0) >> 2, row = q * 32 + lane;
    auto ewait = [&](uint64_t* b, uint32_t par, int where) -> bool {
      const bool r = tc::bar_wait_cluster(b, par, ab, where);
      return __all_sync(0xffffffffu, r);
    };
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int c0 = half * 64;
    uint8_t* sU = half == 0 ? sUg : sUu;
    // this row of this half's U~ starts at zero (later items find the previous item's last delta
    // there, which the first delta of the item clears)
    {
      uint4* z = reinterpret_cast<uint4*>(sU + (row >> 3) * 1024 + (row & 7) * 128);
#pragma unroll
      for (int c = 0; c < 8; ++c) z[c] = make_uint4(0, 0, 0, 0);
    }
    // U~ holds the last delta: +values in block nz_pos, -values in block nz_neg (or none)
    int nz_pos = -1, nz_neg = -1;
    uint32_t unext[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) unext[c] = 0u;
    bool ok = true;
    int sig = 0, glt = 0;
    for (int w = cluster; w < n_items && ok; w += clusters) {
      int g, r0, r1, ft0, nft;
      if (!item(w, g, r0, r1, ft0, nft)) continue;
      const int i = r0 + row, chunk = w % p.n_chunks;
      const bool valid = i < r1;
      int le[KE];
      float gt[KE];
#pragma unroll
      for (int s = 0; s < KE; ++s) { le[s] = 0; gt[s] = 0.f; }
      const __half* urow = p.U;
      if (valid) {
        const int b = p.row_asg[i], t = b / p.kg, j = b % p.kg, k = p.kg * KE;
#pragma unroll
        for (int s = 0; s < KE; ++s) {
          const int e = p.eidx[(size_t)t * k + j * KE + s];
          le[s] = p.tab.local_of[e];
          gt[s] = p.gate[(size_t)t * k + j * KE + s];
        }
        urow = p.U + (p.u_by_token ? (size_t)t * p.G * 2 * KRP + (size_t)g * 2 * KRP : (size_t)i * 2 * KRP) +
               half * KRP;
      }
      auto load_u = [&](int s, uint32_t (&pk)[8]) {
        if (!valid) return;
        const uint4* u4 = reinterpret_cast<const uint4*>(urow + le[s] * kRank);
        const uint4 a = u4[0], b = u4[1];
        pk[0] = a.x; pk[1] = a.y; pk[2] = a.z; pk[3] = a.w;
        pk[4] = b.x; pk[5] = b.y; pk[6] = b.z; pk[7] = b.w;
      };
      auto zero_block = [&](int blk) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, blk * kRank, kTile)) = z;
        *reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, blk * kRank + 8, kTile)) = z;
      };
      // writes the delta of slot s (first slot of a tile: no subtraction) from unext
      auto build_delta = [&](int s) {
        if (!valid) return;
        const int pos = le[s], neg = s > 0 ? le[s - 1] : -1;
        if (neg >= 0) {
          uint4* b0 = reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, neg * kRank, kTile));
          uint4* b1 = reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, neg * kRank + 8, kTile));
          const uint4 v0 = *b0, v1 = *b1;
          constexpr uint32_t F = 0x80008000u;          // exact FP16 negation
          *b0 = make_uint4(v0.x ^ F, v0.y ^ F, v0.z ^ F, v0.w ^ F);
          *b1 = make_uint4(v1.x ^ F, v1.y ^ F, v1.z ^ F, v1.w ^ F);
        }
        if (nz_neg >= 0 && nz_neg != pos && nz_neg != neg) zero_block(nz_neg);
        if (nz_pos >= 0 && nz_pos != pos && nz_pos != neg) zero_block(nz_pos);
        *reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, pos * kRank, kTile)) =
            make_uint4(unext[0], unext[1], unext[2], unext[3]);
        *reinterpret_cast<uint4*>(sU + tc::sw128_offset(row, pos * kRank + 8, kTile)) =
            make_uint4(unext[4], unext[5], unext[6], unext[7]);
        nz_pos = pos; nz_neg = neg;
      };

      // U~ is free here: the residual MMA of the previous item's last slot has completed
      load_u(0, unext);
      build_delta(0);
      tc::fence_async_smem();
      warp_arrive0(&u_ready);
      if (KE > 1) load_u(KE > 1 ? 1 : 0, unext);
      else if (nft > 1) load_u(0, unext);

      // V partials of this row over this thread's columns, per slot, as FP32 pairs (k, k + 1)
      float2 vacc[KE][kRank / 2];
#pragma unroll
      for (int s = 0; s < KE; ++s)
#pragma unroll
        for (int k = 0; k < kRank / 2; ++k) vacc[s][k] = make_float2(0.f, 0.f);

      for (int lt = 0; lt < nft && ok; ++lt, ++glt) {
        const int bsel = glt & 1;
        const uint32_t acc_col = bsel * 2 * NF;
        if (!ewait(&ad_full, glt & 1, 102)) { ok = false; break; }
        float hs[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) hs[c] = 0.f;
#pragma unroll
        for (int s = 0; s < KE; ++s, ++sig) {
          if (!ewait(&acc_full, sig & 1, 103)) { ok = false; break; }
          tc::fence_after();
          const uint8_t* arow = sAdt + le[s] * kRank * 2;       // this row's expert block, column stride KRP
#pragma unroll
          for (int bt = 0; bt < 4; ++bt) {
            uint32_t av[16], bv[16];
            tc::tmem_ld16(tmem + lane_off + acc_col + c0 + 16 * bt, av);
            tc::tmem_ld16(tmem + lane_off + acc_col + NF + c0 + 16 * bt, bv);
            tc::tmem_ld_wait();
            if (bt == 3) {
              // this thread has read acc for this slot: the next slot's residual may land
              tc::fence_before();
              warp_arrive0(&acc_read);
              if (s == KE - 1) warp_arrive0(&acc_empty[bsel]);
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float h = silu_fast(__uint_as_float(av[e])) * __uint_as_float(bv[e]);
              hs[16 * bt + e] += gt[s] * h;
              // v_k += h * A_down^T[k][c] for the 16 ranks of the row's expert
              const int c = c0 + 16 * bt + e;
              const uint4* ap = reinterpret_cast<const uint4*>(arow + (size_t)c * KRP * 2);
              const uint4 w0 = ap[0], w1 = ap[1];
              const uint32_t ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
              const float2 h2 = make_float2(h, h);
#pragma unroll
              for (int k2 = 0; k2 < 8; ++k2) {
                const float2 a2 = __half22float2(*reinterpret_cast<const __half2*>(&ww[k2]));
                vacc[s][k2] = fma2(h2, a2, vacc[s][k2]);
              }
            }
          }
          const bool more = s + 1 < KE || lt + 1 < nft;
          if (more) {
            build_delta(s + 1 < KE ? s + 1 : 0);
            tc::fence_async_smem();
            warp_arrive0(&u_ready);
            const int s2 = (s + 2) % KE;
            const int lt2 = lt + (s + 2) / KE;
            if (lt2 < nft) load_u(s2, unext);
          }
        }
        if (!ok) break;
        warp_arrive(&ad_empty);                        // done with this tile's A_down^T (local)
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.hsum + (size_t)i * f + (ft0 + lt) * NF + c0);
#pragma unroll
          for (int c = 0; c < 64; c += 8)
            dst[c / 8] = make_uint4(tc::pack_bf16(hs[c], hs[c + 1]), tc::pack_bf16(hs[c + 2], hs[c + 3]),
                                    tc::pack_bf16(hs[c + 4], hs[c + 5]), tc::pack_bf16(hs[c + 6], hs[c + 7]));
        }
      }
      if (ok && valid) {
        // partial over this half's columns: V parts [chunk][half]
        float* vp = p.Vpart + (((size_t)chunk * 2 + half) * p.R + i) * KE * kRank;
#pragma unroll
        for (int s = 0; s < KE; ++s)
#pragma unroll
          for (int k = 0; k < kRank; k += 4)
            *reinterpret_cast<float4*>(vp + s * kRank + k) =
                make_float4(gt[s] * vacc[s][k / 2].x, gt[s] * vacc[s][k / 2].y, gt[s] * vacc[s][k / 2 + 1].x,
                            gt[s] * vacc[s][k / 2 + 1].y);
      }
    }
  }
  tc::fence_before();
  // neither CTA leaves while the other may still arrive on its barriers or read its memory
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc_pair(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------------
// 5. V~[i][j*16 + k] = sum over column chunks of the gated v of the slot whose expert is local j
// ------------------------------------------------------------------------------------------
__global__ void v_reduce_kernel(const float* __restrict__ Vpart, const int32_t* __restrict__ row_asg,
                                const int32_t* __restrict__ eidx, GroupTable tab, int R, int kg, int ke,
                                int nchunks, int KRP, __nv_bfloat16* __restrict__ Vt) {
  pdl_wait();
  pdl_trigger();
  // one thread per (row, 16-wide block of V~, quarter of the block): the block of local expert jb
  // holds the gated v of the row's slot routed to that expert (zero if none); both halves (hi,
  // lo of Bdn) get a copy
  const int nblk = KRP / kRank;
  const int w = blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= R * nblk * 4) return;
  const int qt = w & 3, i = (w >> 2) / nblk, jb = (w >> 2) % nblk;
  const int b = row_asg[i], t = b / kg, j = b % kg;
  int slot = -1;
  for (int s = 0; s < ke; ++s)
    if (jb < tab.K && tab.local_of[eidx[(size_t)t * kg * ke + j * ke + s]] == jb) slot = s;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (slot >= 0) {
    const float4* src = reinterpret_cast<const float4*>(Vpart + ((size_t)i * ke + slot) * kRank) + qt;
    const size_t cstride = (size_t)R * ke * kRank / 4;   // float4s per chunk
    int c = 0;
    for (; c + 8 <= nchunks; c += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = src[(c + u) * cstride];
#pragma unroll
      for (int u = 0; u < 8; ++u) { acc.x += v[u].x; acc.y += v[u].y; acc.z += v[u].z; acc.w += v[u].w; }
    }
    for (; c < nchunks; ++c) {
      const float4 v = src[c * cstride];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
  }
  const uint2 pk = make_uint2(tc::pack_bf16(acc.x, acc.y), tc::pack_bf16(acc.z, acc.w));
  uint2* row = reinterpret_cast<uint2*>(Vt + (size_t)i * 2 * KRP);
  row[(jb * kRank) / 4 + qt] = pk;
  row[(KRP + jb * kRank) / 4 + qt] = pk;
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

// BF16 matrix [rows][cols] (row stride cols), box {64, box_rows}, 128-byte swizzle, zero fill.
static bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return make_map(m, base, rows, cols, box_rows);
}

// 16-bit matrix [rows][cols], box {cols, box_rows}, no swizzle (rows land contiguously in shared
// memory, for CUDA-core reads); cols * 2 bytes must be a multiple of 16.
static bool make_map_plain(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_path_ok(const LayerArgs& a) {
  const int KRP = ((a.K * a.r + 63) / 64) * 64;
  return a.bf16 && a.int4 && a.r == kRank && a.K * a.r <= 128 && KRP <= 128 && a.ke <= kMaxKe &&
         a.d % 128 == 0 && a.f % 64 == 0;
}

int tc_krp(const LayerArgs& a) { return ((a.K * a.r + 63) / 64) * 64; }

// Number of d_ff chunks per row tile.  Row tiles are only known on the device, so the host
// estimates them (full tiles plus about half a partial tile per group, or one tile per group
// when groups hold fewer than 128 rows) and picks the chunk count whose waves of one item per SM
// cost least: ceil(items / SMs) x (tiles per chunk + a fixed per-item overhead).
// Which fused gate/up kernel runs: the 256-column one (4b) when K r fits 64 columns, at most
// two slots and d_ff is a multiple of 128; otherwise the 128-column one (4).
static bool up3_ok(const LayerArgs& a) { return tc_krp(a) == 64 && a.ke <= 2 && a.f % kNf3 == 0; }

static bool up4_ok(const LayerArgs& a);

int tc_up_chunks(const LayerArgs& a) {
  const int n_ft = a.f / (up3_ok(a) ? kNf3 : kNf);
  const bool pair = up4_ok(a);
  // The 128-column kernel is persistent: an item boundary costs about a tenth of a tile (the next
  // item's K loop runs under the previous item's slots).  The 256-column kernel pays half a tile
  // per CTA.  The pair kernel walks items too, but on the Mixtral shape finer items that balance
  // its two rounds gained under 1% and added V-partial traffic (28 chunks: 1.377 vs 1.389 ms, V
  // reduction 20 vs 9 us), so it is costed like the 256-column kernel.
  const double item_cost = up3_ok(a) || pair ? 0.5 : 0.1;
  const int full = (a.R + kTile - 1) / kTile;
  // units per chunk that find rows (a group's last tile is ragged: about half of them add one),
  // and how many run at once (a CTA per SM, or a pair of CTAs per two SMs)
  int units = a.R >= kTile * a.G ? full + (a.G + 1) / 2 : (a.R < a.G ? a.R : a.G);
  if (pair) units = a.R >= 2 * kTile * a.G ? (a.R + 2 * kTile - 1) / (2 * kTile) + (a.G + 1) / 2 : units;
  if (units < 1) units = 1;
  const int slots = pair ? 148 / 2 : 148;
  // The pair kernel's clusters running at once cover slots / c consecutive pair tiles: enough
  // chunks that their X rows (256 rows of d_model each) take at most about 40 MB, so that they
  // stay in L2 while W streams past (on the Mixtral shape 4 chunks read 1.05 GB from DRAM per
  // launch, 2 chunks with all 33 pair tiles live 2.87 GB)
  int min_c = 1;
  if (pair) {
    const double band_bytes = 40.0 * (1 << 20), tile_bytes = 2.0 * kTile * a.d * 2;
    const int band = (int)(band_bytes / tile_bytes) > 1 ? (int)(band_bytes / tile_bytes) : 1;
    min_c = (slots + band - 1) / band;
  }
  int best = 0;
  double best_cost = 1e30;
  for (int c = 1; c <= n_ft; ++c) {
    const int per = (n_ft + c - 1) / c;
    if (c > 1 && (n_ft + per - 1) / per != c) continue;     // same split as a smaller count
    if (c < min_c && c < n_ft) continue;
    const double rounds = (double)((units * c + slots - 1) / slots);
    const double cost = rounds * (per + item_cost);
    if (cost < best_cost - 1e-9) { best_cost = cost; best = c; }
  }
  return best > 0 ? best : n_ft;
}

template <int BN, int OUT>
static cudaError_t launch_gemm(const CUtensorMap& A0, const CUtensorMap& A1, const CUtensorMap& B0,
                               const CUtensorMap& B1, int nk0, int nk1, const int32_t* row_begin, int G,
                               int n_out, int b_stride, int b1_off, int tiles, void* out, int out_ld,
                               const int32_t* scatter, DevStatus* st, cudaStream_t stream, const SlotMap& b0s) {
  constexpr int STAGES = BN >= 256 ? 4 : 6;
  const size_t smem = 1024 + (size_t)STAGES * (kTile * 128 + BN * 128);
  static std::atomic<uint64_t> attr{0};
  if (const cudaError_t e = smem_attr_once(tc_gemm_kernel<BN, STAGES, OUT>, smem, attr); e != cudaSuccess) return e;
  dim3 grid(n_out / BN, tiles);
  return launch_pdl(tc_gemm_kernel<BN, STAGES, OUT>, grid, dim3(192), smem, stream, A0, A1, B0, B1, nk0, nk1,
                    row_begin, G, b_stride, b1_off, out, out_ld, scatter, st, b0s);
}

// Persistent version: one CTA per SM over all (row tile, N tile) items.
template <int BN, int OUT>
static cudaError_t launch_gemm_persist(const CUtensorMap& A0, const CUtensorMap& A1, const CUtensorMap& B0,
                                       const CUtensorMap& B1, int nk0, int nk1, const int32_t* row_begin, int G,
                                       int n_out, int b_stride, int b1_off, int tiles, void* out, int out_ld,
                                       const int32_t* scatter, DevStatus* st, cudaStream_t stream,
                                       const SlotMap& b0s) {
  constexpr int STAGES = BN >= 256 ? 4 : 6;
  const size_t smem = 1024 + (size_t)STAGES * (kTile * 128 + BN * 128);
  static std::atomic<uint64_t> attr{0};
  if (const cudaError_t e = smem_attr_once(tc_gemm_persist_kernel<BN, STAGES, OUT>, smem, attr); e != cudaSuccess)
    return e;
  int dev = 0, sms = 0;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
  if (cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev); e != cudaSuccess) return e;
  const int n_tiles = n_out / BN, items = tiles * n_tiles;
  return launch_pdl(tc_gemm_persist_kernel<BN, STAGES, OUT>, dim3(items < sms ? items : sms), dim3(192), smem, stream,
                    A0, A1, B0, B1, nk0, nk1, row_begin, G, b_stride, b1_off, tiles, n_tiles, out, out_ld, scatter, st,
                    b0s);
}

// CTA-pair version: grid.x = 2 x (an upper bound of the row-tile pairs), clusters of two CTAs
// along x (the pair of a cta_group::2 MMA is formed along x), grid.y = N tiles of BN.
template <int BN, int OUT>
static cudaError_t launch_gemm_pair(const CUtensorMap& A0, const CUtensorMap& A1, const CUtensorMap& B0,
                                    const CUtensorMap& B1, int nk0, int nk1, const int32_t* row_begin, int G,
                                    int n_out, int b_stride, int b1_off, int pairs, void* out, int out_ld,
                                    const int32_t* scatter, DevStatus* st, cudaStream_t stream, const SlotMap& b0s,
                                    int dense_rows = 0, int band = 0) {
  constexpr int STAGES = BN >= 256 ? 6 : 8;
  const size_t smem = 1024 + (size_t)STAGES * (kTile * 128 + (BN / 2) * 128);
  static std::atomic<uint64_t> attr{0};
  if (const cudaError_t e = smem_attr_once(tc_gemm_pair_kernel<BN, STAGES, OUT>, smem, attr); e != cudaSuccess) return e;
  return launch_pdl_cluster(tc_gemm_pair_kernel<BN, STAGES, OUT>, dim3(2 * pairs, n_out / BN), dim3(192),
                            dim3(2, 1, 1), smem, stream, A0, A1, B0, B1, nk0, nk1, row_begin, G, b_stride, b1_off,
                            out, out_ld, scatter, st, dense_rows, b0s, band);
}

template <int KRP, int KE>
static cudaError_t launch_up_ke(const CUtensorMap* maps, const UpArgs& p, int nchunks, int tiles, cudaStream_t stream) {
  constexpr int STAGES = KRP >= 128 ? 3 : 4;
  constexpr int RBUF = KRP >= 128 ? 1 : 2;
  const size_t smem = 1024 + (size_t)STAGES * (kTile * 128 + 2 * kNf * 128) +
                      (size_t)RBUF * (2 * (KRP * kNf * 2) + KRP * 128) + 2 * (kTile * KRP * 2) + kTile * 128;
  static std::atomic<uint64_t> attr{0};
  if (const cudaError_t e = smem_attr_once(ffn_up_tc_kernel<KRP, STAGES, KE, RBUF>, smem, attr); e != cudaSuccess) return e;
  // one CTA per SM walks the (row tile, chunk) items (fewer CTAs when there are fewer items)
  int dev = 0, sms = 0;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
  if (cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev); e != cudaSuccess) return e;
  const int items = nchunks * tiles;
  return launch_pdl(ffn_up_tc_kernel<KRP, STAGES, KE, RBUF>, dim3(items < sms ? items : sms), dim3(kUpWarps * 32),
                    smem, stream, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p);
}

template <int KE>
static cudaError_t launch_up4p(const CUtensorMap* maps, const UpArgs& p, cudaStream_t stream) {
  const size_t smem = 1024 + (size_t)kStages4p * (kTile * 128 + kNf3 * 128) + 2 * (size_t)((kNf3 / 2) * 64 * 2) +
                      (size_t)kNf3 * 64 * 2 + 2 * (size_t)(kTile * 64 * 2);
  static std::atomic<uint64_t> attr{0};
  if (const cudaError_t e = smem_attr_once(ffn_up4p_kernel<KE>, smem, attr); e != cudaSuccess) return e;
  // the kernel's warpgroups trade registers on the assumption that it launches with
  // kUp4RegsLaunch per thread; with any other count the epilogue's increase could never be met
  static std::atomic<int> regs_checked{0};
  if (!regs_checked.load(std::memory_order_acquire)) {
    cudaFuncAttributes fa;
    if (const cudaError_t e = cudaFuncGetAttributes(&fa, ffn_up4p_kernel<KE>); e != cudaSuccess) return e;
    if (fa.numRegs != kUp4RegsLaunch) return cudaErrorInvalidConfiguration;
    regs_checked.store(1, std::memory_order_release);
  }
  // one cluster per pair of SMs that can hold one at once, walking the (pair tile, chunk) items
  // (fewer clusters when there are fewer items)
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  if (const cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
  int mc = dev >= 0 && dev < 64 ? max_clusters[dev].load(std::memory_order_acquire) : 0;
  if (mc <= 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kUpWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = 2; at.val.clusterDim.y = 1; at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    if (const cudaError_t e = cudaOccupancyMaxActiveClusters(&mc, ffn_up4p_kernel<KE>, &cfg); e != cudaSuccess) return e;
    if (mc <= 0) return cudaErrorInvalidConfiguration;
    if (dev >= 0 && dev < 64) max_clusters[dev].store(mc, std::memory_order_release);
  }
  const int items = p.n_row_tiles * p.n_chunks;
  const int clusters = items < mc ? items : mc;
  return launch_pdl_cluster(ffn_up4p_kernel<KE>, dim3(2 * clusters), dim3(kUpWarps * 32), dim3(2, 1, 1), smem,
                            stream, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p);
}

template <int KE>
static cudaError_t launch_up3(const CUtensorMap* maps, const UpArgs& p, int nchunks, int tiles, cudaStream_t stream) {
  const size_t smem = 1024 + (size_t)kStages3 * (kTile * 128 + 2 * kNf3 * 128) + 2 * (size_t)(kNf3 * 64 * 2) +
                      (size_t)64 * kNf3 * 2 + 2 * (size_t)(kTile * 64 * 2);
  static std::atomic<uint64_t> attr{0};
  if (const cudaError_t e = smem_attr_once(ffn_up3_kernel<KE>, smem, attr); e != cudaSuccess) return e;
  return launch_pdl(ffn_up3_kernel<KE>, dim3(nchunks, tiles), dim3(kUp3Warps * 32), smem, stream, maps[0], maps[1],
                    maps[2], maps[3], maps[4], maps[5], p);
}

template <int KRP>
static cudaError_t launch_up(const CUtensorMap* maps, const UpArgs& p, int nchunks, int tiles, cudaStream_t stream) {
  switch (p.ke) {
    case 1: return launch_up_ke<KRP, 1>(maps, p, nchunks, tiles, stream);
    case 2: return launch_up_ke<KRP, 2>(maps, p, nchunks, tiles, stream);
    case 3: return launch_up_ke<KRP, 3>(maps, p, nchunks, tiles, stream);
    default: return launch_up_ke<KRP, 4>(maps, p, nchunks, tiles, stream);
  }
}

// The double-buffered pair form (4c) hides its heavier epilogue (V on the CUDA cores) only behind
// long K loops over many rows; shorter ones run the single-buffered form (4b).
static bool up4_ok(const LayerArgs& a) { return up3_ok(a) && a.d >= 4096 && a.R >= 2048; }

static PrepArgs prep_args(const LayerArgs& a, const ResidPtrs& rp, const TcBufs& b) {
  PrepArgs pa;
  for (int m = 0; m < 3; ++m) { pa.A[m] = rp.A[m]; pa.B[m] = rp.B[m]; }
  pa.Ain = b.Ain; pa.Bgs = b.Bgs; pa.Bus = b.Bus; pa.Adn = b.Adn; pa.Bdn = b.Bdn;
  pa.G = a.G; pa.K = a.K; pa.d = a.d; pa.f = a.f; pa.r = a.r; pa.KRP = tc_krp(a);
  pa.need_ain = a.R > kUSimtMaxRows;             // the CUDA-core U kernel reads the codes itself
  const bool up4 = up4_ok(a);
  pa.adn_f16 = up3_ok(a) && !up4;
  pa.Adt = up4 ? b.Adt : nullptr;
  return pa;
}

bool tc_u_dense(const LayerArgs& a) {
  // the dense U runs beside the routing on the side stream: it pays while it is short next to
  // the routing (small workload, 8.6 GFLOP: 0.145 -> 0.137 ms per step); as long as the routing
  // (Mixtral shape, 34 GFLOP) it only competes with it for SMs, and the routed U after the
  // gather is 0.6% faster per step
  const double flops = 4.0 * a.T * a.G * 2 * tc_krp(a) * a.d;   // hi + lo stacks
  return tc_path_ok(a) && a.R > kUSimtMaxRows && a.G * 2 * tc_krp(a) <= 512 && flops <= 16e9;
}

// 1. residual stacks (weights only: may run on another stream, concurrently with the routing),
//    and, when tc_u_dense, U = A^T x of every token for every group (token order: it needs no
//    routing either) -- a dense GEMM of x against all groups' stacked A^T, which the gate/up
//    kernel then reads at (token, group)
cudaError_t launch_resid_prep(const LayerArgs& a, const ResidPtrs& rp, const TcBufs& b, const void* x,
                              DevStatus* status, cudaStream_t st, bool stacks) {
  if (a.R == 0 && stacks) return cudaSuccess;
  const PrepArgs pa = prep_args(a, rp, b);
  const int G = a.G, d = a.d, f = a.f, KRP = tc_krp(a);
  cudaError_t e = cudaSuccess;
  if (stacks) {
    launch_pdl(resid_prep_rows_kernel, dim3(148 * 4), dim3(256), 0, st, pa, a.tab);
    launch_pdl(resid_prep_t_kernel, dim3(G * (2 * (f / 64) + d / 64 + (pa.Adt ? f / 64 : 0))), dim3(256), 0, st, pa,
               a.tab);
    prof_mark("resid_prep", st);
    e = cudaGetLastError();
  }
  // the dense U GEMM needs the tokens: a call that only prepares the stacks (x == null) stops here
  if (e != cudaSuccess || !tc_u_dense(a) || a.T == 0 || x == nullptr || status == nullptr) return e;
  CUtensorMap mXt, mA;
  if (!make_map(&mXt, x, (uint64_t)a.T, d, kTile) || !make_map(&mA, b.Ain, (uint64_t)G * 4 * KRP, d, KRP))
    return cudaErrorInvalidValue;
  e = launch_gemm_pair<128, kOutF16>(mXt, mXt, mA, mA, d / 64, d / 64, nullptr, G, G * 2 * KRP, 4 * KRP, 2 * KRP,
                                     (a.T + 2 * kTile - 1) / (2 * kTile), b.Ud, G * 2 * KRP, nullptr, status, st,
                                     identity_slots(), a.T);
  prof_mark("u_gemm", st);
  return e;
}

cudaError_t launch_ffn_tc(const LayerArgs& a, const void* x, const void* wg, const void* wu, const void* wd,
                          const ResidPtrs& rp, const int32_t* eidx, const float* gate, const int32_t* row_asg,
                          const int32_t* row_begin, void* y_rows, const TcBufs& b, DevStatus* status,
                          cudaEvent_t prep_done, cudaStream_t st, bool prepared) {
  if (a.R == 0) return cudaSuccess;
  const int KRP = tc_krp(a), G = a.G, d = a.d, f = a.f, R = a.R;
  const int tiles = (R + kTile - 1) / kTile + G;
  cudaError_t e;

  // 1. residual stacks, unless already enqueued elsewhere (prep_done: recorded after them)
  const PrepArgs pa = prep_args(a, rp, b);
  const bool u_simt = R <= kUSimtMaxRows;
  const bool up3 = up3_ok(a), up4 = up4_ok(a);
  const bool u_dense = tc_u_dense(a);
  if (!prep_done && (e = launch_resid_prep(a, rp, b, x, status, st, !prepared)) != cudaSuccess) return e;

  // 2. rows of x in (group, token) order (the CUDA-core U kernel writes them itself)
  if (!u_simt) {
    launch_pdl(gather_rows_kernel, dim3(148 * 8), dim3(256), 0, st, (const __nv_bfloat16*)x, row_asg, R, d, a.kg,
               b.X);
    prof_mark("gather_rows", st);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }

  CUtensorMap mX, mAhi, mAlo, mWg, mWu, mBg, mBu, mAd, mH, mVt, mWd, mBd, mAdt;
  const uint64_t Rp = R < kTile ? kTile : R;   // row buffers hold at least one full tile
  // Ain is [G][2 (hi, lo)][2*KRP][d]: rows g*4*KRP + n (hi) and g*4*KRP + 2*KRP + n (lo)
  // pair GEMMs: each CTA of a pair holds half of the B tile
  const int pairs = (R + 2 * kTile - 1) / (2 * kTile) + G;
  const int nf_up = up3 ? kNf3 : kNf;
  // The pair form pays a cluster handshake per CTA; it gains on K loops of d_ff >= 2048 over many
  // rows (on shorter ones, or one-wave decode batches, the single-CTA form is faster).
  const bool down_pair = d % 256 == 0 && f >= 2048 && R >= 2048;
  bool ok = make_map(&mX, b.X, Rp, d, kTile) &&
            make_map(&mAhi, b.Ain, (uint64_t)G * 4 * KRP, d, KRP) &&
            make_map(&mWg, wg, (uint64_t)a.wslots * f, d, nf_up) && make_map(&mWu, wu, (uint64_t)a.wslots * f, d, nf_up) &&
            make_map(&mBg, b.Bgs, (uint64_t)G * f, KRP, nf_up) && make_map(&mBu, b.Bus, (uint64_t)G * f, KRP, nf_up) &&
            make_map(&mAd, b.Adn, (uint64_t)G * KRP, f, KRP) && make_map(&mH, b.hsum, Rp, f, kTile) &&
            make_map(&mVt, b.Vt, Rp, 2 * KRP, kTile);
  mAlo = mAhi;
  const int BN2 = down_pair ? 128 : (d % 256 == 0 ? 256 : 128);   // B box rows: half of N = 256 for pairs
  ok = ok && make_map(&mWd, wd, (uint64_t)a.wslots * d, f, BN2) && make_map(&mBd, b.Bdn, (uint64_t)G * d, 2 * KRP, BN2);
  if (up4) ok = ok && make_map_plain(&mAdt, b.Adt, (uint64_t)G * f, KRP, kNf3);
  if (!ok) return cudaErrorInvalidValue;

  // 3. U = X (Ain_hi + Ain_lo)^T (FP32 accumulation, FP16 out): the hi stack is at rows g*4*KRP, the lo stack 2*KRP later
  if (prep_done && !u_simt && !u_dense && (e = cudaStreamWaitEvent(st, prep_done, 0)) != cudaSuccess) return e;
  if (u_dense) {
    // U came with the residual stacks
  } else if (u_simt) {
    e = launch_pdl(u_simt_kernel, dim3(R, 2, (KRP + 31) / 32), dim3(256), (size_t)d * 2, st, (const __nv_bfloat16*)x,
                   row_asg, eidx, pa, a.tab, a.kg, a.ke, b.U, b.X);
    prof_mark("u_simt", st);
  } else {
    e = (2 * KRP == 256)
            ? launch_gemm_pair<256, kOutF16>(mX, mX, mAhi, mAlo, d / 64, d / 64, row_begin, G, 2 * KRP, 4 * KRP,
                                             2 * KRP, pairs, b.U, 2 * KRP, nullptr, status, st, identity_slots())
            : launch_gemm_pair<128, kOutF16>(mX, mX, mAhi, mAlo, d / 64, d / 64, row_begin, G, 2 * KRP, 4 * KRP,
                                             2 * KRP, pairs, b.U, 2 * KRP, nullptr, status, st, identity_slots());
    prof_mark("u_gemm", st);
  }
  if (e != cudaSuccess) return e;

  // 4. fused gate/up
  if (prep_done && (u_simt || u_dense) && (e = cudaStreamWaitEvent(st, prep_done, 0)) != cudaSuccess) return e;
  UpArgs p;
  p.row_begin = row_begin; p.row_asg = row_asg; p.eidx = eidx; p.gate = gate; p.hsum = b.hsum;
  p.U = u_dense ? b.Ud : b.U;
  p.u_by_token = u_dense ? 1 : 0;
  p.sAd = rp.A[2].scales;
  p.Vpart = b.Vpart; p.status = status; p.tab = a.tab; p.G = G; p.d = d; p.f = f; p.kg = a.kg; p.ke = a.ke;
  p.R = R; p.n_ftiles = f / nf_up;
  const int nchunks = tc_up_chunks(a);
  p.ftiles_per_chunk = (p.n_ftiles + nchunks - 1) / nchunks;
  p.n_row_tiles = up4 ? pairs : tiles;         // the pair kernel's items are 256-row pair tiles
  p.n_chunks = nchunks;
  if (up4) {
    CUtensorMap mBgP, mBuP;     // halves of the B_gate / B_up tiles (64 rows per CTA of a pair)
    if (!make_map(&mBgP, b.Bgs, (uint64_t)G * f, KRP, kNf3 / 2) || !make_map(&mBuP, b.Bus, (uint64_t)G * f, KRP, kNf3 / 2))
      return cudaErrorInvalidValue;
    const CUtensorMap mp[6] = {mX, mWg, mWu, mBgP, mBuP, mAdt};
    e = a.ke == 1 ? launch_up4p<1>(mp, p, st) : launch_up4p<2>(mp, p, st);
  } else {
    const CUtensorMap maps[6] = {mX, mWg, mWu, mBg, mBu, mAd};
    if (up3)
      e = a.ke == 1 ? launch_up3<1>(maps, p, nchunks, tiles, st) : launch_up3<2>(maps, p, nchunks, tiles, st);
    else
      e = KRP == 128 ? launch_up<128>(maps, p, nchunks, tiles, st) : launch_up<64>(maps, p, nchunks, tiles, st);
  }
  prof_mark("ffn_up_tc", st);
  if (e != cudaSuccess) return e;

  // 5. V~
  launch_pdl(v_reduce_kernel, dim3((R * (KRP / kRank) * 4 + 255) / 256), dim3(256), 0, st, (const float*)b.Vpart, row_asg,
             eidx, a.tab, R, a.kg, a.ke, up4 ? 2 * nchunks : nchunks, KRP, b.Vt);
  prof_mark("v_reduce", st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  // 6. Y = [hsum | V~] [Wd | Bdn]^T, rows to their token slot
  // the pair form runs its tiles in bands of kDownBand pair tiles across all d_model tiles
  constexpr int kDownBand = 8;
  // many waves of single-CTA tiles: the persistent form overlaps each tile's epilogue with the
  // next tile's K loop
  const bool down_persist = !down_pair && BN2 == 256 && tiles * (d / 256) > 2 * 148;
  SlotMap wd_slots;                              // W_down rows of group g start at wslot[g] * d
  for (int i = 0; i < kMaxE; ++i) wd_slots.s[i] = a.tab.wslot[i];
  e = down_pair ? launch_gemm_pair<256, kOutBf16>(mH, mVt, mWd, mBd, f / 64, 2 * KRP / 64, row_begin, G, d, d, 0,
                                                  pairs, y_rows, d, row_asg, status, st, wd_slots, 0, kDownBand)
      : down_persist ? launch_gemm_persist<256, kOutBf16>(mH, mVt, mWd, mBd, f / 64, 2 * KRP / 64, row_begin, G, d,
                                                          d, 0, tiles, y_rows, d, row_asg, status, st, wd_slots)
                : (BN2 == 256 ? launch_gemm<256, kOutBf16>(mH, mVt, mWd, mBd, f / 64, 2 * KRP / 64, row_begin, G, d,
                                                           d, 0, tiles, y_rows, d, row_asg, status, st, wd_slots)
                              : launch_gemm<128, kOutBf16>(mH, mVt, mWd, mBd, f / 64, 2 * KRP / 64, row_begin, G, d,
                                                           d, 0, tiles, y_rows, d, row_asg, status, st, wd_slots));
  prof_mark("ffn_down_tc", st);
  return e;
}

}  // namespace moe
