// Expert computation on the tcgen05 tensor cores (BF16 layers, INT4 group-64 residual).
//
// "Breaking the MoE LLM Trilemma: Dynamic Expert Clustering with Structured Compression"
// (paper notes), key design 2: W~_i = W_base^g + B_i A_i^T and W~_i x = W_base^g x + B_i (A_i^T x),
// the base product computed once for all of a group's experts on the same tokens.  Key design 4:
// BF16/FP16 base, INT4 residual.  Expert body: SwiGLU ("混合专家模型的路由机制与工程落地" 1.2).
//
// Rows are (token, group) pairs in (group, token) order; each row carries k_e experts.
//   1. resid_prep   BF16 stacks of the group's K experts, KRP = K*r padded to 64, holding the
//                   dequantised values exactly: A_gate^T/A_up^T as hi+lo BF16 pairs
//                   (Ain [G][2][2*KRP][d]), B_gate/B_up and A_down^T as their integer codes
//                   (Bgs/Bus [G][f][KRP], Adn [G][KRP][f]; the FP16 scale, constant over a
//                   64-column tile, is applied on the other side of the product), B_down as a
//                   hi|lo pair along K (Bdn [G][d][2*KRP]).
//   2. gather_rows  X[i] = x[token(i)] (BF16 rows in (group, token) order).
//   3. U GEMM       U[i] = X[i] (Ain_hi + Ain_lo)_g^T, FP32: A^T x for every expert of the group.
//   4. ffn_up       per 128-row x 64-column tile of group g: base [Hg|Hu] = X [Wg|Wu]^T once;
//                   per expert slot s: R_s = U~_s [Bgs|Bus]^T (U~_s = the row's slot-s block of U
//                   times the tile's B scales, other blocks zero), h_s = silu(Hg + R_gate) *
//                   (Hu + R_up), hsum += gate_s h_s, and v_s += A_down,e_s^T h_s via
//                   V = h_s Adn_g^T times the tile's A_down scales (tcgen05).
//   5. v_reduce     sums the v partials of the column chunks into V~ [R][2*KRP] (gate-scaled,
//                   block of each slot's expert, repeated for the hi and lo halves of Bdn).
//   6. down GEMM    Y[i] = [hsum | V~][i] [Wd_g | Bdn_g]^T, written to the row's token slot.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int kTile = 128;      // rows per tile (MMA M)
constexpr int kNf = 64;         // d_ff columns per gate/up tile
constexpr int kEpiThreads = 128;

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
struct PrepArgs {
  ResidView A[3], B[3];
  __nv_bfloat16 *Ain, *Bgs, *Bus, *Adn, *Bdn;
  int G, K, d, f, r, KRP;
};

// Integer code (u - 8) of element c of rank row k of expert e (INT4 group-64 format).
__device__ __forceinline__ float code_at(const ResidView& v, int e, int k, int c) {
  const uint8_t b = ((const uint8_t*)v.vals)[((size_t)e * v.r + k) * (v.n / 2) + (c >> 1)];
  return (float)(((c & 1) ? (b & 0xF) : (b >> 4)) - 8);
}

// Every output element written exactly once per launch.  Row-major outputs: 8 consecutive
// elements per work item; transposed outputs: one KRP-wide row per work item.
__global__ void resid_prep_kernel(PrepArgs p, GroupTable tab) {
  const int G = p.G, K = p.K, r = p.r, KRP = p.KRP, d = p.d, f = p.f;
  const size_t nAin = (size_t)G * 2 * KRP * (d / 8);   // hi/lo pairs written together
  const size_t nAdn = (size_t)G * KRP * (f / 8);
  const size_t nBg = (size_t)G * f;
  const size_t nBd = (size_t)G * d;
  const size_t total = nAin + nAdn + 2 * nBg + nBd;
  for (size_t w = blockIdx.x * (size_t)blockDim.x + threadIdx.x; w < total; w += (size_t)gridDim.x * blockDim.x) {
    if (w < nAin) {
      // Ain[g][0][m*KRP + j*r + k][c] = hi, Ain[g][1][...] = lo of A_m,e_j^T[k][c]
      const int c8 = (int)(w % (d / 8)) * 8;
      const size_t rowg = w / (d / 8);
      const int g = (int)(rowg / (2 * KRP)), row = (int)(rowg % (2 * KRP));
      const int m = row / KRP, jk = row % KRP, j = jk / r, k = jk % r;
      uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
      if (j < K) {
        const int e = tab.member[g * K + j];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float v0 = p.A[m].at(e, k, c8 + 2 * q), v1 = p.A[m].at(e, k, c8 + 2 * q + 1);
          const __nv_bfloat16 h0 = __float2bfloat16_rn(v0), h1 = __float2bfloat16_rn(v1);
          hi[q] = tc::pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
          lo[q] = tc::pack_bf16(v0 - __bfloat162float(h0), v1 - __bfloat162float(h1));
        }
      }
      __nv_bfloat16* dst = p.Ain + ((size_t)g * 2 * (2 * KRP) + row) * d + c8;
      *reinterpret_cast<uint4*>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(dst + (size_t)2 * KRP * d) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    } else if (w < nAin + nAdn) {
      // Adn[g][j*r + k][c] = code of A_down,e_j^T[k][c]
      const size_t idx = w - nAin;
      const int c8 = (int)(idx % (f / 8)) * 8;
      const size_t rowg = idx / (f / 8);
      const int g = (int)(rowg / KRP), jk = (int)(rowg % KRP), j = jk / r, k = jk % r;
      uint32_t out[4] = {0u, 0u, 0u, 0u};
      if (j < K) {
        const int e = tab.member[g * K + j];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          out[q] = tc::pack_bf16(code_at(p.A[2], e, k, c8 + 2 * q), code_at(p.A[2], e, k, c8 + 2 * q + 1));
      }
      *reinterpret_cast<uint4*>(p.Adn + rowg * f + c8) = make_uint4(out[0], out[1], out[2], out[3]);
    } else {
      size_t idx = w - nAin - nAdn;
      int m, n, width;
      __nv_bfloat16* base;
      if (idx < nBg) { m = 0; n = f; base = p.Bgs; width = KRP; }
      else if (idx < 2 * nBg) { idx -= nBg; m = 1; n = f; base = p.Bus; width = KRP; }
      else { idx -= 2 * nBg; m = 2; n = d; base = p.Bdn; width = 2 * KRP; }
      const int g = (int)(idx / n), c = (int)(idx % n);
      const ResidView& v = p.B[m];
      __nv_bfloat16* dst = base + idx * width;
      for (int jk0 = 0; jk0 < KRP; jk0 += 8) {
        uint32_t out[4], lo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float t2[2], l2[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int jk = jk0 + 2 * q + h, j = jk / r, k = jk % r;
            if (j >= K) { t2[h] = 0.f; l2[h] = 0.f; continue; }
            const int e = tab.member[g * K + j];
            if (m < 2) {            // B_gate / B_up: integer code, scale folded into U~
              t2[h] = code_at(v, e, k, c);
              l2[h] = 0.f;
            } else {                // B_down: exact value as hi + lo
              const float val = v.at(e, k, c);
              t2[h] = __bfloat162float(__float2bfloat16_rn(val));
              l2[h] = val - t2[h];
            }
          }
          out[q] = tc::pack_bf16(t2[0], t2[1]);
          lo[q] = tc::pack_bf16(l2[0], l2[1]);
        }
        *reinterpret_cast<uint4*>(dst + jk0) = make_uint4(out[0], out[1], out[2], out[3]);
        if (m == 2) *reinterpret_cast<uint4*>(dst + KRP + jk0) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
  }
}

// ------------------------------------------------------------------------------------------
// 2. X rows in (group, token) order
// ------------------------------------------------------------------------------------------
__global__ void gather_rows_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ row_asg,
                                   int R, int d, int kg, __nv_bfloat16* __restrict__ X) {
  const int per_row = d / 8;
  const size_t n = (size_t)R * per_row;
  for (size_t w = blockIdx.x * (size_t)blockDim.x + threadIdx.x; w < n; w += (size_t)gridDim.x * blockDim.x) {
    const int i = (int)(w / per_row), c = (int)(w % per_row) * 8;
    const int t = row_asg[i] / kg;
    *reinterpret_cast<uint4*>(X + (size_t)i * d + c) = *reinterpret_cast<const uint4*>(x + (size_t)t * d + c);
  }
}

// ------------------------------------------------------------------------------------------
// 3/6. Generic grouped GEMM: out[row] = [A0 | A1][i] [B0_g | B1_g]^T (BF16 in, FP32 acc, BF16 or
//      FP32 out).  Group g's B rows start at g*b_stride in B0 and at g*b_stride + b1_off in B1.
// ------------------------------------------------------------------------------------------
template <int BN, int STAGES, bool OUT_F32>
__global__ void __launch_bounds__(192, 1) tc_gemm_kernel(
    const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
    const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1, int nk0, int nk1,
    const int32_t* __restrict__ row_begin, int G, int b_stride, int b1_off, void* __restrict__ out, int out_ld,
    const int32_t* __restrict__ scatter, DevStatus* status) {
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
      tc::tma_load_2d(sB + s * B_BYTES, first ? &mB0 : &mB1, &full[s], kx, g * b_stride + (first ? 0 : b1_off) + n0);
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
          if constexpr (OUT_F32) {
            uint4* d4 = reinterpret_cast<uint4*>((float*)out + orow * out_ld + n0 + c);
#pragma unroll
            for (int e = 0; e < 4; ++e) d4[e] = make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
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
// 4. Fused gate/up tile: base once, per-slot residual, SwiGLU, gated sum, down-residual partials
// ------------------------------------------------------------------------------------------
constexpr int kMaxKe = 4;
constexpr int kRank = 16;      // residual rank handled by this kernel

struct UpArgs {
  const int32_t* row_begin;
  const int32_t* row_asg;
  const int32_t* eidx;
  const float* gate;
  const float* U;           // [R][2*KRP]: A_gate^T x | A_up^T x of the group's experts
  const __half *sBg, *sBu, *sAd;   // FP16 scales [E][16][f/64] of B_gate, B_up, A_down^T
  __nv_bfloat16* hsum;      // [R][f]
  float* Vpart;             // [nchunks][R][ke][16]
  DevStatus* status;
  GroupTable tab;
  int G, d, f, kg, ke, R, n_ftiles, ftiles_per_chunk;
};

template <int KRP, int STAGES>
__global__ void __launch_bounds__(192, 1) ffn_up_tc_kernel(
    const __grid_constant__ CUtensorMap mX, const __grid_constant__ CUtensorMap mWg,
    const __grid_constant__ CUtensorMap mWu, const __grid_constant__ CUtensorMap mBg,
    const __grid_constant__ CUtensorMap mBu, const __grid_constant__ CUtensorMap mAd, const UpArgs p) {
  constexpr uint32_t X_BYTES = kTile * 128, W_BYTES = 2 * kNf * 128, STAGE_BYTES = X_BYTES + W_BYTES;
  constexpr uint32_t BRES_BYTES = KRP * kNf * 2;          // one of Bg / Bu tiles (64 rows x KRP)
  constexpr uint32_t AD_BYTES = KRP * 128;                 // KRP rows x 64 columns
  constexpr uint32_t UT_BYTES = kTile * KRP * 2;           // 128 rows x KRP
  constexpr uint32_t H_BYTES = kTile * 128;                // 128 rows x 64 columns
  constexpr int KATOM = KRP / 64;
  constexpr uint32_t COL_BASE = 0, COL_R = 2 * kNf, COL_V = 4 * kNf;
  static_assert(COL_V + KRP <= 512, "TMEM budget");

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[STAGES], empty[STAGES];
  __shared__ uint64_t res_full, res_empty, acc_empty, u_ready, r_full, h_ready, v_full, fin;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  int g, r0, r1;
  if (!tile_of(p.row_begin, p.G, blockIdx.y, g, r0, r1)) return;
  const int ft0 = blockIdx.x * p.ftiles_per_chunk;
  const int ft1 = min(ft0 + p.ftiles_per_chunk, p.n_ftiles);
  if (ft0 >= ft1) return;
  const int nft = ft1 - ft0;
  const int nkb = p.d / 64;

  uint8_t* smem = align1024(smem_raw);
  uint8_t* sStage = smem;
  uint8_t* sBg = sStage + STAGES * STAGE_BYTES;
  uint8_t* sBu = sBg + BRES_BYTES;
  uint8_t* sAd = sBu + BRES_BYTES;
  uint8_t* sUg = sAd + AD_BYTES;
  uint8_t* sUu = sUg + UT_BYTES;
  uint8_t* sH = sUu + UT_BYTES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tc::Abort ab{&abort_flag, p.status};
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { tc::bar_init(&full[s], 1); tc::bar_init(&empty[s], 1); }
    tc::bar_init(&res_full, 1);
    tc::bar_init(&res_empty, 1);
    tc::bar_init(&acc_empty, kEpiThreads);
    tc::bar_init(&u_ready, kEpiThreads);
    tc::bar_init(&r_full, 1);
    tc::bar_init(&h_ready, kEpiThreads);
    tc::bar_init(&v_full, 1);
    tc::bar_init(&fin, 1);
    abort_flag = 0;
    tc::bar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, 512);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_base;
  const int ke = p.ke, f = p.f;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer: per f-tile the d/64 stages, then the residual tiles
    tc::prefetch_map(&mX); tc::prefetch_map(&mWg); tc::prefetch_map(&mWu);
    tc::prefetch_map(&mBg); tc::prefetch_map(&mBu); tc::prefetch_map(&mAd);
    int kc = 0;
    bool ok = true;
    for (int lt = 0; lt < nft && ok; ++lt) {
      const int n0 = (ft0 + lt) * kNf;
      for (int kb = 0; kb < nkb; ++kb, ++kc) {
        const int s = kc % STAGES, it = kc / STAGES;
        if (kc >= STAGES && !tc::bar_wait(&empty[s], (it - 1) & 1, ab, 11)) { ok = false; break; }
        uint8_t* st = sStage + s * STAGE_BYTES;
        tc::bar_expect_tx(&full[s], STAGE_BYTES);
        tc::tma_load_2d(st, &mX, &full[s], kb * 64, r0);
        tc::tma_load_2d(st + X_BYTES, &mWg, &full[s], kb * 64, g * f + n0);
        tc::tma_load_2d(st + X_BYTES + kNf * 128, &mWu, &full[s], kb * 64, g * f + n0);
      }
      if (!ok) break;
      if (lt > 0 && !tc::bar_wait(&res_empty, (lt - 1) & 1, ab, 12)) break;
      tc::bar_expect_tx(&res_full, 2 * BRES_BYTES + AD_BYTES);
#pragma unroll
      for (int a = 0; a < KATOM; ++a) {
        tc::tma_load_2d(sBg + a * kNf * 128, &mBg, &res_full, a * 64, g * f + n0);
        tc::tma_load_2d(sBu + a * kNf * 128, &mBu, &res_full, a * 64, g * f + n0);
      }
      tc::tma_load_2d(sAd, &mAd, &res_full, n0, g * KRP);
    }
    if (abort_flag) tc::drain_copies();
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t id_base = tc::idesc_bf16(kTile, 2 * kNf);
    constexpr uint32_t id_res = tc::idesc_bf16(kTile, kNf);
    constexpr uint32_t id_v = tc::idesc_bf16(kTile, KRP);
    int kc = 0, pu = 0, ph = 0;
    bool ok = true;
    for (int lt = 0; lt < nft && ok; ++lt) {
      if (lt > 0 && !tc::bar_wait(&acc_empty, (lt - 1) & 1, ab, 21)) break;
      tc::fence_after();
      for (int kb = 0; kb < nkb; ++kb, ++kc) {
        const int s = kc % STAGES, it = kc / STAGES;
        if (!tc::bar_wait(&full[s], it & 1, ab, 22)) { ok = false; break; }
        tc::fence_after();
        const uint32_t a0 = tc::smem_u32(sStage + s * STAGE_BYTES);
        const uint32_t b0 = a0 + X_BYTES;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_bf16(tmem + COL_BASE, tc::sdesc(a0 + 32 * k), tc::sdesc(b0 + 32 * k), id_base, (kb | k) != 0);
        tc::mma_commit(&empty[s]);
      }
      if (!ok) break;
      if (!tc::bar_wait(&res_full, lt & 1, ab, 23)) break;
      tc::fence_after();
      const uint32_t ug = tc::smem_u32(sUg), uu = tc::smem_u32(sUu);
      const uint32_t bg = tc::smem_u32(sBg), bu = tc::smem_u32(sBu);
      const uint32_t hh = tc::smem_u32(sH), ad = tc::smem_u32(sAd);
      for (int s = 0; s < ke && ok; ++s) {
        if (!tc::bar_wait(&u_ready, pu & 1, ab, 24)) { ok = false; break; }
        ++pu;
        tc::fence_after();
#pragma unroll
        for (int kk = 0; kk < KRP / 16; ++kk) {
          const uint32_t off_u = (kk >> 2) * (kTile * 128) + (kk & 3) * 32;
          const uint32_t off_b = (kk >> 2) * (kNf * 128) + (kk & 3) * 32;
          tc::mma_bf16(tmem + COL_R, tc::sdesc(ug + off_u), tc::sdesc(bg + off_b), id_res, kk != 0);
          tc::mma_bf16(tmem + COL_R + kNf, tc::sdesc(uu + off_u), tc::sdesc(bu + off_b), id_res, kk != 0);
        }
        tc::mma_commit(&r_full);
        if (!tc::bar_wait(&h_ready, ph & 1, ab, 25)) { ok = false; break; }
        ++ph;
        tc::fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tmem + COL_V, tc::sdesc(hh + 32 * kk), tc::sdesc(ad + 32 * kk), id_v, kk != 0);
        tc::mma_commit(&v_full);
      }
      tc::mma_commit(&res_empty);
    }
    tc::mma_commit(&fin);
    const uint64_t t0 = tc::now_ns();
    while (!tc::bar_test(&fin, 0) && tc::now_ns() - t0 < tc::kWaitNs) {}
  } else if (warp >= 2) {
    // ---------------- epilogue: one thread per tile row
    const int q = warp & 3, row = q * 32 + lane, i = r0 + row;
    const bool valid = i < r1;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    int le[kMaxKe];
    float gt[kMaxKe];
    const float* urow = nullptr;
    int eid[kMaxKe];
    for (int s = 0; s < kMaxKe; ++s) eid[s] = 0;
    for (int s = 0; s < kMaxKe; ++s) { le[s] = 0; gt[s] = 0.f; }
    if (valid) {
      const int b = p.row_asg[i], t = b / p.kg, j = b % p.kg, k = p.kg * ke;
      for (int s = 0; s < ke; ++s) {
        const int e = p.eidx[(size_t)t * k + j * ke + s];
        le[s] = p.tab.local_of[e];
        eid[s] = e;
        gt[s] = p.gate[(size_t)t * k + j * ke + s];
      }
      urow = p.U + (size_t)i * 2 * KRP;
    }
    // zero this row of U~gate / U~up
    for (int a = 0; a < KATOM; ++a) {
      uint4* zg = reinterpret_cast<uint4*>(sUg + a * kTile * 128 + (row >> 3) * 1024 + (row & 7) * 128);
      uint4* zu = reinterpret_cast<uint4*>(sUu + a * kTile * 128 + (row >> 3) * 1024 + (row & 7) * 128);
#pragma unroll
      for (int c = 0; c < 8; ++c) { zg[c] = make_uint4(0, 0, 0, 0); zu[c] = make_uint4(0, 0, 0, 0); }
    }
    float vacc[kMaxKe][kRank];
#pragma unroll
    for (int s = 0; s < kMaxKe; ++s)
#pragma unroll
      for (int k = 0; k < kRank; ++k) vacc[s][k] = 0.f;
    int pr = 0, pv = 0, cur = -1;
    bool ok = true;
    for (int lt = 0; lt < nft && ok; ++lt) {
      const int n0 = (ft0 + lt) * kNf;
      float hs[kNf];
#pragma unroll
      for (int c = 0; c < kNf; ++c) hs[c] = 0.f;
      for (int s = 0; s < ke; ++s) {
        // U~ for slot s: this row's block le[s] holds A^T x of expert e_s times the B scales of
        // this 64-column tile (one scale group), every other block 0
        if (valid) {
          const uint4 zero = make_uint4(0, 0, 0, 0);
          if (cur >= 0 && cur != le[s]) {
            *reinterpret_cast<uint4*>(sUg + tc::sw128_offset(row, cur * kRank, kTile)) = zero;
            *reinterpret_cast<uint4*>(sUg + tc::sw128_offset(row, cur * kRank + 8, kTile)) = zero;
            *reinterpret_cast<uint4*>(sUu + tc::sw128_offset(row, cur * kRank, kTile)) = zero;
            *reinterpret_cast<uint4*>(sUu + tc::sw128_offset(row, cur * kRank + 8, kTile)) = zero;
          }
          const float* ug = urow + le[s] * kRank;
          const float* uu = urow + KRP + le[s] * kRank;
          const size_t sc0 = (size_t)eid[s] * kRank * (f / 64) + n0 / 64;
          uint32_t pg[8], pu_[8];
#pragma unroll
          for (int k2 = 0; k2 < kRank; k2 += 2) {
            const float g0 = ug[k2] * __half2float(p.sBg[sc0 + (size_t)k2 * (f / 64)]);
            const float g1 = ug[k2 + 1] * __half2float(p.sBg[sc0 + (size_t)(k2 + 1) * (f / 64)]);
            const float u0 = uu[k2] * __half2float(p.sBu[sc0 + (size_t)k2 * (f / 64)]);
            const float u1 = uu[k2 + 1] * __half2float(p.sBu[sc0 + (size_t)(k2 + 1) * (f / 64)]);
            pg[k2 / 2] = tc::pack_bf16(g0, g1);
            pu_[k2 / 2] = tc::pack_bf16(u0, u1);
          }
          *reinterpret_cast<uint4*>(sUg + tc::sw128_offset(row, le[s] * kRank, kTile)) = make_uint4(pg[0], pg[1], pg[2], pg[3]);
          *reinterpret_cast<uint4*>(sUg + tc::sw128_offset(row, le[s] * kRank + 8, kTile)) = make_uint4(pg[4], pg[5], pg[6], pg[7]);
          *reinterpret_cast<uint4*>(sUu + tc::sw128_offset(row, le[s] * kRank, kTile)) = make_uint4(pu_[0], pu_[1], pu_[2], pu_[3]);
          *reinterpret_cast<uint4*>(sUu + tc::sw128_offset(row, le[s] * kRank + 8, kTile)) = make_uint4(pu_[4], pu_[5], pu_[6], pu_[7]);
          cur = le[s];
        }
        tc::fence_async_smem();
        tc::bar_arrive(&u_ready);
        if (!tc::bar_wait(&r_full, pr & 1, ab, 31)) { ok = false; break; }
        ++pr;
        tc::fence_after();
#pragma unroll
        for (int c = 0; c < kNf; c += 16) {
          uint32_t bgv[16], buv[16], rgv[16], ruv[16];
          tc::tmem_ld16(tmem + lane_off + COL_BASE + c, bgv);
          tc::tmem_ld16(tmem + lane_off + COL_BASE + kNf + c, buv);
          tc::tmem_ld16(tmem + lane_off + COL_R + c, rgv);
          tc::tmem_ld16(tmem + lane_off + COL_R + kNf + c, ruv);
          tc::tmem_ld_wait();
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float h2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const float a = __uint_as_float(bgv[e + u]) + __uint_as_float(rgv[e + u]);
              const float bb = __uint_as_float(buv[e + u]) + __uint_as_float(ruv[e + u]);
              h2[u] = silu_f(a) * bb;
              hs[c + e + u] += gt[s] * h2[u];
            }
            pk[e / 2] = tc::pack_bf16(h2[0], h2[1]);
          }
          *reinterpret_cast<uint4*>(sH + tc::sw128_offset(row, c, kTile)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(sH + tc::sw128_offset(row, c + 8, kTile)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
        tc::fence_before();
        tc::fence_async_smem();
        tc::bar_arrive(&h_ready);
        if (!tc::bar_wait(&v_full, pv & 1, ab, 32)) { ok = false; break; }
        ++pv;
        tc::fence_after();
#pragma unroll
        for (int jb = 0; jb < KRP / 16; ++jb) {
          uint32_t vv[16];
          tc::tmem_ld16(tmem + lane_off + COL_V + jb * 16, vv);
          tc::tmem_ld_wait();
          if (jb == le[s] && valid) {
            const size_t sc0 = (size_t)eid[s] * kRank * (f / 64) + n0 / 64;
#pragma unroll
            for (int k = 0; k < kRank; ++k) {
              const float val = __uint_as_float(vv[k]) * __half2float(p.sAd[sc0 + (size_t)k * (f / 64)]);
#pragma unroll
              for (int s2 = 0; s2 < kMaxKe; ++s2)
                if (s2 == s) vacc[s2][k] += val;
            }
          }
        }
      }
      if (!ok) break;
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(p.hsum + (size_t)i * f + n0);
#pragma unroll
        for (int c = 0; c < kNf; c += 8)
          dst[c / 8] = make_uint4(tc::pack_bf16(hs[c], hs[c + 1]), tc::pack_bf16(hs[c + 2], hs[c + 3]),
                                  tc::pack_bf16(hs[c + 4], hs[c + 5]), tc::pack_bf16(hs[c + 6], hs[c + 7]));
      }
      tc::fence_before();
      tc::bar_arrive(&acc_empty);
    }
    if (ok && valid) {
      float* vp = p.Vpart + ((size_t)blockIdx.x * p.R + i) * ke * kRank;
#pragma unroll
      for (int s = 0; s < kMaxKe; ++s)
        if (s < ke)
#pragma unroll
          for (int k = 0; k < kRank; ++k) vp[s * kRank + k] = gt[s] * vacc[s][k];
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
// 5. V~[i][j*16 + k] = sum over column chunks of the gated v of the slot whose expert is local j
// ------------------------------------------------------------------------------------------
__global__ void v_reduce_kernel(const float* __restrict__ Vpart, const int32_t* __restrict__ row_asg,
                                const int32_t* __restrict__ eidx, GroupTable tab, int R, int kg, int ke,
                                int nchunks, int KRP, __nv_bfloat16* __restrict__ Vt) {
  const size_t n = (size_t)R * KRP;
  for (size_t w = blockIdx.x * (size_t)blockDim.x + threadIdx.x; w < n; w += (size_t)gridDim.x * blockDim.x) {
    const int i = (int)(w / KRP), col = (int)(w % KRP), jl = col / kRank, k = col % kRank;
    const int b = row_asg[i], t = b / kg, j = b % kg;
    float acc = 0.f;
    for (int s = 0; s < ke; ++s) {
      const int e = eidx[(size_t)t * kg * ke + j * ke + s];
      if (tab.local_of[e] != jl) continue;
      for (int c = 0; c < nchunks; ++c) acc += Vpart[(((size_t)c * R + i) * ke + s) * kRank + k];
    }
    const __nv_bfloat16 v = __float2bfloat16_rn(acc);
    Vt[(size_t)i * 2 * KRP + col] = v;          // multiplies the hi half of Bdn
    Vt[(size_t)i * 2 * KRP + KRP + col] = v;    // and the lo half
  }
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

template <typename K>
static cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

bool tc_path_ok(const LayerArgs& a) {
  const int KRP = ((a.K * a.r + 63) / 64) * 64;
  return a.bf16 && a.int4 && a.r == kRank && a.K * a.r <= 128 && KRP <= 128 && a.ke <= kMaxKe &&
         a.d % 128 == 0 && a.f % 64 == 0;
}

int tc_krp(const LayerArgs& a) { return ((a.K * a.r + 63) / 64) * 64; }

int tc_up_chunks(const LayerArgs& a) {
  const int n_ft = a.f / kNf;
  const int tiles = (a.R + kTile - 1) / kTile + 1;
  int want = (2 * 148 + tiles - 1) / tiles;
  if (want < 1) want = 1;
  if (want > n_ft) want = n_ft;
  const int per = (n_ft + want - 1) / want;
  return (n_ft + per - 1) / per;
}

template <int BN, bool OUT_F32>
static cudaError_t launch_gemm(const CUtensorMap& A0, const CUtensorMap& A1, const CUtensorMap& B0,
                               const CUtensorMap& B1, int nk0, int nk1, const int32_t* row_begin, int G,
                               int n_out, int b_stride, int b1_off, int tiles, void* out, int out_ld,
                               const int32_t* scatter, DevStatus* st, cudaStream_t stream) {
  constexpr int STAGES = BN >= 256 ? 4 : 6;
  const size_t smem = 1024 + (size_t)STAGES * (kTile * 128 + BN * 128);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(tc_gemm_kernel<BN, STAGES, OUT_F32>, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(n_out / BN, tiles);
  tc_gemm_kernel<BN, STAGES, OUT_F32><<<grid, 192, smem, stream>>>(A0, A1, B0, B1, nk0, nk1, row_begin, G,
                                                                  b_stride, b1_off, out, out_ld, scatter, st);
  return cudaGetLastError();
}

template <int KRP>
static cudaError_t launch_up(const CUtensorMap* maps, const UpArgs& p, int nchunks, int tiles, cudaStream_t stream) {
  constexpr int STAGES = KRP >= 128 ? 3 : 4;
  const size_t smem = 1024 + (size_t)STAGES * (kTile * 128 + 2 * kNf * 128) + 2 * (KRP * kNf * 2) + KRP * 128 +
                      2 * (kTile * KRP * 2) + kTile * 128;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(ffn_up_tc_kernel<KRP, STAGES>, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(nchunks, tiles);
  ffn_up_tc_kernel<KRP, STAGES><<<grid, 192, smem, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p);
  return cudaGetLastError();
}

cudaError_t launch_ffn_tc(const LayerArgs& a, const void* x, const void* wg, const void* wu, const void* wd,
                          const ResidPtrs& rp, const int32_t* eidx, const float* gate, const int32_t* row_asg,
                          const int32_t* row_begin, void* y_rows, const TcBufs& b, DevStatus* status,
                          cudaStream_t st) {
  if (a.R == 0) return cudaSuccess;
  const int KRP = tc_krp(a), G = a.G, d = a.d, f = a.f, R = a.R;
  const int tiles = (R + kTile - 1) / kTile + G;
  cudaError_t e;

  // 1. residual stacks
  PrepArgs pa;
  for (int m = 0; m < 3; ++m) { pa.A[m] = rp.A[m]; pa.B[m] = rp.B[m]; }
  pa.Ain = b.Ain; pa.Bgs = b.Bgs; pa.Bus = b.Bus; pa.Adn = b.Adn; pa.Bdn = b.Bdn;
  pa.G = G; pa.K = a.K; pa.d = d; pa.f = f; pa.r = a.r; pa.KRP = KRP;
  resid_prep_kernel<<<148 * 8, 256, 0, st>>>(pa, a.tab);
  prof_mark("resid_prep", st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  // 2. rows of x in (group, token) order
  gather_rows_kernel<<<148 * 8, 256, 0, st>>>((const __nv_bfloat16*)x, row_asg, R, d, a.kg, b.X);
  prof_mark("gather_rows", st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  CUtensorMap mX, mAhi, mAlo, mWg, mWu, mBg, mBu, mAd, mH, mVt, mWd, mBd;
  const uint64_t Rp = R < kTile ? kTile : R;   // row buffers hold at least one full tile
  // Ain is [G][2 (hi, lo)][2*KRP][d]: rows g*4*KRP + n (hi) and g*4*KRP + 2*KRP + n (lo)
  bool ok = make_map(&mX, b.X, Rp, d, kTile) &&
            make_map(&mAhi, b.Ain, (uint64_t)G * 4 * KRP, d, 2 * KRP) &&
            make_map(&mWg, wg, (uint64_t)G * f, d, kNf) && make_map(&mWu, wu, (uint64_t)G * f, d, kNf) &&
            make_map(&mBg, b.Bgs, (uint64_t)G * f, KRP, kNf) && make_map(&mBu, b.Bus, (uint64_t)G * f, KRP, kNf) &&
            make_map(&mAd, b.Adn, (uint64_t)G * KRP, f, KRP) && make_map(&mH, b.hsum, Rp, f, kTile) &&
            make_map(&mVt, b.Vt, Rp, 2 * KRP, kTile);
  mAlo = mAhi;
  const int BN2 = d % 256 == 0 ? 256 : 128;
  ok = ok && make_map(&mWd, wd, (uint64_t)G * d, f, BN2) && make_map(&mBd, b.Bdn, (uint64_t)G * d, 2 * KRP, BN2);
  if (!ok) return cudaErrorInvalidValue;

  // 3. U = X (Ain_hi + Ain_lo)^T in FP32: the hi stack is at rows g*4*KRP, the lo stack 2*KRP later
  e = (2 * KRP == 256)
          ? launch_gemm<256, true>(mX, mX, mAhi, mAlo, d / 64, d / 64, row_begin, G, 2 * KRP, 4 * KRP, 2 * KRP,
                                   tiles, b.U, 2 * KRP, nullptr, status, st)
          : launch_gemm<128, true>(mX, mX, mAhi, mAlo, d / 64, d / 64, row_begin, G, 2 * KRP, 4 * KRP, 2 * KRP,
                                   tiles, b.U, 2 * KRP, nullptr, status, st);
  prof_mark("u_gemm", st);
  if (e != cudaSuccess) return e;

  // 4. fused gate/up
  UpArgs p;
  p.row_begin = row_begin; p.row_asg = row_asg; p.eidx = eidx; p.gate = gate; p.U = b.U; p.hsum = b.hsum;
  p.sBg = rp.B[0].scales; p.sBu = rp.B[1].scales; p.sAd = rp.A[2].scales;
  p.Vpart = b.Vpart; p.status = status; p.tab = a.tab; p.G = G; p.d = d; p.f = f; p.kg = a.kg; p.ke = a.ke;
  p.R = R; p.n_ftiles = f / kNf;
  const int nchunks = tc_up_chunks(a);
  p.ftiles_per_chunk = (p.n_ftiles + nchunks - 1) / nchunks;
  const CUtensorMap maps[6] = {mX, mWg, mWu, mBg, mBu, mAd};
  e = KRP == 128 ? launch_up<128>(maps, p, nchunks, tiles, st) : launch_up<64>(maps, p, nchunks, tiles, st);
  prof_mark("ffn_up_tc", st);
  if (e != cudaSuccess) return e;

  // 5. V~
  v_reduce_kernel<<<148 * 4, 256, 0, st>>>(b.Vpart, row_asg, eidx, a.tab, R, a.kg, a.ke, nchunks, KRP, b.Vt);
  prof_mark("v_reduce", st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  // 6. Y = [hsum | V~] [Wd | Bdn]^T, rows to their token slot
  e = BN2 == 256 ? launch_gemm<256, false>(mH, mVt, mWd, mBd, f / 64, 2 * KRP / 64, row_begin, G, d, d, 0,
                                           tiles, y_rows, d, row_asg, status, st)
                 : launch_gemm<128, false>(mH, mVt, mWd, mBd, f / 64, 2 * KRP / 64, row_begin, G, d, d, 0,
                                           tiles, y_rows, d, row_asg, status, st);
  prof_mark("ffn_down_tc", st);
  return e;
}

}  // namespace moe
