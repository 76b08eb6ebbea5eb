// Tensor-core router with exact verification.
//
// The routing decision must equal the one the canonical FP32 order takes (logits summed lane by
// lane in a fixed order, then an xor butterfly; "router in FP32", routing-mechanisms page §3.1).
// That order runs on the CUDA cores only, at about a third of their FMA rate.  This kernel
// computes the logits of 128 tokens per CTA on the tensor cores instead (BF16 x BF16 -> FP32 in
// TMEM, tcgen05.mma), with a bound on how far they can lie from the canonical ones:
//
//   |s_tc - s_canonical| <= delta = c_err * ||x_t|| * ||w_j||  +  2^-22 |s_tc|
//
// where c_err covers both sums' rounding (Cauchy-Schwarz bounds sum |x_i w_i| by the norms; the
// last term covers the bias add).  A token whose top-k_g groups, their order, and the top-k_e
// experts of each chosen group (and their order) are separated from every competitor by more
// than the two deltas takes the same decision in either precision, so its gidx/eidx/gates are
// written here.  Every other token (near ties, exact ties, NaN) is appended to a list that the
// canonical-order kernels recompute, so the indices always equal the canonical ones, bit for bit.
// The gates of verified tokens come from the tensor-core logits (an FP32 sum in another order).
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "kernels.h"
#include "tc.cuh"

namespace moe {

constexpr int kRtcTile = 128;     // tokens per CTA (TMEM lanes)
constexpr int kRtcMaxN = 128;     // router rows per CTA (padded group rows + expert rows)
constexpr int kRtcMaxStages = 8;
constexpr int kRtcSmem = 200 * 1024;
constexpr int kRtcMaxPick = 8;    // k_g and k_e limits of this path

struct RtcArgs {
  const float* bg;      // group-router bias (may be null)
  int T, nk, N, Gp;     // tokens, K blocks of 64, MMA columns (= router rows held), first expert column
  int stages;
  float c_err;
  int kg, ke;
  int32_t *gidx, *eidx;
  float* gate;
  int32_t* redo;        // tokens left to the canonical kernels
  DevStatus* status;    // status->route_redo counts them
  float* dbg;           // null, or [T][2 (G + E)]: each token's logits (groups, then experts) and deltas
  int across;           // MOE_ROUTE_ACROSS: gates from the top k_e over the union of the chosen groups
};

// Sum of squares of one 64-element row of a 128-byte-swizzled tile, into two pairs of partial
// sums (BF16 -> FP32 is exact: the 16 bits move to the top; then paired FP32 FMAs).
__device__ __forceinline__ float2 bf16x2_f32(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ void sumsq_row(const uint8_t* row, int r7, float2 (&acc)[2]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + ((c ^ r7) << 4));
    float2& a = acc[c & 1];
    const float2 f0 = bf16x2_f32(v.x), f1 = bf16x2_f32(v.y), f2 = bf16x2_f32(v.z), f3 = bf16x2_f32(v.w);
    a = fma2(f0, f0, a); a = fma2(f1, f1, a); a = fma2(f2, f2, a); a = fma2(f3, f3, a);
  }
}

// pick_verified for at most 8 candidates held in registers (loops unrolled, no shared-memory
// round trips): the picks' values and ids, best first.
__device__ __forceinline__ bool pick8(const float (&v)[8], const float (&dl)[8], const int (&id)[8], int n, int k,
                                      float (&pv)[kRtcMaxPick], int (&pid)[kRtcMaxPick]) {
  bool ok = true;
  uint32_t picked = 0;
  float prev_lo = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < n) ok &= v[i] == v[i];                              // NaN: not verifiable
#pragma unroll
  for (int j = 0; j < kRtcMaxPick; ++j) {
    pv[j] = 0.f;
    pid[j] = 0;
    if (j < k) {
      float bv = 0.f, bd = 0.f;
      int bi = -1, bid = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const bool cand = i < n && !((picked >> i) & 1u);
        if (cand && (bi < 0 || v[i] > bv || (v[i] == bv && id[i] < bid))) { bv = v[i]; bd = dl[i]; bi = i; bid = id[i]; }
      }
      if (bi < 0) { ok = false; bi = 0; }
      picked |= 1u << bi;
      if (j > 0) ok &= prev_lo > bv + bd;
      prev_lo = bv - bd;
      pv[j] = bv;
      pid[j] = bid;
    }
  }
  if (k < n) {
    float top = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < n && !((picked >> i) & 1u)) top = fmaxf(top, v[i] + dl[i]);
    ok &= prev_lo > top;
  }
  return ok;
}

// Picks the k best of n candidates (value v(i), id(i); ties -> lower id) into (pid, pv), best
// first, and returns whether the picks are verified: each pick's interval [v - dl, v + dl] lies
// strictly above the next pick's and the last pick's above every unpicked candidate's.
template <typename V, typename D, typename I>
__device__ __forceinline__ bool pick_verified(int n, int k, V v, D dl, I id, int (&pidx)[kRtcMaxPick],
                                              float (&pv)[kRtcMaxPick]) {
  bool ok = true;
  float prev_v = 0.f, prev_lo = 0.f;
  int prev_id = -1;
#pragma unroll
  for (int j = 0; j < kRtcMaxPick; ++j) { pidx[j] = 0; pv[j] = 0.f; }
#pragma unroll
  for (int j = 0; j < kRtcMaxPick; ++j) {
    if (j >= k) break;
    float bv = 0.f;
    int bi = -1, bid = 0;
    for (int i = 0; i < n; ++i) {
      const float vi = v(i);
      const int ii = id(i);
      ok &= vi == vi;                                           // NaN: not verifiable
      // candidates after the previous pick in (value desc, id asc) order
      const bool after = j == 0 || vi < prev_v || (vi == prev_v && ii > prev_id);
      if (after && (bi < 0 || vi > bv || (vi == bv && ii < bid))) { bv = vi; bi = i; bid = ii; }
    }
    if (bi < 0) return false;
    const float d = dl(bi);
    if (j > 0) ok &= prev_lo > bv + d;
    pidx[j] = bi;
    pv[j] = bv;
    prev_v = bv; prev_id = bid; prev_lo = bv - d;
  }
  if (k < n) {
    float top = -INFINITY;
    for (int i = 0; i < n; ++i) {
      bool picked = false;
#pragma unroll
      for (int j = 0; j < kRtcMaxPick; ++j) picked |= j < k && pidx[j] == i;
      if (!picked) top = fmaxf(top, v(i) + dl(i));
    }
    ok &= prev_lo > top;
  }
  return ok;
}

__global__ void __launch_bounds__(192, 1) router_tc_kernel(
    const __grid_constant__ CUtensorMap mX, const __grid_constant__ CUtensorMap mWg,
    const __grid_constant__ CUtensorMap mWe, GroupTable tab, RtcArgs p) {
  pdl_wait();
  pdl_trigger();
  constexpr uint32_t A_BYTES = kRtcTile * 128;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kRtcMaxStages], empty[kRtcMaxStages], acc_full, fin;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ float s_wn[kRtcMaxN];
  __shared__ uint8_t s_member[kMaxE];
  const int G = tab.G, E = tab.E, N = p.N, Gp = p.Gp, nk = p.nk, NS = p.stages;
  const uint32_t STAGE = A_BYTES + (uint32_t)N * 128;     // N % 16 == 0: stages stay 1024-byte aligned
  // four accumulators (one per 16-deep MMA of a K block) so that consecutive MMAs are independent
  const uint32_t ncols = 4 * N <= 64 ? 64u : 4 * N <= 128 ? 128u : 4 * N <= 256 ? 256u : 512u;
  uint8_t* smem = tc::align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tc::Abort ab{&abort_flag, p.status};
  const int t0 = blockIdx.x * kRtcTile;

  // router rows no copy writes ([G, Gp) and [Gp + E, N)) hold zeros in every stage
  for (int i = threadIdx.x; i < NS * N; i += blockDim.x) {
    const int s = i / N, r = i % N;
    if ((r >= G && r < Gp) || r >= Gp + E) {
      uint4* z = reinterpret_cast<uint4*>(smem + s * STAGE + A_BYTES + (r >> 3) * 1024 + (r & 7) * 128);
#pragma unroll
      for (int c = 0; c < 8; ++c) z[c] = make_uint4(0, 0, 0, 0);
    }
  }
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_member[i] = tab.member[i];
  tc::fence_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) { tc::bar_init(&full[s], 1); tc::bar_init(&empty[s], 1 + 4); }
    tc::bar_init(&acc_full, 1);
    tc::bar_init(&fin, 1);
    abort_flag = 0;
    tc::bar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, ncols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer: 128 token rows, the group rows at row 0, the expert rows at Gp
    tc::prefetch_map(&mX); tc::prefetch_map(&mWg); tc::prefetch_map(&mWe);
    const uint32_t tx = A_BYTES + (uint32_t)(G + E) * 128;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % NS, it = kb / NS;
      if (kb >= NS && !tc::bar_wait(&empty[s], (it - 1) & 1, ab, 61)) break;
      tc::bar_expect_tx(&full[s], tx);
      uint8_t* st = smem + s * STAGE;
      tc::tma_load_2d(st, &mX, &full[s], kb * 64, t0);
      tc::tma_load_2d(st + A_BYTES, &mWg, &full[s], kb * 64, 0);
      tc::tma_load_2d(st + A_BYTES + Gp * 128, &mWe, &full[s], kb * 64, 0);
    }
    if (abort_flag) tc::drain_copies();
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer: logits[128][N] in TMEM
    const uint32_t idesc = tc::idesc_bf16(kRtcTile, N);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % NS, it = kb / NS;
      if (!tc::bar_wait(&full[s], it & 1, ab, 62)) break;
      tc::fence_after();
      const uint32_t a0 = tc::smem_u32(smem + s * STAGE), b0 = a0 + A_BYTES;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc::mma_bf16(tmem + k * N, tc::sdesc(a0 + 32 * k), tc::sdesc(b0 + 32 * k), idesc, kb != 0);
      tc::mma_commit(&empty[s]);
    }
    tc::mma_commit(&acc_full);
    tc::mma_commit(&fin);
    const uint64_t w0 = tc::now_ns();
    while (!tc::bar_test(&fin, 0) && tc::now_ns() - w0 < tc::kWaitNs) {}
  } else if (warp >= 2) {
    // ---------------- norms during the K loop, then verification and selection (one token per thread)
    const int q = warp & 3, row = q * 32 + lane;
    float2 xa[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)}, wa[2] = {xa[0], xa[0]};
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % NS, it = kb / NS;
      if (!tc::bar_wait(&full[s], it & 1, ab, 63)) break;
      const uint8_t* st = smem + s * STAGE + (row >> 3) * 1024 + (row & 7) * 128;
      sumsq_row(st, row & 7, xa);
      if (row < N) sumsq_row(st + A_BYTES, row & 7, wa);
      __syncwarp();
      if (lane == 0) tc::bar_arrive(&empty[s]);
    }
    const float xn = (xa[0].x + xa[0].y) + (xa[1].x + xa[1].y);
    s_wn[row] = sqrtf((wa[0].x + wa[0].y) + (wa[1].x + wa[1].y));
    asm volatile("bar.sync 1, 128;" ::: "memory");      // stage memory is reused below
    const int t = t0 + row;
    bool unsafe = false;
    if (tc::bar_wait(&acc_full, 0, ab, 64) && !abort_flag) {
      tc::fence_after();
      float* lv = reinterpret_cast<float*>(smem) + row * (kRtcMaxN + 1);
      for (int c = 0; c < N; c += 16) {
        uint32_t v0[16], v1[16], v2[16], v3[16];
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + c;
        tc::tmem_ld16(ta, v0);
        tc::tmem_ld16(ta + N, v1);
        tc::tmem_ld16(ta + 2 * N, v2);
        tc::tmem_ld16(ta + 3 * N, v3);
        tc::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e)
          lv[c + e] = (__uint_as_float(v0[e]) + __uint_as_float(v1[e])) + (__uint_as_float(v2[e]) + __uint_as_float(v3[e]));
      }
      if (t < p.T) {
        for (int g = 0; g < G; ++g)
          if (p.bg) lv[g] = __fadd_rn(lv[g], p.bg[g]);
        const float xs = p.c_err * sqrtf(xn);
        auto delta = [&](int col) { return xs * s_wn[col] + 0x1p-22f * fabsf(lv[col]); };
        if (p.dbg) {
          float* o = p.dbg + (size_t)t * 2 * (G + E);
          for (int g = 0; g < G; ++g) { o[g] = lv[g]; o[G + E + g] = delta(g); }
          for (int e = 0; e < E; ++e) { o[G + e] = lv[Gp + e]; o[2 * G + E + e] = delta(Gp + e); }
        }
        const int K = tab.K, kg = p.kg, ke = p.ke, k = kg * ke;
        // The across-groups reading: the top k_e over the union of the chosen groups' members
        // (candidate i: member i % K of chosen group i / K), verified like the other picks; gates
        // = softmax over them in pick order on their slots (the within-group candidates already
        // written to eidx), zero on the other slots.
        auto across_gates = [&](const int (&gsel)[kRtcMaxPick]) -> bool {
          auto eid = [&](int i) { return (int)s_member[gsel[i / K] * K + i % K]; };
          int pidx[kRtcMaxPick];
          float pv[kRtcMaxPick];
          if (!pick_verified(
                  kg * K, ke, [&](int i) { return lv[Gp + eid(i)]; }, [&](int i) { return delta(Gp + eid(i)); }, eid,
                  pidx, pv))
            return false;
          float q[kRtcMaxPick], den = 0.f;
#pragma unroll
          for (int j = 0; j < kRtcMaxPick; ++j)
            if (j < ke) { q[j] = expf(pv[j] - pv[0]); den += q[j]; }
          for (int s2 = 0; s2 < k; ++s2) {
            const int e = p.eidx[(size_t)t * k + s2];
            float gv2 = 0.f;
#pragma unroll
            for (int j = 0; j < kRtcMaxPick; ++j)
              if (j < ke && eid(pidx[j]) == e) gv2 = q[j] / den;
            p.gate[(size_t)t * k + s2] = gv2;
          }
          return true;
        };
        if (G <= 8 && K <= 8) {
          // register path
          float v8[8], d8[8], gv[kRtcMaxPick];
          int id8[8], gsel[kRtcMaxPick];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            v8[i] = i < G ? lv[i] : 0.f;
            d8[i] = i < G ? delta(i) : 0.f;
            id8[i] = i;
          }
          bool ok = pick8(v8, d8, id8, G, kg, gv, gsel);
          float pe[kRtcMaxPick], pden = 0.f;
#pragma unroll
          for (int j = 0; j < kRtcMaxPick; ++j)
            if (j < kg) { pe[j] = expf(gv[j] - gv[0]); pden += pe[j]; }
#pragma unroll
          for (int j = 0; j < kRtcMaxPick; ++j) {
            if (j >= kg || !ok) break;
            const int g = gsel[j];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int e = i < K ? (int)s_member[g * K + i] : 0;
              id8[i] = e;
              v8[i] = i < K ? lv[Gp + e] : 0.f;
              d8[i] = i < K ? delta(Gp + e) : 0.f;
            }
            float ev[kRtcMaxPick];
            int esel[kRtcMaxPick];
            ok &= pick8(v8, d8, id8, K, ke, ev, esel);
            if (!ok) break;
            p.gidx[(size_t)t * kg + j] = g;
            const float pj = pe[j] / pden;
            float qe[kRtcMaxPick], qden = 0.f;
#pragma unroll
            for (int s2 = 0; s2 < kRtcMaxPick; ++s2)
              if (s2 < ke) { qe[s2] = expf(ev[s2] - ev[0]); qden += qe[s2]; }
#pragma unroll
            for (int s2 = 0; s2 < kRtcMaxPick; ++s2) {
              if (s2 >= ke) break;
              p.eidx[(size_t)t * k + j * ke + s2] = esel[s2];
              p.gate[(size_t)t * k + j * ke + s2] = pj * (qe[s2] / qden);
            }
          }
          if (ok && p.across) ok = across_gates(gsel);
          unsafe = !ok;
        } else {
        int gsel[kRtcMaxPick];
        float gv[kRtcMaxPick];
        bool ok = pick_verified(
            G, kg, [&](int i) { return lv[i]; }, [&](int i) { return delta(i); }, [&](int i) { return i; }, gsel,
            gv);
        // gates as the canonical selection forms them: p_j q_s, softmaxes over the picks in order
        float pe[kRtcMaxPick], pden = 0.f;
#pragma unroll
        for (int j = 0; j < kRtcMaxPick; ++j)
          if (j < kg) { pe[j] = expf(gv[j] - gv[0]); pden += pe[j]; }
#pragma unroll
        for (int j = 0; j < kRtcMaxPick; ++j) {
          if (j >= kg || !ok) break;
          const int g = gsel[j];
          const uint8_t* mem = s_member + g * K;
          int esel[kRtcMaxPick];
          float ev[kRtcMaxPick];
          ok &= pick_verified(
              K, ke, [&](int i) { return lv[Gp + mem[i]]; }, [&](int i) { return delta(Gp + mem[i]); },
              [&](int i) { return (int)mem[i]; }, esel, ev);
          if (!ok) break;
          p.gidx[(size_t)t * kg + j] = g;
          const float pj = pe[j] / pden;
          float qe[kRtcMaxPick], qden = 0.f;
#pragma unroll
          for (int s2 = 0; s2 < kRtcMaxPick; ++s2)
            if (s2 < ke) { qe[s2] = expf(ev[s2] - ev[0]); qden += qe[s2]; }
#pragma unroll
          for (int s2 = 0; s2 < kRtcMaxPick; ++s2) {
            if (s2 >= ke) break;
            p.eidx[(size_t)t * k + j * ke + s2] = mem[esel[s2]];
            p.gate[(size_t)t * k + j * ke + s2] = pj * (qe[s2] / qden);
          }
        }
        if (ok && p.across) ok = across_gates(gsel);
        unsafe = !ok;
        }
      }
    }
    // the warp's unverified tokens go to the list with one atomic
    const uint32_t m = __ballot_sync(0xffffffffu, unsafe);
    if (m) {
      int base = 0;
      if (lane == 0) base = atomicAdd(&p.status->route_redo, __popc(m));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (unsafe) p.redo[base + __popc(m & ((1u << lane) - 1u))] = t;
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, ncols);
  }
}

// Error constant of the verification.  Canonical order: each of 32 partial sums adds d/32
// products, then 5 butterfly adds, one FP32 rounding each (|error| <= (d/32 + 5) 2^-24 sum|x_i w_i|).
// Tensor cores: exact BF16 products, FP32 accumulation in four accumulators summed at the end;
// modelled (with a 4x margin over one truncation per 16-element MMA step, and 8 spare roundings
// for the final adds) as <= (d/8 + 8) 2^-22 sum|x_i w_i|.  The norms themselves
// are FP32 sums (relative error below 1e-3 here): 1% on top.
static float route_tc_c_err(int d) {
  const double c = (d / 8.0 + 8.0) * 0x1p-22 + (d / 32.0 + 6.0) * 0x1p-24;
  return (float)(1.01 * c);
}

int route_tc_columns(const LayerArgs& a) {
  const int Gp = (a.G + 7) / 8 * 8;
  return (Gp + a.E + 15) / 16 * 16;
}

bool route_tc_ok(const LayerArgs& a) {
  return a.bf16 && a.T >= 1024 && route_tc_columns(a) <= kRtcMaxN && a.kg <= kRtcMaxPick &&
         a.ke <= kRtcMaxPick && a.d % 64 == 0;
}

cudaError_t launch_route_tc(const LayerArgs& a, const void* x, const void* wg, const float* bg, const void* we,
                            int32_t* gidx, int32_t* eidx, float* gate, int32_t* redo, DevStatus* status,
                            cudaStream_t st, float* dbg) {
  CUtensorMap mX, mWg, mWe;
  if (!make_map_bf16(&mX, x, (uint64_t)a.T, a.d, kRtcTile) || !make_map_bf16(&mWg, wg, a.G, a.d, a.G) ||
      !make_map_bf16(&mWe, we, a.E, a.d, a.E))
    return cudaErrorInvalidValue;
  RtcArgs p;
  p.bg = bg; p.T = a.T; p.nk = a.d / 64; p.N = route_tc_columns(a); p.Gp = (a.G + 7) / 8 * 8;
  p.c_err = route_tc_c_err(a.d); p.kg = a.kg; p.ke = a.ke;
  p.gidx = gidx; p.eidx = eidx; p.gate = gate; p.redo = redo; p.status = status; p.dbg = dbg;
  p.across = a.across ? 1 : 0;
  const size_t stage = (size_t)(kRtcTile + p.N) * 128;
  p.stages = (int)((kRtcSmem - 1024) / stage);
  if (p.stages > kRtcMaxStages) p.stages = kRtcMaxStages;
  const size_t smem = 1024 + (size_t)p.stages * stage;
  // the logits of the epilogue (128 rows of N + 1 floats) reuse the stages
  if ((size_t)kRtcTile * (kRtcMaxN + 1) * 4 > (size_t)p.stages * stage) return cudaErrorInvalidValue;
  static std::atomic<uint64_t> attr{0};
  if (const cudaError_t e = smem_attr_once(router_tc_kernel, kRtcSmem, attr); e != cudaSuccess) return e;
  const cudaError_t e = launch_pdl(router_tc_kernel, dim3((a.T + kRtcTile - 1) / kRtcTile), dim3(192), smem, st,
                                   mX, mWg, mWe, a.tab, p);
  prof_mark("router_tc", st);
  return e;
}

}  // namespace moe
