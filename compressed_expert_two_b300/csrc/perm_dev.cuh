// Device-side permutation of a small batch by one CTA, shared by the permutation kernels and the
// fused decode pre-pass.  Single-device form of the two-level dispatch of "Breaking the MoE LLM
// Trilemma" (paper notes), key design 3: assignments ordered by (group, expert, token), rows by
// (group, token); deterministic placement (per-warp key masks, warp prefixes, ranks in the warp).
#pragma once
#include "common.cuh"

namespace moe {

// Exclusive scan, in one warp, of cnt(0) .. cnt(n-1) taken in the order given by key_at(pos);
// calls put(pos, key, start) for every position.  Returns the total (in every lane).
template <typename KeyAt, typename Cnt, typename Put>
__device__ __forceinline__ int warp_ordered_scan(int n, int lane, KeyAt key_at, Cnt cnt, Put put) {
  const int per = (n + 31) / 32, lo = min(n, lane * per), hi = min(n, lo + per);
  int local = 0;
  for (int pos = lo; pos < hi; ++pos) local += cnt(key_at(pos));
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - local;
  for (int pos = lo; pos < hi; ++pos) {
    const int key = key_at(pos);
    put(pos, key, run);
    run += cnt(key);
  }
  return __shfl_sync(0xffffffffu, incl, 31);
}

// The whole permutation of up to blockDim.x tokens by one CTA (one token per thread), in
// `fused_smem` of (2 + 2 * (blockDim.x / 32)) * (E + G) ints.  Called by every thread of the CTA.
__device__ __forceinline__ void perm_block(const int32_t* __restrict__ eidx, const GroupTable& tab, int Tn, int kg,
                                           int ke, int32_t* __restrict__ perm, int32_t* __restrict__ inv_pos,
                                           int32_t* __restrict__ ebeg, int32_t* __restrict__ ecnt,
                                           int32_t* __restrict__ gbeg, int32_t* __restrict__ row_asg,
                                           int32_t* __restrict__ row_of, int32_t* __restrict__ rbeg,
                                           int* fused_smem) {
  const int W = blockDim.x >> 5;
  const int E = tab.E, G = tab.G, K = tab.K, k = kg * ke, NK = E + G;
  int* total = fused_smem;                           // [NK] items per key
  int* base = fused_smem + NK;                       // [NK] first position of each key
  int* wpre = fused_smem + 2 * NK;                   // [W][NK] first position of each key in warp w
  uint32_t* wmask = (uint32_t*)(fused_smem + 2 * NK + W * NK);   // [W][NK] lanes of warp w holding the key
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = threadIdx.x;
  const bool valid = t < Tn;
  for (int i = threadIdx.x; i < W * NK; i += blockDim.x) wmask[i] = 0u;
  // slot s of the token: expert my_e[s]; slots s = j * ke open group slot j (its row key)
  int my_e[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) my_e[s] = (valid && s < k) ? eidx[(size_t)t * k + s] : 0;
  __syncthreads();
  if (valid) {
    const uint32_t bit = 1u << lane;
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      if (s >= k) break;
      atomicOr(&wmask[warp * NK + my_e[s]], bit);
      if (s % ke == 0) atomicOr(&wmask[warp * NK + E + tab.group_of[my_e[s]]], bit);
    }
  }
  __syncthreads();
  for (int key = threadIdx.x; key < NK; key += blockDim.x) {
    int c = 0;
    for (int w = 0; w < W; ++w) c += __popc(wmask[w * NK + key]);
    total[key] = c;
  }
  __syncthreads();
  if (warp == 0) {
    // experts group by group (members ascending), then the row keys by group
    const int all = warp_ordered_scan(
        E, lane, [&](int pos) { return (int)tab.member[pos]; }, [&](int key) { return total[key]; },
        [&](int pos, int e, int start) {
          base[e] = start;
          if (ebeg) ebeg[e] = start;
          if (ecnt) ecnt[e] = total[e];
          if (gbeg && pos % K == 0) gbeg[pos / K] = start;
        });
    if (gbeg && lane == 0) gbeg[G] = all;
  } else if (warp == 1) {
    const int all = warp_ordered_scan(
        G, lane, [&](int pos) { return E + pos; }, [&](int key) { return total[key]; },
        [&](int pos, int key, int start) {
          base[key] = start;
          rbeg[pos] = start;
        });
    if (lane == 0) rbeg[G] = all;
  }
  if (W == 1 && warp == 0) {
    // a single warp runs both scans in turn
    __syncwarp();
    const int all = warp_ordered_scan(
        G, lane, [&](int pos) { return E + pos; }, [&](int key) { return total[key]; },
        [&](int pos, int key, int start) {
          base[key] = start;
          rbeg[pos] = start;
        });
    if (lane == 0) rbeg[G] = all;
  }
  __syncthreads();
  for (int key = threadIdx.x; key < NK; key += blockDim.x) {
    int acc = base[key];
    for (int w = 0; w < W; ++w) { wpre[w * NK + key] = acc; acc += __popc(wmask[w * NK + key]); }
  }
  __syncthreads();
  if (!valid) return;
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) {
    if (s >= k) break;
    const int e = my_e[s];
    const int pos = wpre[warp * NK + e] + __popc(wmask[warp * NK + e] & lt);
    if (perm) perm[pos] = t * k + s;
    if (inv_pos) inv_pos[(size_t)t * k + s] = pos;
    if (s % ke == 0) {
      const int j = s / ke, key = E + tab.group_of[e];
      const int rpos = wpre[warp * NK + key] + __popc(wmask[warp * NK + key] & lt);
      row_asg[rpos] = t * kg + j;
      if (row_of) row_of[(size_t)t * kg + j] = rpos;
    }
  }
}

}  // namespace moe
