// Dispatch order: stable counting sorts of the routed work.
//
// Single-device form of the two-level dispatch of "Breaking the MoE LLM Trilemma" (paper notes),
// key design 3: work is grouped by expert group first, then by expert.  Assignments (t, slot)
// are ordered by key (group, expert, token); (token, group-slot) rows by key (group, token).
// Deterministic: per-block histograms, one exclusive scan, then in-block ranks from warp ballots.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kPermBlock = 256;  // tokens per block (8 warps)

// cnt[b][0..E) expert histogram, cnt[b][E..E+G) row (group) histogram of token block b.
__global__ void __launch_bounds__(kPermBlock) perm_count_kernel(const int32_t* __restrict__ eidx,
                                                                GroupTable tab, int Tn, int kg,
                                                                int ke, int32_t* __restrict__ cnt) {
  pdl_wait();
  pdl_trigger();
  __shared__ int sc[kMaxE + kMaxE];
  const int E = tab.E, G = tab.G, k = kg * ke;
  for (int i = threadIdx.x; i < E + G; i += blockDim.x) sc[i] = 0;
  __syncthreads();
  const int t = blockIdx.x * kPermBlock + threadIdx.x;
  if (t < Tn) {
    for (int s = 0; s < k; ++s) atomicAdd(&sc[eidx[(size_t)t * k + s]], 1);
    for (int j = 0; j < kg; ++j) atomicAdd(&sc[E + tab.group_of[eidx[(size_t)t * k + j * ke]]], 1);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E + G; i += blockDim.x) cnt[(size_t)blockIdx.x * (E + G) + i] = sc[i];
}

// One block.  off[b][key] = start of key's items of block b in the final order.
__global__ void perm_scan_kernel(const int32_t* __restrict__ cnt, GroupTable tab, int nblk,
                                 int32_t* __restrict__ off, int32_t* __restrict__ ebeg,
                                 int32_t* __restrict__ ecnt, int32_t* __restrict__ gbeg,
                                 int32_t* __restrict__ rbeg) {
  pdl_wait();
  pdl_trigger();
  __shared__ int total[kMaxE + kMaxE];
  __shared__ int base[kMaxE + kMaxE];
  const int E = tab.E, G = tab.G, K = tab.K, NK = E + G;
  for (int key = threadIdx.x; key < NK; key += blockDim.x) {
    int run = 0;
    for (int b = 0; b < nblk; ++b) {
      off[(size_t)b * NK + key] = run;
      run += cnt[(size_t)b * NK + key];
    }
    total[key] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int g = 0; g < G; ++g) {
      if (gbeg) gbeg[g] = run;
      for (int i = 0; i < K; ++i) {
        const int e = tab.member[g * K + i];
        base[e] = run;
        run += total[e];
      }
    }
    if (gbeg) gbeg[G] = run;
    int rrun = 0;
    for (int g = 0; g < G; ++g) {
      base[E + g] = rrun;
      rbeg[g] = rrun;
      rrun += total[E + g];
    }
    rbeg[G] = rrun;
  }
  __syncthreads();
  for (int key = threadIdx.x; key < NK; key += blockDim.x) {
    if (key < E) {
      if (ebeg) ebeg[key] = base[key];
      if (ecnt) ecnt[key] = total[key];
    }
    for (int b = 0; b < nblk; ++b) off[(size_t)b * NK + key] += base[key];
  }
}

__global__ void __launch_bounds__(kPermBlock) perm_scatter_kernel(
    const int32_t* __restrict__ eidx, GroupTable tab, int Tn, int kg, int ke,
    const int32_t* __restrict__ off, int32_t* __restrict__ perm, int32_t* __restrict__ inv_pos,
    int32_t* __restrict__ row_asg, int32_t* __restrict__ row_of) {
  pdl_wait();
  pdl_trigger();
  constexpr int W = kPermBlock / 32;
  __shared__ uint32_t emask[W][kMaxE];
  __shared__ int epre[W][kMaxE];
  __shared__ uint32_t gmask[W][kMaxE];
  __shared__ int gpre[W][kMaxE];
  const int E = tab.E, G = tab.G, k = kg * ke, NK = E + G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * kPermBlock + threadIdx.x;
  const bool valid = t < Tn;
  int my_e[kMaxK], my_g[kMaxK];
  for (int s = 0; s < k; ++s) my_e[s] = valid ? eidx[(size_t)t * k + s] : -1;
  for (int j = 0; j < kg; ++j) my_g[j] = valid ? (int)tab.group_of[my_e[j * ke]] : -1;
  for (int e = 0; e < E; ++e) {
    bool has = false;
    for (int s = 0; s < k; ++s) has |= (my_e[s] == e);
    const uint32_t m = __ballot_sync(0xffffffffu, has);
    if (lane == 0) emask[warp][e] = m;
  }
  for (int g = 0; g < G; ++g) {
    bool has = false;
    for (int j = 0; j < kg; ++j) has |= (my_g[j] == g);
    const uint32_t m = __ballot_sync(0xffffffffu, has);
    if (lane == 0) gmask[warp][g] = m;
  }
  __syncthreads();
  for (int key = threadIdx.x; key < NK; key += blockDim.x) {
    int run = 0;
    for (int w = 0; w < W; ++w) {
      if (key < E) { epre[w][key] = run; run += __popc(emask[w][key]); }
      else { gpre[w][key - E] = run; run += __popc(gmask[w][key - E]); }
    }
  }
  __syncthreads();
  if (!valid) return;
  const uint32_t lt = (1u << lane) - 1u;
  const int32_t* boff = off + (size_t)blockIdx.x * NK;
  for (int s = 0; s < k; ++s) {
    const int e = my_e[s];
    const int pos = boff[e] + epre[warp][e] + __popc(emask[warp][e] & lt);
    if (perm) perm[pos] = t * k + s;
    if (inv_pos) inv_pos[(size_t)t * k + s] = pos;
  }
  for (int j = 0; j < kg; ++j) {
    const int g = my_g[j];
    const int pos = boff[E + g] + gpre[warp][g] + __popc(gmask[warp][g] & lt);
    row_asg[pos] = t * kg + j;
    if (row_of) row_of[(size_t)t * kg + j] = pos;
  }
}

// Small batches (T <= 1024): the whole permutation in one CTA of 1024 threads, one token per
// thread, placed exactly as perm_scatter_kernel places a block (per-warp key masks from ballots,
// warp prefixes, ranks within the warp) with the key bases scanned in the same order as
// perm_scan_kernel: the same stable (key, token) order, in one launch instead of three.
constexpr int kFusedThreads = 1024;
constexpr int kFusedMaxT = kFusedThreads;
constexpr int kFusedMaxKeys = 128;   // E + G; (2 + 2 x 32) x 128 ints of dynamic shared memory

__global__ void __launch_bounds__(kFusedThreads) perm_fused_kernel(
    const int32_t* __restrict__ eidx, GroupTable tab, int Tn, int kg, int ke, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv_pos, int32_t* __restrict__ ebeg, int32_t* __restrict__ ecnt,
    int32_t* __restrict__ gbeg, int32_t* __restrict__ row_asg, int32_t* __restrict__ row_of,
    int32_t* __restrict__ rbeg) {
  pdl_wait();
  pdl_trigger();
  constexpr int W = kFusedThreads / 32;
  extern __shared__ int fused_smem[];
  const int E = tab.E, G = tab.G, K = tab.K, k = kg * ke, NK = E + G;
  int* total = fused_smem;                           // [NK] items per key
  int* base = fused_smem + NK;                       // [NK] first position of each key
  int* wpre = fused_smem + 2 * NK;                   // [W][NK] first position of each key in warp w
  uint32_t* wmask = (uint32_t*)(fused_smem + 2 * NK + W * NK);   // [W][NK] lanes of warp w holding the key
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = threadIdx.x;
  const bool valid = t < Tn;
  int my_e[kMaxK], my_g[kMaxK];
  for (int s = 0; s < k; ++s) my_e[s] = valid ? eidx[(size_t)t * k + s] : -1;
  for (int j = 0; j < kg; ++j) my_g[j] = valid ? (int)tab.group_of[my_e[j * ke]] : -1;
  for (int key = 0; key < NK; ++key) {
    bool has = false;
    if (key < E) { for (int s = 0; s < k; ++s) has |= (my_e[s] == key); }
    else { for (int j = 0; j < kg; ++j) has |= (my_g[j] == key - E); }
    const uint32_t m = __ballot_sync(0xffffffffu, has);
    if (lane == 0) wmask[warp * NK + key] = m;
  }
  __syncthreads();
  for (int key = threadIdx.x; key < NK; key += blockDim.x) {
    int c = 0;
    for (int w = 0; w < W; ++w) c += __popc(wmask[w * NK + key]);
    total[key] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int g = 0; g < G; ++g) {
      if (gbeg) gbeg[g] = acc;
      for (int i = 0; i < K; ++i) {
        const int e = tab.member[g * K + i];
        if (ebeg) ebeg[e] = acc;
        if (ecnt) ecnt[e] = total[e];
        base[e] = acc;
        acc += total[e];
      }
    }
    if (gbeg) gbeg[G] = acc;
    int racc = 0;
    for (int g = 0; g < G; ++g) {
      rbeg[g] = racc;
      base[E + g] = racc;
      racc += total[E + g];
    }
    rbeg[G] = racc;
  }
  __syncthreads();
  for (int key = threadIdx.x; key < NK; key += blockDim.x) {
    int acc = base[key];
    for (int w = 0; w < W; ++w) { wpre[w * NK + key] = acc; acc += __popc(wmask[w * NK + key]); }
  }
  __syncthreads();
  if (!valid) return;
  const uint32_t lt = (1u << lane) - 1u;
  for (int s = 0; s < k; ++s) {
    const int e = my_e[s];
    const int pos = wpre[warp * NK + e] + __popc(wmask[warp * NK + e] & lt);
    if (perm) perm[pos] = t * k + s;
    if (inv_pos) inv_pos[(size_t)t * k + s] = pos;
  }
  for (int j = 0; j < kg; ++j) {
    const int key = E + my_g[j];
    const int pos = wpre[warp * NK + key] + __popc(wmask[warp * NK + key] & lt);
    row_asg[pos] = t * kg + j;
    if (row_of) row_of[(size_t)t * kg + j] = pos;
  }
}

cudaError_t launch_permute(const LayerArgs& a, const int32_t* eidx, const PermOut& o, int32_t* cnt,
                           int32_t* off, int nblk, cudaStream_t st) {
  if (a.T == 0) {
    // empty batch: offsets are all zero
    cudaError_t e = cudaSuccess;
    if (o.gbeg) e = cudaMemsetAsync(o.gbeg, 0, sizeof(int32_t) * (a.G + 1), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(o.rbeg, 0, sizeof(int32_t) * (a.G + 1), st);
    if (e == cudaSuccess && o.ebeg) e = cudaMemsetAsync(o.ebeg, 0, sizeof(int32_t) * a.E, st);
    if (e == cudaSuccess && o.ecnt) e = cudaMemsetAsync(o.ecnt, 0, sizeof(int32_t) * a.E, st);
    return e;
  }
  if (a.T <= kFusedMaxT && a.E + a.G <= kFusedMaxKeys) {
    const size_t smem = (size_t)(2 + 2 * (kFusedThreads / 32)) * (a.E + a.G) * sizeof(int);
    launch_pdl(perm_fused_kernel, dim3(1), dim3(kFusedThreads), smem, st, eidx, a.tab, a.T, a.kg, a.ke, o.perm,
               o.inv_pos, o.ebeg,
                                                   o.ecnt, o.gbeg, o.row_asg, o.row_of, o.rbeg);
    prof_mark("perm_fused", st);
    return cudaGetLastError();
  }
  launch_pdl(perm_count_kernel, dim3(nblk), dim3(kPermBlock), 0, st, eidx, a.tab, a.T, a.kg, a.ke, cnt);
  prof_mark("perm_count", st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  launch_pdl(perm_scan_kernel, dim3(1), dim3(512), 0, st, (const int32_t*)cnt, a.tab, nblk, off, o.ebeg, o.ecnt,
             o.gbeg, o.rbeg);
  prof_mark("perm_scan", st);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  launch_pdl(perm_scatter_kernel, dim3(nblk), dim3(kPermBlock), 0, st, eidx, a.tab, a.T, a.kg, a.ke,
             (const int32_t*)off, o.perm,
                                                   o.inv_pos, o.row_asg, o.row_of);
  prof_mark("perm_scatter", st);
  return cudaGetLastError();
}

}  // namespace moe
