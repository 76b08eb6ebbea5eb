// Dispatch order: stable counting sorts of the routed work.
//
// Single-device form of the two-level dispatch of "Breaking the MoE LLM Trilemma" (paper notes),
// key design 3: work is grouped by expert group first, then by expert.  Assignments (t, slot)
// are ordered by key (group, expert, token); (token, group-slot) rows by key (group, token).
// Deterministic: per-block histograms, one exclusive scan, then in-block ranks from warp ballots.
#include "common.cuh"
#include "kernels.h"
#include "perm_dev.cuh"

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

// Small batches (T <= 1024): the whole permutation in one CTA, one token per thread (as many
// warps as the batch needs), placed exactly as perm_scatter_kernel places a block (per-warp key
// masks, warp prefixes, ranks within the warp) with the key bases scanned in the same order as
// perm_scan_kernel: the same stable (key, token) order, in one launch instead of three.  The
// masks are built with shared atomicOr (one bit per lane and key; a token holds a key at most
// once); the key bases come from two warp-wide scans (experts in group / member order, then the
// row keys by group).
constexpr int kFusedThreads = 1024;
constexpr int kFusedMaxT = kFusedThreads;
constexpr int kFusedMaxKeys = 512;   // E + G; (2 + 2 x 32) x 512 ints of dynamic shared memory at most

__global__ void __launch_bounds__(kFusedThreads) perm_fused_kernel(
    const int32_t* __restrict__ eidx, GroupTable tab, int Tn, int kg, int ke, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv_pos, int32_t* __restrict__ ebeg, int32_t* __restrict__ ecnt,
    int32_t* __restrict__ gbeg, int32_t* __restrict__ row_asg, int32_t* __restrict__ row_of,
    int32_t* __restrict__ rbeg) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int fused_smem[];
  perm_block(eidx, tab, Tn, kg, ke, perm, inv_pos, ebeg, ecnt, gbeg, row_asg, row_of, rbeg, fused_smem);
}

// Larger batches: the same placement in one cooperative launch.  Block b (256 tokens, as in
// perm_count_kernel / perm_scatter_kernel) builds its per-warp key masks with shared atomicOr
// (one bit per lane and key; a token holds a key at most once, so the masks do not depend on
// the order of the atomics), publishes its key counts, and waits at a grid-wide barrier (every
// block is resident: cooperative launch).  Each block then sums the counts of the blocks before
// it (the scan of perm_scan_kernel, restricted to what the block needs), takes the key bases from
// the totals, and places its items.
constexpr int kCoopBlock = kPermBlock;

__device__ __forceinline__ uint64_t perm_now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// The grid barrier waits for gridDim.x + wait.phantom arrivals and gives up after wait.limit_ns
// (2 s in normal use, with no phantom arrivals).
__global__ void __launch_bounds__(kCoopBlock) perm_coop_kernel(
    const int32_t* __restrict__ eidx, GroupTable tab, int Tn, int kg, int ke, int32_t* __restrict__ cnt,
    DevStatus* status, PermWait wait, int32_t* __restrict__ perm, int32_t* __restrict__ inv_pos, int32_t* __restrict__ ebeg,
    int32_t* __restrict__ ecnt, int32_t* __restrict__ gbeg, int32_t* __restrict__ row_asg,
    int32_t* __restrict__ row_of, int32_t* __restrict__ rbeg) {
  pdl_wait();
  pdl_trigger();
  constexpr int W = kCoopBlock / 32;
  extern __shared__ int coop_smem[];
  const int E = tab.E, G = tab.G, K = tab.K, k = kg * ke, NK = E + G;
  uint32_t* wmask = (uint32_t*)coop_smem;            // [W][NK] lanes of warp w holding the key
  int* wpre = coop_smem + W * NK;                    // [W][NK] items of the key in warps < w
  int* kpos = coop_smem + 2 * W * NK;                // [NK] first position of the key's items of this block
  int* ktot = coop_smem + 2 * W * NK + NK;           // [NK] items of the key in the batch
  __shared__ int s_abort;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nblk = gridDim.x, b = blockIdx.x;
  const int t = b * kCoopBlock + threadIdx.x;
  const bool valid = t < Tn;
  for (int i = threadIdx.x; i < W * NK; i += kCoopBlock) wmask[i] = 0u;
  __syncthreads();
  // slot s of the token: expert my_e[s]; slots s = j * ke open group slot j (its row key)
  int my_e[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) my_e[s] = (valid && s < k) ? eidx[(size_t)t * k + s] : 0;
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
  for (int key = threadIdx.x; key < NK; key += kCoopBlock) {
    int run = 0;
    for (int w = 0; w < W; ++w) { wpre[w * NK + key] = run; run += __popc(wmask[w * NK + key]); }
    cnt[(size_t)b * NK + key] = run;
  }
  // grid-wide barrier on the status word's counter (zeroed before the launch)
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned int* bar = &status->grid_bar;
    atomicAdd(bar, 1u);
    int ab = 0;
    const uint64_t t0 = perm_now_ns();
    for (uint32_t it = 1;; ++it) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
      if (v >= (unsigned int)nblk + wait.phantom) break;
      if ((it & 63) == 0 && perm_now_ns() - t0 > wait.limit_ns) {
        atomicExch(&status->code, (int)MOE_ERR_TIMEOUT);
        atomicExch(&status->where, 90);
        ab = 1;
        break;
      }
    }
    s_abort = ab;
  }
  __syncthreads();
  if (s_abort) return;
  __threadfence();
  // counts of the blocks before this one and of the whole batch, per key
  for (int key = threadIdx.x; key < NK; key += kCoopBlock) {
    int pre = 0, tot = 0;
    for (int bb = 0; bb < nblk; ++bb) {
      const int c = __ldcg(cnt + (size_t)bb * NK + key);
      pre += bb < b ? c : 0;
      tot += c;
    }
    kpos[key] = pre;
    ktot[key] = tot;
  }
  __syncthreads();
  // key order: experts group by group (members ascending), then the row keys by group
  if (warp == 0) {
    const int all = warp_ordered_scan(
        E, lane, [&](int pos) { return (int)tab.member[pos]; }, [&](int key) { return ktot[key]; },
        [&](int pos, int e, int start) {
          kpos[e] += start;
          if (b == 0) {
            if (ebeg) ebeg[e] = start;
            if (ecnt) ecnt[e] = ktot[e];
            if (gbeg && pos % K == 0) gbeg[pos / K] = start;
          }
        });
    if (b == 0 && gbeg && lane == 0) gbeg[G] = all;
  } else if (warp == 1) {
    const int all = warp_ordered_scan(
        G, lane, [&](int pos) { return E + pos; }, [&](int key) { return ktot[key]; },
        [&](int pos, int key, int start) {
          kpos[key] += start;
          if (b == 0) rbeg[pos] = start;
        });
    if (b == 0 && lane == 0) rbeg[G] = all;
  }
  __syncthreads();
  if (!valid) return;
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) {
    if (s >= k) break;
    const int e = my_e[s];
    const int pos = kpos[e] + wpre[warp * NK + e] + __popc(wmask[warp * NK + e] & lt);
    if (perm) perm[pos] = t * k + s;
    if (inv_pos) inv_pos[(size_t)t * k + s] = pos;
    if (s % ke == 0) {
      const int j = s / ke, key = E + tab.group_of[e];
      const int rpos = kpos[key] + wpre[warp * NK + key] + __popc(wmask[warp * NK + key] & lt);
      row_asg[rpos] = t * kg + j;
      if (row_of) row_of[(size_t)t * kg + j] = rpos;
    }
  }
}

// Whether the cooperative form fits: every block resident at once on this device.
static bool coop_fits(int nblk, size_t smem) {
  static int sms[64] = {0}, per_sm[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (sms[dev] == 0) {
    int coop = 0, n = 0, occ = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) return false;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    // occupancy at the largest dynamic shared memory the kernel is launched with (E + G <= 512)
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, perm_coop_kernel, kCoopBlock,
                                                      (size_t)(2 * (kCoopBlock / 32) + 2) * 512 * sizeof(int)) !=
        cudaSuccess)
      return false;
    per_sm[dev] = occ;
    sms[dev] = n;
  }
  (void)smem;
  return nblk <= sms[dev] * per_sm[dev];
}

cudaError_t launch_permute(const LayerArgs& a, const int32_t* eidx, const PermOut& o, int32_t* cnt,
                           int32_t* off, int nblk, DevStatus* status, bool bar_zeroed, cudaStream_t st,
                           PermWait wait) {
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
    const int threads = (a.T + 31) / 32 * 32;
    const size_t smem = (size_t)(2 + 2 * (threads / 32)) * (a.E + a.G) * sizeof(int);
    static std::atomic<uint64_t> attr{0};
    if (const cudaError_t e = smem_attr_once(perm_fused_kernel,
                                             (2 + 2 * (kFusedThreads / 32)) * kFusedMaxKeys * sizeof(int), attr);
        e != cudaSuccess)
      return e;
    launch_pdl(perm_fused_kernel, dim3(1), dim3(threads), smem, st, eidx, a.tab, a.T, a.kg, a.ke, o.perm,
               o.inv_pos, o.ebeg,
                                                   o.ecnt, o.gbeg, o.row_asg, o.row_of, o.rbeg);
    prof_mark("perm_fused", st);
    return cudaGetLastError();
  }
  const size_t coop_smem = (size_t)(2 * (kCoopBlock / 32) + 2) * (a.E + a.G) * sizeof(int);
  if (status != nullptr && a.E + a.G <= 512 && coop_fits(nblk, coop_smem)) {
    if (!bar_zeroed) {
      const cudaError_t e = cudaMemsetAsync(&status->grid_bar, 0, sizeof(status->grid_bar), st);
      if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nblk);
    cfg.blockDim = dim3(kCoopBlock);
    cfg.dynamicSmemBytes = coop_smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, perm_coop_kernel, eidx, a.tab, a.T, a.kg, a.ke, cnt, status, wait, o.perm,
                                       o.inv_pos, o.ebeg, o.ecnt, o.gbeg, o.row_asg, o.row_of, o.rbeg);
    prof_mark("perm_coop", st);
    return e;
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
