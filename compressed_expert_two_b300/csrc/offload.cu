// Idle-group offload: group bases in pinned host memory, a device cache of `slots` groups.
//
// "Breaking the MoE LLM Trilemma" (paper notes), key design 4: whole groups that the current work
// does not use are moved off the GPU (to CPU memory) and brought back when needed, so that peak
// device memory stays near a dense model's.  Here the unit is a group's three base matrices
// (W_gate, W_up [f][d] and W_down [d][f], BF16): the residual factors are small and stay resident.
//
// Protocol per batch (all on the caller's streams, no device allocation):
//   1. moe_hier_route + moe_hier_permute on the compute stream;
//   2. moe_hier_groups_hit: the batch's rows per group, copied to the host (synchronises);
//   3. moe_hier_offload_require: every hit group that is not cached gets a slot -- an empty one,
//      else the least recently used slot whose group the batch does not hit -- and its three
//      matrices are copied host -> device on the copy stream, after the last FFN that read the
//      slot's previous group (an event), with an event recorded when they have landed;
//   4. moe_hier_ffn_offload: the compute stream waits for the hit groups' copies, the FFN kernels
//      read each group's base from its slot (the slot table travels with the launch), and an
//      event after the FFN marks those slots busy until then.
// Batch i+1's steps 1-3 may run while batch i's FFN runs: the copy stream never overwrites a slot
// before the FFN that reads it has finished, and the FFN never starts before its groups landed.
#include <string.h>

#include <new>

#include "common.cuh"
#include "kernels.h"

struct moe_hier_offload {
  int dev;
  int G, slots, d, f;
  size_t gu_bytes, dn_bytes;                 // bytes of one group's W_gate (= W_up) and W_down
  const char *host_gate, *host_up, *host_down;
  char *cache_gate, *cache_up, *cache_down;
  int slot_group[256];                       // group held by each slot (-1: empty)
  int group_slot[256];                       // slot of each group (-1: not cached)
  uint64_t last_use[256];                    // tick of the last require that hit the slot's group
  uint64_t tick;
  bool required[256];                        // groups of the last require call
  cudaEvent_t ready[256];                    // the slot's copy has landed
  cudaEvent_t busy[256];                     // the last FFN that read the slot has finished
  bool busy_recorded[256];
  uint64_t bytes_copied, misses, hits;
};

namespace moe {
// FFN with the bases read from the cache (api.cu).
int ffn_with_slots(const moe_hier_desc* desc, const void* x, const int32_t* group_map_host, const void* w_gate,
                   const void* w_up, const void* w_down, int wslots, const uint8_t* wslot,
                   const moe_hier_resid* resid, const int32_t* eidx, const float* gate, const int32_t* row_asg,
                   const int32_t* row_begin, void* y_rows, void* ws, size_t ws_bytes, void* stream);
}  // namespace moe

using namespace moe;

extern "C" {

int moe_hier_offload_create(const moe_hier_desc* desc, const void* w_gate_host, const void* w_up_host,
                            const void* w_down_host, void* cache_gate, void* cache_up, void* cache_down,
                            int32_t slots, moe_hier_offload** out) {
  if (!out) return MOE_ERR_INVALID;
  *out = nullptr;
  if (!desc || !w_gate_host || !w_up_host || !w_down_host || !cache_gate || !cache_up || !cache_down)
    return MOE_ERR_INVALID;
  if (desc->G <= 0 || desc->G > 255 || desc->d_model <= 0 || desc->d_ff <= 0) return MOE_ERR_INVALID;
  if (slots < 1 || slots > desc->G) return MOE_ERR_INVALID;
  if (desc->act_dtype != MOE_BF16 || desc->resid_fmt != MOE_RESID_INT4_G64) return MOE_ERR_UNSUPPORTED;
  if (((uintptr_t)cache_gate | (uintptr_t)cache_up | (uintptr_t)cache_down) & 15) return MOE_ERR_INVALID;
  moe_hier_offload* h = new (std::nothrow) moe_hier_offload();
  if (!h) return MOE_ERR_INVALID;
  memset(h, 0, sizeof(*h));
  if (cudaGetDevice(&h->dev) != cudaSuccess) { delete h; return MOE_ERR_CUDA; }
  h->G = desc->G; h->slots = slots; h->d = desc->d_model; h->f = desc->d_ff;
  h->gu_bytes = (size_t)h->f * h->d * 2;
  h->dn_bytes = (size_t)h->d * h->f * 2;
  h->host_gate = (const char*)w_gate_host; h->host_up = (const char*)w_up_host; h->host_down = (const char*)w_down_host;
  h->cache_gate = (char*)cache_gate; h->cache_up = (char*)cache_up; h->cache_down = (char*)cache_down;
  for (int i = 0; i < 256; ++i) { h->slot_group[i] = -1; h->group_slot[i] = -1; }
  for (int s = 0; s < slots; ++s) {
    if (cudaEventCreateWithFlags(&h->ready[s], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->busy[s], cudaEventDisableTiming) != cudaSuccess) {
      for (int t = 0; t <= s; ++t) {
        if (h->ready[t]) cudaEventDestroy(h->ready[t]);
        if (h->busy[t]) cudaEventDestroy(h->busy[t]);
      }
      delete h;
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
  }
  *out = h;
  return MOE_OK;
}

int moe_hier_offload_destroy(moe_hier_offload* h) {
  if (!h) return MOE_ERR_INVALID;
  for (int s = 0; s < h->slots; ++s) {
    cudaEventSynchronize(h->busy[s]);
    cudaEventSynchronize(h->ready[s]);
    cudaEventDestroy(h->ready[s]);
    cudaEventDestroy(h->busy[s]);
  }
  delete h;
  return MOE_OK;
}

int moe_hier_groups_hit(const moe_hier_desc* desc, const int32_t* row_begin, int32_t* hit_host, void* stream) {
  if (!desc || !row_begin || !hit_host || desc->G <= 0 || desc->G > 255) return MOE_ERR_INVALID;
  int32_t rb[257];
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(rb, row_begin, sizeof(int32_t) * (desc->G + 1), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  for (int g = 0; g < desc->G; ++g) hit_host[g] = rb[g + 1] > rb[g] ? 1 : 0;
  return MOE_OK;
}

int moe_hier_offload_require(moe_hier_offload* h, const int32_t* hit_host, int32_t* copied, void* copy_stream) {
  if (!h || !hit_host) return MOE_ERR_INVALID;
  int n_hit = 0;
  for (int g = 0; g < h->G; ++g) n_hit += hit_host[g] != 0;
  if (n_hit > h->slots) return MOE_ERR_INVALID;            // the batch needs more groups than slots
  cudaStream_t cs = (cudaStream_t)copy_stream;
  ++h->tick;
  for (int g = 0; g < h->G; ++g) {
    h->required[g] = hit_host[g] != 0;
    if (h->required[g] && h->group_slot[g] >= 0) {
      h->last_use[h->group_slot[g]] = h->tick;
      ++h->hits;
    }
  }
  int n_copied = 0;
  for (int g = 0; g < h->G; ++g) {
    if (!h->required[g] || h->group_slot[g] >= 0) continue;
    // victim: an empty slot, else the least recently used slot whose group this batch does not hit
    int victim = -1;
    for (int s = 0; s < h->slots && victim < 0; ++s)
      if (h->slot_group[s] < 0) victim = s;
    if (victim < 0) {
      uint64_t best = ~0ull;
      for (int s = 0; s < h->slots; ++s) {
        const int og = h->slot_group[s];
        if (h->required[og]) continue;
        if (h->last_use[s] < best) { best = h->last_use[s]; victim = s; }
      }
    }
    if (victim < 0) return MOE_ERR_INVALID;                 // cannot happen: n_hit <= slots
    const int old = h->slot_group[victim];
    if (old >= 0) h->group_slot[old] = -1;
    cudaError_t e = cudaSuccess;
    if (h->busy_recorded[victim]) e = cudaStreamWaitEvent(cs, h->busy[victim], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h->cache_gate + victim * h->gu_bytes, h->host_gate + (size_t)g * h->gu_bytes, h->gu_bytes,
                          cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h->cache_up + victim * h->gu_bytes, h->host_up + (size_t)g * h->gu_bytes, h->gu_bytes,
                          cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h->cache_down + victim * h->dn_bytes, h->host_down + (size_t)g * h->dn_bytes, h->dn_bytes,
                          cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess) e = cudaEventRecord(h->ready[victim], cs);
    if (e != cudaSuccess) {
      h->slot_group[victim] = -1;                          // the slot's contents are unknown now
      return MOE_ERR_CUDA;
    }
    h->slot_group[victim] = g;
    h->group_slot[g] = victim;
    h->last_use[victim] = h->tick;
    h->bytes_copied += 2 * h->gu_bytes + h->dn_bytes;
    ++h->misses;
    ++n_copied;
  }
  if (copied) *copied = n_copied;
  return MOE_OK;
}

int moe_hier_ffn_offload(moe_hier_offload* h, const moe_hier_desc* desc, const void* x,
                         const int32_t* group_map_host, const moe_hier_resid* resid, const int32_t* eidx,
                         const float* gate, const int32_t* row_asg, const int32_t* row_begin, void* y_rows,
                         void* ws, size_t ws_bytes, void* stream) {
  if (!h || !desc || desc->G != h->G || desc->d_model != h->d || desc->d_ff != h->f) return MOE_ERR_INVALID;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t wslot[kMaxE];
  // groups without a slot point one past the cache: the kernels' tensor maps end there, so a
  // tile of such a group (a caller that skipped moe_hier_offload_require) reads zeros, not memory
  for (int g = 0; g < kMaxE; ++g)
    wslot[g] = (uint8_t)(g < h->G && h->group_slot[g] >= 0 ? h->group_slot[g] : h->slots);
  for (int g = 0; g < h->G; ++g)
    if (h->required[g] && h->group_slot[g] >= 0 &&
        cudaStreamWaitEvent(s, h->ready[h->group_slot[g]], 0) != cudaSuccess)
      return MOE_ERR_CUDA;
  const int st = ffn_with_slots(desc, x, group_map_host, h->cache_gate, h->cache_up, h->cache_down, h->slots, wslot,
                                resid, eidx, gate, row_asg, row_begin, y_rows, ws, ws_bytes, stream);
  if (st != MOE_OK) return st;
  for (int g = 0; g < h->G; ++g) {
    const int sl = h->group_slot[g];
    if (!h->required[g] || sl < 0) continue;
    if (cudaEventRecord(h->busy[sl], s) != cudaSuccess) return MOE_ERR_CUDA;
    h->busy_recorded[sl] = true;
  }
  return MOE_OK;
}

int moe_hier_offload_stats(const moe_hier_offload* h, uint64_t* bytes_copied, uint64_t* misses, uint64_t* hits,
                           int32_t* slot_group) {
  if (!h) return MOE_ERR_INVALID;
  if (bytes_copied) *bytes_copied = h->bytes_copied;
  if (misses) *misses = h->misses;
  if (hits) *hits = h->hits;
  if (slot_group)
    for (int s = 0; s < h->slots; ++s) slot_group[s] = h->slot_group[s];
  return MOE_OK;
}

}  // extern "C"
