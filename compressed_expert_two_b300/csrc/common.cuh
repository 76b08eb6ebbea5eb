// Shared device helpers of libmoehier (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/moehier.h"

namespace moe {

// Programmatic dependent launch.  Every kernel of the layer is launched with programmatic stream
// serialization, so that its CTAs may be scheduled while the previous kernel drains.  Before its
// first global read or write a kernel waits for all prerequisite grids to complete
// (griddepcontrol.wait; a no-op when the launch had no programmatic dependency) and lets the next
// kernel be scheduled (griddepcontrol.launch_dependents).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, dim3 cluster,
                                             size_t smem, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster.x * cluster.y * cluster.z > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster.x;
    attr[1].val.clusterDim.y = cluster.y;
    attr[1].val.clusterDim.z = cluster.z;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                     Args&&... args) {
  return launch_pdl_cluster(kernel, grid, block, dim3(1, 1, 1), smem, st, std::forward<Args>(args)...);
}

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current device, once per device
// (`done` holds one bit per device index; the attribute belongs to the device, so a process that
// drives several GPUs sets it on each).  Setting it twice is harmless, so two host threads that
// race on a device's first launch only repeat the call.
template <typename K>
static inline cudaError_t smem_attr_once(K kernel, size_t bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

constexpr int kMaxE = 256;
constexpr int kMaxK = 16;     // k_g * k_e
constexpr int kMaxRank = 64;
constexpr int kQGroup = 64;   // INT4 elements per FP16 scale

// Group membership, passed to kernels by value (no device allocation for the host group map).
struct GroupTable {
  int E, G, K;
  uint8_t member[kMaxE];    // member[g*K + i] = i-th expert (ascending id) of group g
  uint8_t group_of[kMaxE];  // group of expert e
  uint8_t local_of[kMaxE];  // position of expert e inside its group
  uint8_t wslot[kMaxE];     // slot of group g's base matrices in the base arrays (g, unless the
                            // bases are offloaded and group g sits in cache slot wslot[g])
};

// Device status word at the start of every workspace (bounded waits report here).
struct DevStatus {
  int code;
  int where;
  unsigned int grid_bar;   // arrivals at the permutation's grid-wide barrier (zeroed before it)
  int route_redo;          // tokens the tensor-core router leaves to the canonical-order kernels
};

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Element c of an INT4 group-64 rank row (codes [n/2] bytes, scales [n/64] fp16).
__device__ __forceinline__ float int4_at(const uint8_t* codes, const __half* scales, int c) {
  const uint8_t b = codes[c >> 1];
  const int u = (c & 1) ? (b & 0xF) : (b >> 4);
  return (float)(u - 8) * __half2float(scales[c / kQGroup]);
}

// Residual factor element: rank row k of expert e, column c (n columns per rank row).
struct ResidView {
  const void* vals;     // F32 [E][r][n] or INT4 bytes [E][r][n/2]
  const __half* scales; // [E][r][n/64] (INT4)
  int n, r;
  bool int4;
  __device__ __forceinline__ float at(int e, int k, int c) const {
    const size_t row = (size_t)e * r + k;
    if (int4) return int4_at((const uint8_t*)vals + row * (n / 2), scales + row * (n / kQGroup), c);
    return ((const float*)vals)[row * n + c];
  }
};

// Two independent IEEE round-to-nearest FMAs in one instruction: (a.x*b.x + c.x, a.y*b.y + c.y).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long ra = *reinterpret_cast<unsigned long long*>(&a);
  unsigned long long rb = *reinterpret_cast<unsigned long long*>(&b);
  unsigned long long rc = *reinterpret_cast<unsigned long long*>(&c);
  unsigned long long rd;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  return *reinterpret_cast<float2*>(&rd);
}

// a.lo * b.lo + c and a.hi * b.hi + c for two BF16 values packed in a 32-bit word (low half =
// lower address), one rounding: the mixed-precision FMA of sm_100 and later.
__device__ __forceinline__ float fma_bf16_lo(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
      " fma.rn.f32.bf16 %0, al, bl, %3;\n}" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_bf16_hi(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
      " fma.rn.f32.bf16 %0, ah, bh, %3;\n}" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }
// SiLU from the fast exponential and reciprocal intrinsics (relative error ~1e-6); for z << 0
// the denominator overflows to +inf and the result is -0.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

}  // namespace moe
