// Host-side launchers of libmoehier (internal to the library).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// Validated layer shape plus the group table, shared by every launcher.
struct LayerArgs {
  int T, d, f, E, G, K, kg, ke, k, r;
  bool bf16;        // act dtype BF16 (else FP32)
  bool int4;        // residual INT4 group-64 (else FP32)
  int R;            // rows = T * kg
  bool across;      // MOE_ROUTE_ACROSS: top k_e over the union of the chosen groups
  int wslots;       // group slots in the base arrays w_gate / w_up / w_down (G, or the cache size)
  GroupTable tab;
};

// Workspace carving (offsets in bytes from ws; every region 256-byte aligned).
struct Plan {
  size_t status, logits, redo, gidx, eidx, gate;
  size_t perm, inv_pos, ebeg, ecnt, gbeg, row_asg, row_of, rbeg;
  size_t cnt, off;   // per-block histograms and their exclusive offsets
  int nblk;          // permutation blocks
  size_t U, H, hsum, V, yrows;
  // tensor-core path
  bool tc;
  int krp, nchunks;
  size_t X, Ain, Bgs, Bus, Adt, Adn, Bdn, Ubf, Ud, hsum_bf, Vpart, Vt;
  size_t total;
};

Plan make_plan(const LayerArgs& a);

// Profiling marks (see moe_hier_profile_begin): call right after every kernel launch.
void prof_start(cudaStream_t st);
void prof_mark(const char* kernel_name, cudaStream_t st);

// Routing.  logits: [T][G+E] FP32 scratch; redo: [T] int32 scratch; status->route_redo must be
// zero on entry when status_zeroed (else it is cleared here).
cudaError_t launch_route(const LayerArgs& a, const void* x, const void* wg, const float* bg,
                         const void* we, float* logits, int32_t* redo, int32_t* gidx, int32_t* eidx,
                         float* gate, DevStatus* status, bool status_zeroed, cudaStream_t st);
// The tensor-core router with exact verification (route_tc.cu): writes the verified tokens and
// lists the others in redo[0 .. status->route_redo).
bool route_tc_ok(const LayerArgs& a);
int route_tc_columns(const LayerArgs& a);
// dbg (test aid): null, or [T][2 (G + E)] FP32 receiving each token's tensor-core logits (groups,
// then experts, bias included) and the verification half-widths delta of the same candidates.
cudaError_t launch_route_tc(const LayerArgs& a, const void* x, const void* wg, const float* bg, const void* we,
                            int32_t* gidx, int32_t* eidx, float* gate, int32_t* redo, DevStatus* status,
                            cudaStream_t st, float* dbg = nullptr);
// BF16 [rows][cols] tensor map, box {64, box_rows}, 128-byte swizzle (ffn_tc.cu).
bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);

struct PermOut {
  int32_t *perm, *inv_pos, *ebeg, *ecnt, *gbeg, *row_asg, *row_of, *rbeg;
};
// Limit of the cooperative permutation's grid-wide wait and the arrivals it expects beyond the
// permutation's own blocks (0 in normal use; a positive count makes the wait run out, which is how
// the failure path is tested without faulting or hanging the GPU).
struct PermWait {
  uint64_t limit_ns;
  unsigned int phantom;
};
constexpr PermWait kPermWaitDefault{2000000000ull, 0u};
cudaError_t launch_permute(const LayerArgs& a, const int32_t* eidx, const PermOut& o, int32_t* cnt,
                           int32_t* off, int nblk, DevStatus* status, bool bar_zeroed, cudaStream_t st,
                           PermWait wait = kPermWaitDefault);

struct ResidPtrs {
  ResidView A[3], B[3];
};
struct FfnBufs {
  float* U;      // [R][ke][2][r]
  float* H;      // [R][ke][f]
  float* hsum;   // [R][f]
  float* V;      // [R][ke][r]
};
cudaError_t launch_ffn_simt(const LayerArgs& a, const void* x, const void* wg, const void* wu,
                            const void* wd, const ResidPtrs& rp, const int32_t* eidx,
                            const float* gate, const int32_t* row_asg, const int32_t* row_begin,
                            void* y_rows, const FfnBufs& b, cudaStream_t st);

struct TcBufs {
  __nv_bfloat16 *X, *Ain;
  __half *Bgs, *Bus, *Adt;
  __nv_bfloat16 *Adn, *Bdn;
  __half* U;
  __nv_bfloat16 *hsum, *Vt;
  float* Vpart;
  __half* Ud;               // [T][G*2*KRP] U in token order (tc_u_dense)
};
bool tc_path_ok(const LayerArgs& a);
int tc_krp(const LayerArgs& a);
int tc_up_chunks(const LayerArgs& a);
cudaError_t launch_ffn_tc(const LayerArgs& a, const void* x, const void* wg, const void* wu, const void* wd,
                          const ResidPtrs& rp, const int32_t* eidx, const float* gate, const int32_t* row_asg,
                          const int32_t* row_begin, void* y_rows, const TcBufs& b, DevStatus* status,
                          cudaEvent_t prep_done, cudaStream_t st, bool prepared = false);
// The first step of launch_ffn_tc: the residual stacks (weights only; skipped with stacks = false,
// when the caller prepared them once) and, when tc_u_dense, U = A^T x of every token for every
// group.  launch_ffn_tc skips it when given prep_done, an event recorded after this call's work
// (it then waits for the event); with prepared = true it runs only the dense U GEMM itself.
cudaError_t launch_resid_prep(const LayerArgs& a, const ResidPtrs& rp, const TcBufs& b, const void* x,
                              DevStatus* status, cudaStream_t st, bool stacks = true);
// Whether U is computed densely, in token order for every group, with the residual stacks.
bool tc_u_dense(const LayerArgs& a);

cudaError_t launch_combine(const LayerArgs& a, const void* y_rows, void* y, cudaStream_t st);

// Compression step (compress.cu): one matrix kind of every expert.
struct CmpArgs {
  int E, G, d_out, d_in, r, l, power_iters;
  uint8_t member[kMaxE];     // member[g*K + i]: i-th expert (ascending id) of group g
  uint8_t group_of[kMaxE];
};
size_t cmp_workspace_bytes(const CmpArgs& c);
cudaError_t launch_compress(const CmpArgs& c, const void* W, const float* omega, void* base_out, uint8_t* Aq,
                            __half* As, uint8_t* Bq, __half* Bs, float* sigma, double* err, float* At_out,
                            float* Bt_out, void* ws, cudaStream_t st);
cudaError_t launch_quant_int4(const float* v, size_t rows, int n, uint8_t* codes, __half* scales, cudaStream_t st);

}  // namespace moe
