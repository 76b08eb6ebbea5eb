/*
 * moehier.h -- C ABI of libmoehier.so: the forward pass of a clustered, compressed
 * Mixture-of-Experts layer on one NVIDIA B300 (sm_103a).
 *
 * The layer ("Breaking the MoE LLM Trilemma: Dynamic Expert Clustering with Structured
 * Compression", paper notes, overall framework and key designs 2-4):
 *   E experts are split into G groups of K = E/G.  Expert i of group g has, for each of its three
 *   matrices m in {gate, up, down}, the weight  W~_i = W_base^g + B_i A_i^T  (key design 2, W~
 *   equation), A_i in R^{d_in x r}, B_i in R^{d_out x r}; the base is BF16 (FP32 in the FP32
 *   format) and the residual INT4 (key design 4).  A token is routed to its top-k_g groups by the
 *   group router and, inside each chosen group, to that group's top-k_e experts by the expert
 *   router (key design 3).  The expert body is the SwiGLU FFN  W~_down (silu(W~_gate x) * W~_up x)
 *   and the layer output is the gated sum  y = sum_i G_i(x) E_i(x)  ("混合专家模型的路由机制与
 *   工程落地", section 1.2).  Gates: softmax over the k_g selected group logits times the softmax
 *   over the k_e selected expert logits inside the group ("MoE架构演进白皮书", chapter 1 top-2
 *   code: top-k of the logits, then softmax of the selected ones).  Dropless.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, except group_map_host (host
 *     memory, read during the call only).  Row-major, nn.Linear layout (W is [d_out][d_in]).
 *   - The library never allocates device memory, frees or synchronises (except
 *     moe_hier_get_status, which synchronises the given stream).  Work is enqueued on `stream`
 *     (a cudaStream_t; NULL = the legacy default stream) and the call returns.  moe_hier_forward
 *     also runs its weight-only step (the residual stacks) on a second stream that it creates,
 *     with two events, on its first call in a host thread (per device); the work forks from and
 *     rejoins `stream` through those events, so it is also captured by a CUDA graph capture of
 *     `stream`.  Scratch memory is the caller's workspace
 *     `ws` of `ws_bytes` bytes (>= moe_hier_workspace_size), 256-byte aligned.  Calls that share
 *     a workspace must be ordered on one stream; distinct workspaces may run concurrently.
 *   - Return value: MOE_OK, or a negative moe_status.  MOE_ERR_INVALID / _UNSUPPORTED /
 *     _WORKSPACE are detected on the host before anything is enqueued.  MOE_ERR_CUDA means a
 *     launch failed (cudaGetLastError); earlier steps of the call may already be enqueued.
 *     Conditions found on the device (a bounded wait that ran out) are written to a status word
 *     in the workspace and reported by moe_hier_get_status.  moe_hier_forward clears the word
 *     when it starts; the stand-alone calls only set it, so a caller that uses them alone
 *     clears it by zeroing the first 16 bytes of `ws` (a zero-filled workspace starts clear).
 *   - Inputs must be finite; NaN logits give unspecified routing.
 *   - Device arrays start on 16-byte boundaries (as cudaMalloc and PyTorch allocations do);
 *     x, y, the weights and the residual codes are checked (MOE_ERR_INVALID otherwise).
 *
 * Shapes (T tokens, d = d_model, f = d_ff, k = k_g * k_e routed experts per token)
 *   x         [T][d]            act dtype          y [T][d] act dtype
 *   w_group   [G][d]            act dtype          b_group [G] float32 or NULL
 *   w_expert  [E][d]            act dtype          group_map_host [E] int32, exactly K per group
 *   w_gate, w_up [G][f][d]      act dtype          w_down [G][d][f] act dtype
 *   residual of matrix m (0 gate, 1 up, 2 down), d_in/d_out = (d,f), (d,f), (f,d):
 *     A[m] = A^T rank-major [E][r][d_in],  B[m] = B^T rank-major [E][r][d_out]
 *     MOE_RESID_F32:      float32 values; sA/sB unused (NULL)
 *     MOE_RESID_INT4_G64: uint8 [E][r][n/2], element 2j in the HIGH nibble and 2j+1 in the LOW
 *       nibble of byte j, value = (nibble - 8) * scale, one FP16 scale per 64 consecutive
 *       elements: sA[m] [E][r][d_in/64], sB[m] [E][r][d_out/64] ("MoE架构演进白皮书" section 3.2
 *       unpack convention: even offset high nibble, zero point 8).
 *   Routing outputs: gidx [T][k_g] int32 (best group first); eidx [T][k] int32 global expert ids,
 *     slot = group rank * k_e + expert rank (best first); gate [T][k] float32.
 *   Router arithmetic ("混合专家模型的路由机制与工程落地" section 3.1: the router runs in FP32),
 *     in a fixed order so indices are reproducible: 32 partial sums, partial l owning the
 *     elements i with (i mod 128) div 4 == l added in ascending i (fl32 product, fl32 add), then
 *     s_l += s_{l xor o} for o = 16, 8, 4, 2, 1; logit = fl32(s_0 + b).  Ties: lower index first.
 */
#ifndef MOEHIER_H
#define MOEHIER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = -1,      /* bad shape, pointer, group map or descriptor                    */
  MOE_ERR_UNSUPPORTED = -2,  /* valid layer, but no kernel for this dtype / format / size       */
  MOE_ERR_WORKSPACE = -3,    /* ws NULL, misaligned, or smaller than moe_hier_workspace_size    */
  MOE_ERR_CUDA = -4,         /* a CUDA launch or runtime call failed                           */
  MOE_ERR_TIMEOUT = -5       /* a bounded device-side wait ran out (reported via get_status)   */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;
typedef enum { MOE_RESID_F32 = 0, MOE_RESID_INT4_G64 = 1 } moe_resid_fmt;
/* Level-2 routing ("Breaking the MoE LLM Trilemma", key design 3).
 *   MOE_ROUTE_WITHIN: the top-k_e experts inside each chosen group (k_g k_e active experts),
 *     gate = p_g q_e (softmax over the chosen group logits times the softmax over the group's
 *     chosen expert logits).
 *   MOE_ROUTE_ACROSS: the top-k_e experts over the union of the chosen groups' members (k_e active
 *     experts), gate = softmax over their logits.  The slot layout stays the within-group one --
 *     eidx holds each chosen group's top-k_e members, which contain every expert the union's
 *     top-k_e picks -- and the slots it does not pick get gate 0, so they add nothing to y. */
typedef enum { MOE_ROUTE_WITHIN = 0, MOE_ROUTE_ACROSS = 1 } moe_route_mode;

typedef struct {
  int32_t T, d_model, d_ff, E, G;
  int32_t topk_group;   /* k_g, 1 <= k_g <= G                                                  */
  int32_t topk_expert;  /* k_e, 1 <= k_e <= K = E/G (per chosen group)                         */
  int32_t rank;         /* r >= 0; r == 0 means no residual (residual pointers may be NULL)      */
  int32_t act_dtype;    /* moe_dtype of x, y, routers and base weights                           */
  int32_t resid_fmt;    /* moe_resid_fmt                                                         */
  int32_t route_mode;   /* moe_route_mode (0, the within-group reading, when zero-initialised)    */
} moe_hier_desc;
/* Limits: T >= 0; d_model % 128 == 0; d_ff % 64 == 0; E % G == 0; E <= 256; k_e*k_g <= 16;
 * r <= 64.  INT4 residuals need a BF16 layer, F32 residuals an F32 layer.                    */

typedef struct {
  const void* A[3];   /* gate, up, down: A^T [E][r][d_in]  (F32 values or packed INT4)         */
  const void* B[3];   /* gate, up, down: B^T [E][r][d_out]                                      */
  const void* sA[3];  /* FP16 scales of A (INT4 only)                                           */
  const void* sB[3];  /* FP16 scales of B (INT4 only)                                           */
} moe_hier_resid;

/* Bytes of workspace the calls below need for this layer (0 on an invalid descriptor; then
 * *status_out, if non-NULL, holds the reason). */
size_t moe_hier_workspace_size(const moe_hier_desc* desc, int* status_out);

/* Level-1 and level-2 routing ("Breaking the MoE LLM Trilemma", key design 3).
 * Writes gidx, eidx and gate (shapes above).  Uses the workspace for the logits and, on the
 * tensor-core path (BF16, T >= 1024, router rows beyond what the fused kernel holds), for the
 * list of tokens whose decision the tensor-core logits do not settle provably: those are
 * recomputed in the canonical FP32 order, so the indices are the canonical ones in every case;
 * the gates of the other tokens come from the tensor-core logits (another FP32 summation order,
 * "router in FP32", routing-mechanisms page §3.1). */
int moe_hier_route(const moe_hier_desc* desc, const void* x, const void* w_group,
                   const float* b_group, const void* w_expert, const int32_t* group_map_host,
                   int32_t* gidx, int32_t* eidx, float* gate,
                   void* ws, size_t ws_bytes, void* stream);

/* Single-device form of the two-level dispatch (key design 3): stable counting sorts.
 *   Assignments a = t*k + slot, ordered by key (group, expert, token):
 *     perm [T*k] (position -> a), inv_pos [T*k] (a -> position),
 *     expert_begin [E], expert_count [E] (indexed by expert id), group_begin [G+1].
 *   (token, group-slot) rows b = t*k_g + j, ordered by key (group, token):
 *     row_asg [T*k_g] (position -> b), row_of [T*k_g] (b -> position), row_begin [G+1].
 * Every output is exact (integers, deterministic).  Any output pointer except row_asg and
 * row_begin may be NULL to skip it. */
int moe_hier_permute(const moe_hier_desc* desc, const int32_t* group_map_host, const int32_t* eidx,
                     int32_t* perm, int32_t* inv_pos, int32_t* expert_begin, int32_t* expert_count,
                     int32_t* group_begin, int32_t* row_asg, int32_t* row_of, int32_t* row_begin,
                     void* ws, size_t ws_bytes, void* stream);

/* Expert computation with base reuse (key design 2: W~ x = W_base x + B (A^T x), the base term
 * computed once per (token, group) and shared by the group's experts on that token), SwiGLU
 * and gating.  For each row (t, j) in row_asg order with group g and experts e_s (s < k_e):
 *   y_rows[t][j] = sum_s gate[t][j*k_e+s] * W~_down,e_s (silu(W~_gate,e_s x_t) * W~_up,e_s x_t)
 * y_rows is [T][k_g][d] in TOKEN order (act dtype); with k_g == 1 it can be y itself.
 * row_asg / row_begin come from moe_hier_permute. */
int moe_hier_ffn(const moe_hier_desc* desc, const void* x, const int32_t* group_map_host,
                 const void* w_gate, const void* w_up, const void* w_down,
                 const moe_hier_resid* resid, const int32_t* eidx, const float* gate,
                 const int32_t* row_asg, const int32_t* row_begin, void* y_rows,
                 void* ws, size_t ws_bytes, void* stream);

/* y[t] = sum_{j < k_g} y_rows[t][j] (slot order), act dtype in and out, FP32 sum
 * ("混合专家模型的路由机制与工程落地" section 1.2 combine).  y may alias y_rows when k_g == 1. */
int moe_hier_combine(const moe_hier_desc* desc, const void* y_rows, void* y, void* stream);

/* The whole layer: route -> permute -> ffn -> combine, enqueued back to back.
 * gidx_opt, eidx_opt, gate_opt, perm_opt (may be NULL) receive copies of the routing results. */
int moe_hier_forward(const moe_hier_desc* desc, const void* x, const void* w_group,
                     const float* b_group, const void* w_expert, const int32_t* group_map_host,
                     const void* w_gate, const void* w_up, const void* w_down,
                     const moe_hier_resid* resid, void* y,
                     int32_t* gidx_opt, int32_t* eidx_opt, float* gate_opt, int32_t* perm_opt,
                     void* ws, size_t ws_bytes, void* stream);

/* Prepared residual stacks.  The tensor-core path multiplies FP16/BF16 stacks of the residual
 * factors that it builds from the INT4 codes (weights only: they do not depend on the tokens).
 * moe_hier_forward rebuilds them on every call, overlapped with routing; a caller that runs the
 * same layer many times (decode) builds them once with moe_hier_prepare into a buffer of
 * moe_hier_prepared_size bytes (device, 256-byte aligned, owned by the caller) and calls
 * moe_hier_forward_prepared, which reads them from there and skips the rebuild.  The stacks' form
 * depends on the descriptor (which kernels a batch of T tokens uses), so prepare with the
 * descriptor the forward calls use, and again after the residual factors change.  Results equal
 * moe_hier_forward's bit for bit.  BF16 layers with INT4 residuals only (MOE_ERR_UNSUPPORTED
 * otherwise); MOE_ERR_WORKSPACE if prep is missing, misaligned or too small. */
size_t moe_hier_prepared_size(const moe_hier_desc* desc, int* status_out);
int moe_hier_prepare(const moe_hier_desc* desc, const int32_t* group_map_host, const moe_hier_resid* resid,
                     void* prep, size_t prep_bytes, void* stream);
int moe_hier_forward_prepared(const moe_hier_desc* desc, const void* x, const void* w_group,
                              const float* b_group, const void* w_expert, const int32_t* group_map_host,
                              const void* w_gate, const void* w_up, const void* w_down,
                              const moe_hier_resid* resid, const void* prep, size_t prep_bytes, void* y,
                              int32_t* gidx_opt, int32_t* eidx_opt, float* gate_opt, int32_t* perm_opt,
                              void* ws, size_t ws_bytes, void* stream);

/* Synchronises `stream`, then returns the device status word of `ws` (MOE_OK or
 * MOE_ERR_TIMEOUT), or MOE_ERR_CUDA if the stream reported an error. */
int moe_hier_get_status(const void* ws, void* stream);

/* Static text for a moe_status value. */
const char* moe_hier_status_string(int status);

/* Static text of the last CUDA error that an entry point called on this host thread reported as
 * MOE_ERR_CUDA ("no error" if none).  A diagnostic aid without a counterpart in the pages. */
const char* moe_hier_last_cuda_error(void);

/* Profiling aid (the pages have no counterpart; it changes no result).  After
 * moe_hier_profile_begin(events, n), the entry points called on this host thread record
 * events[0] on their stream before their first kernel and events[i] right after their i-th
 * kernel launch (i = 1 .. n-1; later launches are not marked).  `events` are cudaEvent_t
 * handles owned by the caller.  moe_hier_profile_end stops recording and returns the number of
 * kernels launched since begin; names[i] (i < max_names, names may be NULL) receives a static
 * string naming the i-th kernel.  Kernel i ran between events[i] and events[i+1]. */
int moe_hier_profile_begin(void* const* events, int n_events);
int moe_hier_profile_end(const char** names, int max_names);

/* ---------------------------------------------------------------------------------------------
 * Compression: the step that produces a layer's weights from dense experts ("Breaking the MoE
 * LLM Trilemma", key design 2: the group's shared base is the mean of its experts' weights, each
 * expert keeps a rank-r residual initialised by a truncated SVD of W_i - W_base^g, quality is the
 * Frobenius reconstruction error; key design 4: 16-bit base, INT4 residual).  One call handles
 * one matrix kind (gate, up or down) of every expert.
 *   base[g] = bf16(fl32(sum over the group's members, ascending id, of W_i) / K) (FP32 adds,
 *     round to nearest even);
 *   R_i = W_i - base[g(i)] (the stored base); its best rank-r approximation B_i A_i^T, computed by a
 *     randomised range finder with `power_iters` subspace iterations on `sketch` columns (the
 *     Gaussian test matrix omega is an input), split evenly: B = U_r S^{1/2}, A = V_r S^{1/2};
 *   A^T [E][r][d_in] and B^T [E][r][d_out] stored in the layer's INT4 group-64 format: scale =
 *     fp16(absmax/7), code = clamp(rint(w/scale), -7, 7) + 8 (FP32 decisions), element 2j in the
 *     high nibble of byte j -- the moe_hier_resid layout of that matrix kind;
 *   sigma [E][r] the singular values kept; err [E] (nullable) ||W_i - (base + B A^T)||_F / ||W_i||_F
 *     with A, B dequantised from the stored codes (FP64).
 * Shapes: W [E][d_out][d_in] BF16 (device), omega [d_in][sketch] FP32 (device), group_map_host
 * [E] int32 (host, exactly E/G experts per group), base [G][d_out][d_in] BF16 (device);
 * At_f32 [E][r][d_in], Bt_f32 [E][r][d_out] FP32 (device, nullable): the factors before
 * quantisation.  Limits: E % G == 0, E <= 256, d_in and d_out multiples of 128, 1 <= rank <= 32,
 * rank < sketch <= 64, 0 <= power_iters <= 16.  MOE_ERR_INVALID / _WORKSPACE as elsewhere. */
typedef struct {
  int32_t E, G;
  int32_t d_out, d_in;   /* the matrix kind's shape: W_i is [d_out][d_in]                        */
  int32_t rank;          /* r kept                                                               */
  int32_t sketch;        /* l = r + oversampling, columns of the test matrix                      */
  int32_t power_iters;   /* subspace iterations                                                  */
} moe_hier_compress_desc;

size_t moe_hier_compress_workspace_size(const moe_hier_compress_desc* desc, int* status_out);
int moe_hier_compress(const moe_hier_compress_desc* desc, const void* w, const int32_t* group_map_host,
                      const float* omega, void* base, void* A_codes, void* A_scales, void* B_codes,
                      void* B_scales, float* sigma, double* err, float* At_f32, float* Bt_f32,
                      void* ws, size_t ws_bytes, void* stream);

/* INT4 group-64 quantisation alone (the rule of moe_hier_compress): v [rows][n] FP32 (device,
 * n % 64 == 0) -> codes [rows][n/2] uint8, scales [rows][n/64] FP16 (device). */
int moe_hier_quantise_int4(const float* v, int64_t rows, int32_t n, void* codes, void* scales, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Idle-group offload ("Breaking the MoE LLM Trilemma", key design 4: groups the current work does
 * not use are moved to CPU memory and brought back when needed).  The caller keeps the three base
 * arrays of every group in PINNED host memory (w_gate_host, w_up_host [G][f][d], w_down_host
 * [G][d][f], BF16, e.g. from cudaHostAlloc or cudaHostRegister) and provides a device cache of
 * `slots` groups (cache_gate, cache_up [slots][f][d], cache_down [slots][d][f]).  The handle is
 * host memory only (plus 2 * slots CUDA events); it belongs to the device current at creation.
 * BF16 layers with INT4 residuals (the tensor-core path) only: MOE_ERR_UNSUPPORTED otherwise.
 *
 * Per batch, with x, the routers and the residual factors resident as usual:
 *   moe_hier_route, moe_hier_permute      (compute stream; row_begin as usual)
 *   moe_hier_groups_hit                   copies row_begin to the host and synchronises that
 *                                         stream: hit_host[g] = 1 if the batch has rows in g;
 *   moe_hier_offload_require              every hit group not in the cache gets a slot (an empty
 *                                         one, else the least recently used slot whose group is
 *                                         not hit) and its three matrices are copied host->device
 *                                         on copy_stream, after the last FFN that read that slot
 *                                         has finished; *copied (nullable) = groups copied.
 *                                         MOE_ERR_INVALID if the batch hits more groups than slots;
 *   moe_hier_ffn_offload                  moe_hier_ffn with the bases read from the cache: the
 *                                         stream waits for the hit groups' copies, then the FFN
 *                                         kernels run; a group that was not required reads zeros.
 *   moe_hier_combine                      as usual.
 * The next batch's route / permute / groups_hit / require may be issued while this batch's FFN
 * runs (the copy stream waits on the slots' last readers).  One handle is used from one host
 * thread at a time.  Results equal moe_hier_ffn's on resident bases bit for bit. */
typedef struct moe_hier_offload moe_hier_offload;

int moe_hier_offload_create(const moe_hier_desc* desc, const void* w_gate_host, const void* w_up_host,
                            const void* w_down_host, void* cache_gate, void* cache_up, void* cache_down,
                            int32_t slots, moe_hier_offload** out);
int moe_hier_offload_destroy(moe_hier_offload* handle);
int moe_hier_groups_hit(const moe_hier_desc* desc, const int32_t* row_begin, int32_t* hit_host, void* stream);
int moe_hier_offload_require(moe_hier_offload* handle, const int32_t* hit_host, int32_t* copied,
                             void* copy_stream);
int moe_hier_ffn_offload(moe_hier_offload* handle, const moe_hier_desc* desc, const void* x,
                         const int32_t* group_map_host, const moe_hier_resid* resid, const int32_t* eidx,
                         const float* gate, const int32_t* row_asg, const int32_t* row_begin, void* y_rows,
                         void* ws, size_t ws_bytes, void* stream);
/* Totals since creation: bytes copied host->device, groups copied (misses), hit groups found in
 * the cache (hits); slot_group (nullable, [slots]) = the group each slot holds (-1: empty). */
int moe_hier_offload_stats(const moe_hier_offload* handle, uint64_t* bytes_copied, uint64_t* misses,
                           uint64_t* hits, int32_t* slot_group);

/* Test aids.  The pages have no counterpart; neither changes a result of the calls above.
 *
 * moe_hier_debug_set_wait sets, for the calling process, the limit of the grid-wide wait inside
 * the single-launch form of moe_hier_permute (batches of more than 1024 tokens; default 2 s;
 * wait_ns = 0 keeps the default) and a number of arrivals that the wait expects beyond the
 * launch's own blocks (default 0).  With phantom_arrivals > 0 the wait cannot complete: every
 * block gives up after the limit, writes MOE_ERR_TIMEOUT to the workspace status word (read it
 * with moe_hier_get_status) and returns without placing its items, so that call's outputs are
 * unspecified and the stream stays usable.  This drives the failure path of a bounded device
 * wait without faulting or hanging the GPU.  Only moe_hier_permute reads the setting
 * (moe_hier_forward always runs with the defaults); moe_hier_debug_set_wait(0, 0) restores them.
 * MOE_ERR_INVALID if phantom_arrivals < 0. */
int moe_hier_debug_set_wait(uint64_t wait_ns, int phantom_arrivals);

/* Runs the tensor-core router alone (BF16 layers with T >= 1024, at most 128 router columns
 * after padding the group rows to 8, k_g and k_e <= 8; MOE_ERR_UNSUPPORTED otherwise) and writes,
 * for every token t, out[t][0 .. G+E) = its FP32 tensor-core logits (group logits with the bias,
 * then expert logits) and out[t][G+E .. 2(G+E)) = the half-widths delta of the intervals the
 * router verified its decision with, for the same candidates.  out: device, [T][2(G+E)] FP32.
 * The routing results go to the workspace.  With it a test checks the router's bound
 * |s_tc - s_canonical| <= delta element by element ("router in FP32", routing-mechanisms page
 * section 3.1, is what makes the canonical logits the reference). */
int moe_hier_debug_route_tc(const moe_hier_desc* desc, const void* x, const void* w_group,
                            const float* b_group, const void* w_expert, const int32_t* group_map_host,
                            float* out, void* ws, size_t ws_bytes, void* stream);

/* moe_hier_permute for callers that cannot supply a workspace: a host that owns all device
 * memory through its own pool and allows no other allocation, or a latency-critical loop that
 * may not pay an allocation's implicit device synchronisation.  The paper has no counterpart;
 * this is a deployment convenience.  Arguments and outputs are those of moe_hier_permute,
 * without ws/ws_bytes.  The scratch (per-block histograms and offsets) is a fixed array of
 * 65,536 int32 (256 KiB) inside the library, held by every GPU that loads the library until the
 * process exits; a layer needs 2 * ceil(T/256) * (E + G) of them, and larger layers are rejected
 * with MOE_ERR_WORKSPACE before anything is enqueued (batches of at most 1024 tokens are
 * permuted by a single-CTA kernel that uses no scratch).  The call allocates nothing.  The first
 * call on a device looks up the array's device address (with that device current) and keeps it
 * for the life of the process; make that first call before any stream capture, and do not call
 * cudaDeviceReset on a device between calls (a reset would leave the kept address stale).  All calls share the one array and each kernel
 * overwrites every entry it later reads, so nothing needs clearing between calls, but calls
 * whose work overlaps on the GPU (other streams, other host threads) race on it. */
int moe_hier_permute_noalloc(const moe_hier_desc* desc, const int32_t* group_map_host,
                             const int32_t* eidx, int32_t* perm, int32_t* inv_pos,
                             int32_t* expert_begin, int32_t* expert_count, int32_t* group_begin,
                             int32_t* row_asg, int32_t* row_of, int32_t* row_begin, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOEHIER_H */
