// C ABI of libmoehier: descriptor validation, workspace planning and launch sequencing.
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// ---- profiling marks (per host thread) ----
static thread_local void* const* g_prof_ev = nullptr;
static thread_local int g_prof_n = 0, g_prof_i = 0, g_prof_launches = 0;
static thread_local const char* g_prof_names[256];

void prof_start(cudaStream_t st) {
  if (g_prof_ev && g_prof_i == 0 && g_prof_n > 0) {
    cudaEventRecord((cudaEvent_t)g_prof_ev[0], st);
    g_prof_i = 1;
  }
}

void prof_mark(const char* name, cudaStream_t st) {
  if (!g_prof_ev) return;
  if (g_prof_launches < 256) g_prof_names[g_prof_launches] = name;
  ++g_prof_launches;
  if (g_prof_i > 0 && g_prof_i < g_prof_n) cudaEventRecord((cudaEvent_t)g_prof_ev[g_prof_i++], st);
}

static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

Plan make_plan(const LayerArgs& a) {
  Plan p{};
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
  const size_t T = a.T, R = a.R, k = a.k, E = a.E, G = a.G;
  p.status = take(sizeof(DevStatus));
  p.logits = take(T * (G + E) * 4);
  p.redo = take(T * 4);
  p.gidx = take(T * a.kg * 4);
  p.eidx = take(T * k * 4);
  p.gate = take(T * k * 4);
  p.perm = take(T * k * 4);
  p.inv_pos = take(T * k * 4);
  p.ebeg = take(E * 4);
  p.ecnt = take(E * 4);
  p.gbeg = take((G + 1) * 4);
  p.row_asg = take(R * 4);
  p.row_of = take(R * 4);
  p.rbeg = take((G + 1) * 4);
  p.nblk = (a.T + 255) / 256;
  p.cnt = take((size_t)p.nblk * (E + G) * 4);
  p.off = take((size_t)p.nblk * (E + G) * 4);
  p.tc = tc_path_ok(a);
  if (p.tc) {
    const size_t Rp = R < 128 ? 128 : R, KRP = tc_krp(a), d = a.d, f = a.f;
    p.krp = (int)KRP;
    p.nchunks = tc_up_chunks(a);
    p.X = take(Rp * d * 2);
    p.Ain = take(G * 4 * KRP * d * 2);
    p.Bgs = take(G * f * KRP * 2);
    p.Bus = take(G * f * KRP * 2);
    p.Adt = take(G * f * KRP * 2);
    p.Adn = take(G * KRP * f * 2);
    p.Bdn = take(G * d * 2 * KRP * 2);
    p.Ubf = take(Rp * 2 * KRP * 2);
    p.Ud = take(tc_u_dense(a) ? T * G * 2 * KRP * 2 : 0);
    p.hsum_bf = take(Rp * f * 2);
    p.Vpart = take((size_t)p.nchunks * 2 * R * a.ke * a.r * 4);   // up to two partials per chunk
    p.Vt = take(Rp * 2 * KRP * 2);
  } else {
    p.U = take(R * a.ke * 2 * a.r * 4);
    p.H = take(R * a.ke * (size_t)a.f * 4);
    p.hsum = take(R * (size_t)a.f * 4);
    p.V = take(R * a.ke * a.r * 4);
  }
  p.yrows = take(a.kg > 1 ? T * a.kg * (size_t)a.d * (a.bf16 ? 2 : 4) : 0);
  p.total = o;
  return p;
}

// Host-side validation of the descriptor and group map; fills the kernel argument block.
static int validate(const moe_hier_desc* desc, const int32_t* group_map, LayerArgs* a) {
  if (!desc) return MOE_ERR_INVALID;
  const moe_hier_desc& D = *desc;
  if (D.T < 0 || D.d_model <= 0 || D.d_ff <= 0 || D.E <= 0 || D.G <= 0) return MOE_ERR_INVALID;
  if (D.E % D.G != 0 || D.E > kMaxE) return MOE_ERR_INVALID;
  const int K = D.E / D.G;
  if (D.topk_group < 1 || D.topk_group > D.G) return MOE_ERR_INVALID;
  if (D.topk_expert < 1 || D.topk_expert > K) return MOE_ERR_INVALID;
  if (D.topk_group * D.topk_expert > kMaxK) return MOE_ERR_UNSUPPORTED;
  if (K > 32) return MOE_ERR_UNSUPPORTED;
  if (D.d_model % 128 != 0 || D.d_ff % 64 != 0) return MOE_ERR_INVALID;
  if (D.rank < 0) return MOE_ERR_INVALID;
  if (D.rank > kMaxRank) return MOE_ERR_UNSUPPORTED;
  if (D.act_dtype != MOE_F32 && D.act_dtype != MOE_BF16) return MOE_ERR_INVALID;
  if (D.resid_fmt != MOE_RESID_F32 && D.resid_fmt != MOE_RESID_INT4_G64) return MOE_ERR_INVALID;
  if ((D.act_dtype == MOE_BF16) != (D.resid_fmt == MOE_RESID_INT4_G64)) return MOE_ERR_UNSUPPORTED;
  if (D.route_mode != MOE_ROUTE_WITHIN && D.route_mode != MOE_ROUTE_ACROSS) return MOE_ERR_INVALID;
  memset(a, 0, sizeof(*a));
  a->T = D.T; a->d = D.d_model; a->f = D.d_ff; a->E = D.E; a->G = D.G; a->K = K;
  a->kg = D.topk_group; a->ke = D.topk_expert; a->k = a->kg * a->ke; a->r = D.rank;
  a->bf16 = D.act_dtype == MOE_BF16;
  a->int4 = D.resid_fmt == MOE_RESID_INT4_G64;
  a->R = a->T * a->kg;
  a->across = D.route_mode == MOE_ROUTE_ACROSS;
  a->wslots = D.G;
  for (int g = 0; g < D.G; ++g) a->tab.wslot[g] = (uint8_t)g;
  a->tab.E = D.E; a->tab.G = D.G; a->tab.K = K;
  if (group_map) {
    int fill[kMaxE];
    for (int g = 0; g < D.G; ++g) fill[g] = 0;
    for (int e = 0; e < D.E; ++e) {
      const int g = group_map[e];
      if (g < 0 || g >= D.G || fill[g] >= K) return MOE_ERR_INVALID;
      a->tab.member[g * K + fill[g]] = (uint8_t)e;   // ascending e inside each group
      a->tab.group_of[e] = (uint8_t)g;
      a->tab.local_of[e] = (uint8_t)fill[g];
      ++fill[g];
    }
  }
  return MOE_OK;
}

static int check_ws(const Plan& p, void* ws, size_t ws_bytes) {
  if (!ws || ((uintptr_t)ws & 255) != 0 || ws_bytes < p.total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

template <typename P> static P* at(void* ws, size_t off) { return (P*)((char*)ws + off); }

static ResidPtrs resid_ptrs(const LayerArgs& a, const moe_hier_resid* r) {
  ResidPtrs rp{};
  const int din[3] = {a.d, a.d, a.f}, dout[3] = {a.f, a.f, a.d};
  for (int m = 0; m < 3; ++m) {
    rp.A[m] = ResidView{r ? r->A[m] : nullptr, r ? (const __half*)r->sA[m] : nullptr, din[m], a.r, a.int4};
    rp.B[m] = ResidView{r ? r->B[m] : nullptr, r ? (const __half*)r->sB[m] : nullptr, dout[m], a.r, a.int4};
  }
  return rp;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

static bool resid_ok(const LayerArgs& a, const moe_hier_resid* r) {
  if (a.r == 0) return true;
  if (!r) return false;
  for (int m = 0; m < 3; ++m) {
    if (!r->A[m] || !r->B[m] || !aligned16(r->A[m]) || !aligned16(r->B[m])) return false;
    if (a.int4 && (!r->sA[m] || !r->sB[m])) return false;
  }
  return true;
}

// The residual stacks of the tensor-core path (weights only) in a buffer of their own: the
// regions a workspace would hold, at offsets relative to that buffer.
struct StackLayout {
  size_t Ain, Bgs, Bus, Adt, Adn, Bdn, total;
};
static StackLayout stack_layout(const Plan& p) {
  StackLayout l;
  l.Ain = 0;
  l.Bgs = p.Bgs - p.Ain;
  l.Bus = p.Bus - p.Ain;
  l.Adt = p.Adt - p.Ain;
  l.Adn = p.Adn - p.Ain;
  l.Bdn = p.Bdn - p.Ain;
  l.total = p.Ubf - p.Ain;          // the stacks are consecutive in the plan, Ubf follows them
  return l;
}

// Workspace pointers of the tensor-core path; with `prep` the residual stacks come from there.
static TcBufs tc_bufs(const Plan& p, void* ws, void* prep = nullptr) {
  TcBufs b{at<__nv_bfloat16>(ws, p.X),   at<__nv_bfloat16>(ws, p.Ain),    at<__half>(ws, p.Bgs),
           at<__half>(ws, p.Bus),        at<__half>(ws, p.Adt),           at<__nv_bfloat16>(ws, p.Adn),
           at<__nv_bfloat16>(ws, p.Bdn),
           at<__half>(ws, p.Ubf), at<__nv_bfloat16>(ws, p.hsum_bf), at<__nv_bfloat16>(ws, p.Vt),
           at<float>(ws, p.Vpart), at<__half>(ws, p.Ud)};
  if (prep) {
    const StackLayout l = stack_layout(p);
    b.Ain = at<__nv_bfloat16>(prep, l.Ain);
    b.Bgs = at<__half>(prep, l.Bgs);
    b.Bus = at<__half>(prep, l.Bus);
    b.Adt = at<__half>(prep, l.Adt);
    b.Adn = at<__nv_bfloat16>(prep, l.Adn);
    b.Bdn = at<__nv_bfloat16>(prep, l.Bdn);
  }
  return b;
}

static cudaError_t run_ffn(const LayerArgs& a, const Plan& p, void* ws, const void* x, const void* wg,
                           const void* wu, const void* wd, const moe_hier_resid* resid, const int32_t* eidx,
                           const float* gate, const int32_t* row_asg, const int32_t* row_begin, void* y_rows,
                           cudaEvent_t prep_done, cudaStream_t s, void* prep = nullptr) {
  if (p.tc)
    return launch_ffn_tc(a, x, wg, wu, wd, resid_ptrs(a, resid), eidx, gate, row_asg, row_begin, y_rows,
                         tc_bufs(p, ws, prep), at<DevStatus>(ws, p.status), prep_done, s, prep != nullptr);
  FfnBufs b{at<float>(ws, p.U), at<float>(ws, p.H), at<float>(ws, p.hsum), at<float>(ws, p.V)};
  return launch_ffn_simt(a, x, wg, wu, wd, resid_ptrs(a, resid), eidx, gate, row_asg, row_begin, y_rows, b, s);
}

// moe_hier_forward enqueues the weight-only residual preparation on a second stream, so that it
// runs while the tokens are routed and permuted.  One such stream and two events per host thread
// and device, created on first use and kept until the thread exits (no device memory).
struct SideStream {
  int dev = -1;
  cudaStream_t st = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  ~SideStream() {
    if (join) cudaEventDestroy(join);
    if (fork) cudaEventDestroy(fork);
    if (st) cudaStreamDestroy(st);
  }
};
static thread_local SideStream g_side;

static SideStream* side_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (g_side.st && g_side.dev == dev) return &g_side;
  if (g_side.st) return nullptr;                    // created for another device: run serially
  if (cudaStreamCreateWithFlags(&g_side.st, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&g_side.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&g_side.join, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  g_side.dev = dev;
  return &g_side;
}

// Test setting of the permutation's grid-wide wait (moe_hier_debug_set_wait); read by
// moe_hier_permute only.
static std::atomic<uint64_t> g_wait_ns{0};
static std::atomic<unsigned int> g_wait_phantom{0};

static PermWait perm_wait_setting() {
  PermWait w = kPermWaitDefault;
  const uint64_t ns = g_wait_ns.load(std::memory_order_relaxed);
  if (ns) w.limit_ns = ns;
  w.phantom = g_wait_phantom.load(std::memory_order_relaxed);
  return w;
}

// The last CUDA error a call of this host thread returned as MOE_ERR_CUDA.
static thread_local cudaError_t g_last_cuda_error = cudaSuccess;

static int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  g_last_cuda_error = e;
  return MOE_ERR_CUDA;
}

static int forward_impl(const moe_hier_desc* desc, const void* x, const void* w_group, const float* b_group,
                        const void* w_expert, const int32_t* group_map_host, const void* w_gate, const void* w_up,
                        const void* w_down, const moe_hier_resid* resid, void* prep, size_t prep_bytes, void* y,
                        int32_t* gidx_opt, int32_t* eidx_opt, float* gate_opt, int32_t* perm_opt, void* ws,
                        size_t ws_bytes, void* stream) {
  LayerArgs a;
  if (!group_map_host) return MOE_ERR_INVALID;
  int st = validate(desc, group_map_host, &a);
  if (st != MOE_OK) return st;
  if (a.T > 0 && (!x || !w_group || !w_expert || !w_gate || !w_up || !w_down || !y ||
                  !resid_ok(a, resid)))
    return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(w_group) || !aligned16(w_expert) || !aligned16(w_gate) || !aligned16(w_up) ||
      !aligned16(w_down) || !aligned16(y))
    return MOE_ERR_INVALID;
  const Plan p = make_plan(a);
  if ((st = check_ws(p, ws, ws_bytes)) != MOE_OK) return st;
  if (prep) {
    if (!p.tc) return MOE_ERR_UNSUPPORTED;
    if (((uintptr_t)prep & 255) != 0 || prep_bytes < stack_layout(p).total) return MOE_ERR_WORKSPACE;
  }
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* gidx = gidx_opt ? gidx_opt : at<int32_t>(ws, p.gidx);
  int32_t* eidx = eidx_opt ? eidx_opt : at<int32_t>(ws, p.eidx);
  float* gate = gate_opt ? gate_opt : at<float>(ws, p.gate);
  int32_t* perm = perm_opt ? perm_opt : at<int32_t>(ws, p.perm);
  prof_start(s);
  cudaError_t e = cudaMemsetAsync(at<DevStatus>(ws, p.status), 0, sizeof(DevStatus), s);
  // residual stacks (unless prepared) and the dense U GEMM (when the layer uses it) on the side
  // stream, concurrently with routing and permutation (in order, on `s`, when profiling per kernel)
  cudaEvent_t prep_done = nullptr;
  const bool side_work = p.tc && a.T > 0 && (!prep || tc_u_dense(a));
  SideStream* side = (side_work && !g_prof_ev) ? side_stream() : nullptr;
  if (e == cudaSuccess && side) {
    e = cudaEventRecord(side->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->st, side->fork, 0);
    if (e == cudaSuccess)
      e = launch_resid_prep(a, resid_ptrs(a, resid), tc_bufs(p, ws, prep), x, at<DevStatus>(ws, p.status), side->st,
                            prep == nullptr);
    if (e == cudaSuccess) e = cudaEventRecord(side->join, side->st);
    prep_done = side->join;
  }
  PermOut o{perm, at<int32_t>(ws, p.inv_pos), at<int32_t>(ws, p.ebeg), at<int32_t>(ws, p.ecnt),
            at<int32_t>(ws, p.gbeg), at<int32_t>(ws, p.row_asg), at<int32_t>(ws, p.row_of),
            at<int32_t>(ws, p.rbeg)};
  if (e == cudaSuccess)
    e = launch_route(a, x, w_group, b_group, w_expert, at<float>(ws, p.logits), at<int32_t>(ws, p.redo), gidx,
                     eidx, gate, at<DevStatus>(ws, p.status), true, s);
  if (e == cudaSuccess)
    e = launch_permute(a, eidx, o, at<int32_t>(ws, p.cnt), at<int32_t>(ws, p.off), p.nblk,
                       at<DevStatus>(ws, p.status), true, s);
  void* yrows = a.kg > 1 ? at<void>(ws, p.yrows) : y;
  if (e == cudaSuccess)
    e = run_ffn(a, p, ws, x, w_gate, w_up, w_down, resid, eidx, gate, o.row_asg, o.rbeg, yrows, prep_done, s, prep);
  if (e == cudaSuccess) e = launch_combine(a, yrows, y, s);
  // the side stream's work rejoins `s` on every path (a capture must not end with it forked)
  if (prep_done) {
    const cudaError_t j = cudaStreamWaitEvent(s, prep_done, 0);
    if (e == cudaSuccess) e = j;
  }
  return cuda_status(e);
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_hier_workspace_size(const moe_hier_desc* desc, int* status_out) {
  LayerArgs a;
  const int st = validate(desc, nullptr, &a);
  if (status_out) *status_out = st;
  if (st != MOE_OK) return 0;
  return make_plan(a).total;
}

int moe_hier_route(const moe_hier_desc* desc, const void* x, const void* w_group,
                   const float* b_group, const void* w_expert, const int32_t* group_map_host,
                   int32_t* gidx, int32_t* eidx, float* gate, void* ws, size_t ws_bytes,
                   void* stream) {
  LayerArgs a;
  if (!group_map_host) return MOE_ERR_INVALID;
  int st = validate(desc, group_map_host, &a);
  if (st != MOE_OK) return st;
  if (a.T > 0 && (!x || !w_group || !w_expert || !gidx || !eidx || !gate)) return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(w_group) || !aligned16(w_expert)) return MOE_ERR_INVALID;
  const Plan p = make_plan(a);
  if ((st = check_ws(p, ws, ws_bytes)) != MOE_OK) return st;
  prof_start((cudaStream_t)stream);
  return cuda_status(launch_route(a, x, w_group, b_group, w_expert, at<float>(ws, p.logits),
                                  at<int32_t>(ws, p.redo), gidx, eidx, gate, at<DevStatus>(ws, p.status),
                                  false, (cudaStream_t)stream));
}

int moe_hier_permute(const moe_hier_desc* desc, const int32_t* group_map_host, const int32_t* eidx,
                     int32_t* perm, int32_t* inv_pos, int32_t* expert_begin, int32_t* expert_count,
                     int32_t* group_begin, int32_t* row_asg, int32_t* row_of, int32_t* row_begin,
                     void* ws, size_t ws_bytes, void* stream) {
  LayerArgs a;
  if (!group_map_host) return MOE_ERR_INVALID;
  int st = validate(desc, group_map_host, &a);
  if (st != MOE_OK) return st;
  if (!row_begin || (a.T > 0 && (!eidx || !row_asg))) return MOE_ERR_INVALID;
  const Plan p = make_plan(a);
  if ((st = check_ws(p, ws, ws_bytes)) != MOE_OK) return st;
  PermOut o{perm, inv_pos, expert_begin, expert_count, group_begin, row_asg, row_of, row_begin};
  prof_start((cudaStream_t)stream);
  return cuda_status(launch_permute(a, eidx, o, at<int32_t>(ws, p.cnt), at<int32_t>(ws, p.off),
                                    p.nblk, at<DevStatus>(ws, p.status), false, (cudaStream_t)stream,
                                    perm_wait_setting()));
}

int moe_hier_ffn(const moe_hier_desc* desc, const void* x, const int32_t* group_map_host,
                 const void* w_gate, const void* w_up, const void* w_down,
                 const moe_hier_resid* resid, const int32_t* eidx, const float* gate,
                 const int32_t* row_asg, const int32_t* row_begin, void* y_rows, void* ws,
                 size_t ws_bytes, void* stream) {
  LayerArgs a;
  if (!group_map_host) return MOE_ERR_INVALID;
  int st = validate(desc, group_map_host, &a);
  if (st != MOE_OK) return st;
  if (a.T > 0 && (!x || !w_gate || !w_up || !w_down || !eidx || !gate || !row_asg || !row_begin ||
                  !y_rows || !resid_ok(a, resid)))
    return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(y_rows))
    return MOE_ERR_INVALID;
  const Plan p = make_plan(a);
  if ((st = check_ws(p, ws, ws_bytes)) != MOE_OK) return st;
  prof_start((cudaStream_t)stream);
  return cuda_status(run_ffn(a, p, ws, x, w_gate, w_up, w_down, resid, eidx, gate, row_asg, row_begin, y_rows,
                             nullptr, (cudaStream_t)stream));
}

int moe_hier_combine(const moe_hier_desc* desc, const void* y_rows, void* y, void* stream) {
  LayerArgs a;
  int st = validate(desc, nullptr, &a);
  if (st != MOE_OK) return st;
  if (a.T > 0 && (!y_rows || !y)) return MOE_ERR_INVALID;
  prof_start((cudaStream_t)stream);
  return cuda_status(launch_combine(a, y_rows, y, (cudaStream_t)stream));
}

int moe_hier_forward(const moe_hier_desc* desc, const void* x, const void* w_group,
                     const float* b_group, const void* w_expert, const int32_t* group_map_host,
                     const void* w_gate, const void* w_up, const void* w_down,
                     const moe_hier_resid* resid, void* y, int32_t* gidx_opt, int32_t* eidx_opt,
                     float* gate_opt, int32_t* perm_opt, void* ws, size_t ws_bytes, void* stream) {
  return forward_impl(desc, x, w_group, b_group, w_expert, group_map_host, w_gate, w_up, w_down, resid, nullptr, 0, y,
                      gidx_opt, eidx_opt, gate_opt, perm_opt, ws, ws_bytes, stream);
}

size_t moe_hier_prepared_size(const moe_hier_desc* desc, int* status_out) {
  LayerArgs a;
  int st = validate(desc, nullptr, &a);
  const Plan p = st == MOE_OK ? make_plan(a) : Plan{};
  if (st == MOE_OK && !p.tc) st = MOE_ERR_UNSUPPORTED;
  if (status_out) *status_out = st;
  return st == MOE_OK ? stack_layout(p).total : 0;
}

int moe_hier_prepare(const moe_hier_desc* desc, const int32_t* group_map_host, const moe_hier_resid* resid,
                     void* prep, size_t prep_bytes, void* stream) {
  LayerArgs a;
  if (!group_map_host) return MOE_ERR_INVALID;
  int st = validate(desc, group_map_host, &a);
  if (st != MOE_OK) return st;
  const Plan p = make_plan(a);
  if (!p.tc) return MOE_ERR_UNSUPPORTED;
  if (!resid_ok(a, resid)) return MOE_ERR_INVALID;
  if (!prep || ((uintptr_t)prep & 255) != 0 || prep_bytes < stack_layout(p).total) return MOE_ERR_WORKSPACE;
  prof_start((cudaStream_t)stream);
  // the stacks alone: no tokens are needed (x = null skips the dense U GEMM)
  return cuda_status(launch_resid_prep(a, resid_ptrs(a, resid), tc_bufs(p, prep, prep), nullptr, nullptr,
                                       (cudaStream_t)stream, true));
}

int moe_hier_forward_prepared(const moe_hier_desc* desc, const void* x, const void* w_group, const float* b_group,
                              const void* w_expert, const int32_t* group_map_host, const void* w_gate,
                              const void* w_up, const void* w_down, const moe_hier_resid* resid, const void* prep,
                              size_t prep_bytes, void* y, int32_t* gidx_opt, int32_t* eidx_opt, float* gate_opt,
                              int32_t* perm_opt, void* ws, size_t ws_bytes, void* stream) {
  if (!prep) return MOE_ERR_WORKSPACE;
  return forward_impl(desc, x, w_group, b_group, w_expert, group_map_host, w_gate, w_up, w_down, resid,
                      const_cast<void*>(prep), prep_bytes, y, gidx_opt, eidx_opt, gate_opt, perm_opt, ws, ws_bytes,
                      stream);
}

static int compress_args(const moe_hier_compress_desc* d, const int32_t* group_map, CmpArgs* c) {
  if (!d) return MOE_ERR_INVALID;
  if (d->E <= 0 || d->G <= 0 || d->E % d->G != 0 || d->E > kMaxE) return MOE_ERR_INVALID;
  if (d->d_in <= 0 || d->d_out <= 0 || d->d_in % 128 != 0 || d->d_out % 128 != 0) return MOE_ERR_INVALID;
  if (d->rank < 1 || d->rank > 32 || d->sketch <= d->rank || d->sketch > 64) return MOE_ERR_INVALID;
  if (d->power_iters < 0 || d->power_iters > 16) return MOE_ERR_INVALID;
  memset(c, 0, sizeof(*c));
  c->E = d->E; c->G = d->G; c->d_out = d->d_out; c->d_in = d->d_in; c->r = d->rank; c->l = d->sketch;
  c->power_iters = d->power_iters;
  if (group_map) {
    const int K = d->E / d->G;
    int fill[kMaxE] = {0};
    for (int e = 0; e < d->E; ++e) {
      const int g = group_map[e];
      if (g < 0 || g >= d->G || fill[g] >= K) return MOE_ERR_INVALID;
      c->member[g * K + fill[g]++] = (uint8_t)e;
      c->group_of[e] = (uint8_t)g;
    }
  }
  return MOE_OK;
}

size_t moe_hier_compress_workspace_size(const moe_hier_compress_desc* desc, int* status_out) {
  CmpArgs c;
  const int st = compress_args(desc, nullptr, &c);
  if (status_out) *status_out = st;
  return st == MOE_OK ? cmp_workspace_bytes(c) : 0;
}

int moe_hier_compress(const moe_hier_compress_desc* desc, const void* w, const int32_t* group_map_host,
                      const float* omega, void* base, void* A_codes, void* A_scales, void* B_codes, void* B_scales,
                      float* sigma, double* err, float* At_f32, float* Bt_f32, void* ws, size_t ws_bytes,
                      void* stream) {
  CmpArgs c;
  if (!group_map_host) return MOE_ERR_INVALID;
  int st = compress_args(desc, group_map_host, &c);
  if (st != MOE_OK) return st;
  if (!w || !omega || !base || !A_codes || !A_scales || !B_codes || !B_scales || !sigma) return MOE_ERR_INVALID;
  if (!aligned16(w) || !aligned16(omega) || !aligned16(base) || !aligned16(A_codes) || !aligned16(B_codes) ||
      ((uintptr_t)A_scales & 1) || ((uintptr_t)B_scales & 1) || ((uintptr_t)sigma & 3) || ((uintptr_t)err & 7) ||
      !aligned16(At_f32) || !aligned16(Bt_f32))
    return MOE_ERR_INVALID;
  if (!ws || ((uintptr_t)ws & 255) != 0 || ws_bytes < cmp_workspace_bytes(c)) return MOE_ERR_WORKSPACE;
  prof_start((cudaStream_t)stream);
  return cuda_status(launch_compress(c, w, omega, base, (uint8_t*)A_codes, (__half*)A_scales, (uint8_t*)B_codes,
                                     (__half*)B_scales, sigma, err, At_f32, Bt_f32, ws, (cudaStream_t)stream));
}

int moe_hier_quantise_int4(const float* v, int64_t rows, int32_t n, void* codes, void* scales, void* stream) {
  if (rows < 0 || n <= 0 || n % 64 != 0) return MOE_ERR_INVALID;
  if (rows > 0 && (!v || !codes || !scales || ((uintptr_t)v & 7) || ((uintptr_t)scales & 1))) return MOE_ERR_INVALID;
  prof_start((cudaStream_t)stream);
  return cuda_status(launch_quant_int4(v, (size_t)rows, n, (uint8_t*)codes, (__half*)scales, (cudaStream_t)stream));
}

int moe_hier_debug_set_wait(uint64_t wait_ns, int phantom_arrivals) {
  if (phantom_arrivals < 0) return MOE_ERR_INVALID;
  g_wait_ns.store(wait_ns, std::memory_order_relaxed);
  g_wait_phantom.store((unsigned int)phantom_arrivals, std::memory_order_relaxed);
  return MOE_OK;
}

int moe_hier_debug_route_tc(const moe_hier_desc* desc, const void* x, const void* w_group, const float* b_group,
                            const void* w_expert, const int32_t* group_map_host, float* out, void* ws,
                            size_t ws_bytes, void* stream) {
  LayerArgs a;
  if (!group_map_host) return MOE_ERR_INVALID;
  int st = validate(desc, group_map_host, &a);
  if (st != MOE_OK) return st;
  if (!route_tc_ok(a) || a.across) return MOE_ERR_UNSUPPORTED;
  if (!x || !w_group || !w_expert || !out) return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(w_group) || !aligned16(w_expert)) return MOE_ERR_INVALID;
  const Plan p = make_plan(a);
  if ((st = check_ws(p, ws, ws_bytes)) != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  DevStatus* status = at<DevStatus>(ws, p.status);
  cudaError_t e = cudaMemsetAsync(&status->route_redo, 0, sizeof(int), s);
  if (e == cudaSuccess)
    e = launch_route_tc(a, x, w_group, b_group, w_expert, at<int32_t>(ws, p.gidx), at<int32_t>(ws, p.eidx),
                        at<float>(ws, p.gate), at<int32_t>(ws, p.redo), status, s, out);
  return cuda_status(e);
}

int moe_hier_get_status(const void* ws, void* stream) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  DevStatus h{};
  if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  return h.code;
}

int moe_hier_profile_begin(void* const* events, int n_events) {
  if (!events || n_events < 1) return MOE_ERR_INVALID;
  g_prof_ev = events;
  g_prof_n = n_events;
  g_prof_i = 0;
  g_prof_launches = 0;
  return MOE_OK;
}

int moe_hier_profile_end(const char** names, int max_names) {
  const int n = g_prof_launches;
  for (int i = 0; names && i < max_names && i < n && i < 256; ++i) names[i] = g_prof_names[i];
  g_prof_ev = nullptr;
  g_prof_n = g_prof_i = g_prof_launches = 0;
  return n;
}

const char* moe_hier_last_cuda_error(void) {
  return g_last_cuda_error == cudaSuccess ? "no error" : cudaGetErrorString(g_last_cuda_error);
}

const char* moe_hier_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"

// FFN whose base matrices sit in `wslots` group slots (group g in slot wslot[g]): the offload
// cache (offload.cu).  Tensor-core layers only.
namespace moe {
int ffn_with_slots(const moe_hier_desc* desc, const void* x, const int32_t* group_map_host, const void* w_gate,
                   const void* w_up, const void* w_down, int wslots, const uint8_t* wslot,
                   const moe_hier_resid* resid, const int32_t* eidx, const float* gate, const int32_t* row_asg,
                   const int32_t* row_begin, void* y_rows, void* ws, size_t ws_bytes, void* stream) {
  LayerArgs a;
  if (!group_map_host) return MOE_ERR_INVALID;
  int st = validate(desc, group_map_host, &a);
  if (st != MOE_OK) return st;
  if (a.T > 0 && (!x || !w_gate || !w_up || !w_down || !eidx || !gate || !row_asg || !row_begin || !y_rows ||
                  !resid_ok(a, resid)))
    return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(y_rows))
    return MOE_ERR_INVALID;
  const Plan p = make_plan(a);
  if (!p.tc) return MOE_ERR_UNSUPPORTED;
  if ((st = check_ws(p, ws, ws_bytes)) != MOE_OK) return st;
  a.wslots = wslots;
  for (int g = 0; g < a.G; ++g) a.tab.wslot[g] = wslot[g];
  prof_start((cudaStream_t)stream);
  return cuda_status(run_ffn(a, p, ws, x, w_gate, w_up, w_down, resid, eidx, gate, row_asg, row_begin, y_rows,
                             nullptr, (cudaStream_t)stream));
}
}  // namespace moe

// ------------------------------------------------------------------------------------------
// Permutation without a workspace argument.
//
// Some callers cannot hand the library a workspace: a host that owns every byte of device
// memory through its own pool and forbids any other allocation, or a latency-critical loop in
// which the implicit device synchronisation of an allocation is not allowed.  For them the
// permutation's only scratch -- the per-block histograms and their offsets -- lives in the
// fixed array below, which every GPU that loads the library holds until the process exits.
// ------------------------------------------------------------------------------------------
namespace moe {

constexpr int kNoAllocScratchInts = 65536;  // 256 KiB: histograms + offsets, 2 * nblk * (E + G) ints
static __device__ __align__(256) int32_t g_perm_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
static std::mutex g_scratch_mu;
static int32_t* g_scratch_dev[kMaxDevices];   // device address of g_perm_scratch, per device

// Device address of the scratch array on the current device (looked up on the first call made
// with that device current).  In host code `g_perm_scratch` names a host-side stand-in, never
// the device memory, so kernels must receive this address instead.
static cudaError_t scratch_on_current_device(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_perm_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_dev[dev] = (int32_t*)p;
  }
  *out = g_scratch_dev[dev];
  return cudaSuccess;
}

}  // namespace moe

extern "C" int moe_hier_permute_noalloc(const moe_hier_desc* desc, const int32_t* group_map_host,
                                        const int32_t* eidx, int32_t* perm, int32_t* inv_pos,
                                        int32_t* expert_begin, int32_t* expert_count, int32_t* group_begin,
                                        int32_t* row_asg, int32_t* row_of, int32_t* row_begin, void* stream) {
  LayerArgs a;
  if (!group_map_host) return MOE_ERR_INVALID;
  int st = validate(desc, group_map_host, &a);
  if (st != MOE_OK) return st;
  if (!row_begin || (a.T > 0 && (!eidx || !row_asg))) return MOE_ERR_INVALID;
  const int nblk = (a.T + 255) / 256;
  const size_t need = 2 * (size_t)nblk * (size_t)(a.E + a.G);
  if (need > (size_t)kNoAllocScratchInts) return MOE_ERR_WORKSPACE;   // layer too large for the fixed scratch
  int32_t* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  // The count kernel writes every histogram entry and the scan every offset it later reads, so
  // nothing left in the array by an earlier call is used.
  int32_t* cnt = scratch;
  int32_t* off = scratch + (size_t)nblk * (a.E + a.G);
  PermOut o{perm, inv_pos, expert_begin, expert_count, group_begin, row_asg, row_of, row_begin};
  prof_start((cudaStream_t)stream);
  return cuda_status(launch_permute(a, eidx, o, cnt, off, nblk, nullptr, false, (cudaStream_t)stream));
}
