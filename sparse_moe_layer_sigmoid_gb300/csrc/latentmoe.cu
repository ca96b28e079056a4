// Host orchestrator and C-ABI entry points of the LatentMoE layer (declared in latentmoe.h).
//
// One forward pass enqueues, on the caller's stream and without any host synchronisation:
//   router logits -> sigmoid/top-k/p -> dispatch (count, scan, scatter) -> W_down ->
//   row scatter into expert-contiguous batches -> grouped gate/up GLU -> grouped down x p ->
//   fixed-order combine + RMSNorm -> shared-expert gate/up GLU -> final GEMM
//   y = [shared activations | RMSNorm(u)] . [shared down | W_up]^T
// (page "Lesson 6 - LatentMoE", kimi-k3-course.pages.dev, eq. 11 and eq. 13).
// W_down and the shared experts' gate/up GLU depend on x alone: on the tensor-core path they run
// on the handle's second stream, forked from the caller's stream by an event at the start of the
// call and joined back (an event wait) before the row scatter and before the final GEMM, so they
// overlap the routing chain (router, top-k, dispatch) and the routed experts.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <new>

#include "common.cuh"
#include "internal.h"
#include "latentmoe.h"

using namespace lmoe;

struct lmoe_handle {
  lmoe_config cfg;
  int device;
  int num_sms;
  uint8_t* ws;
  size_t ws_bytes;
  uint32_t* status;
  float* logits;
  int32_t* refine_list;   // [T] tokens whose top-k boundary is settled exactly
  int32_t* refine_count;  // [2]: refined tokens, near ties of the last routing
  int32_t* idx;
  float* p;
  DispatchBuffers db;
  int max_tiles;
  int max_tiles_s;
  int max_tiles_p;
  int max_tiles_m;
  void* z;
  void* z_perm;  // gathered expert-contiguous rows (or their MXFP4 records); reused for the routed down output
  void* a;       // routed GLU activations [T*k][h] (or their MXFP4 records)
  void* act_cat; // [T][N_s*h_s + l]: shared GLU activations | RMSNorm(u)
  void* x_stage; // forward_host staging
  void* y_stage;
  void* wr_split; // bf16 hi/mid/lo terms of an fp32 W_r [3][E][d] (bf16 activations only)
  float* splitk;  // split-K partial accumulators of dense tensor-core GEMMs with <= 128 rows
  size_t splitk_bytes;
  int last_launches;
  uint64_t timeout_ns;
  int inject;
  int last_T;                                 // T of the last call (for latentmoe_debug_buffer)
  cudaEvent_t stage_ev[LMOE_NUM_STAGES + 1];  // caller-owned; recording on when stage_on
  bool stage_on;
  int marked;                                 // index of the last stage event recorded
  cudaStream_t aux;                           // second stream: W_down and the shared GLU
  cudaEvent_t ev_fork, ev_wdown, ev_shared;   // fork from / joins into the caller's stream
  float* splitk_aux;                          // split-K partials of GEMMs on the second stream
  int32_t* ep_plan;                           // expert-parallel emulation: plan (<= kMaxEpRanks ranks)
  int32_t* ep_row_of;                         // [T*k]: send position of row (t, j)
};

namespace {

constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;

size_t dtype_bytes(int dt) { return dt == kF32 ? 4 : 2; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

lmoe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA; }

enum Stage : int {
  kStRouter = 0, kStTopk, kStDispatch, kStWDown, kStScatter, kStGlu, kStDown, kStCombine, kStSharedGlu, kStFinal
};
const char* const kStageNames[LMOE_NUM_STAGES] = {
    "router_logits", "topk", "dispatch", "w_down", "scatter_rows", "routed_gate_up_glu", "routed_down",
    "combine_rmsnorm", "shared_gate_up_glu", "final_gemm"};

// Stage i spans stage_ev[i] .. stage_ev[i+1]; skipped stages get zero width.
void stages_start(lmoe_handle* h, cudaStream_t s) {
  if (!h->stage_on) return;
  cudaEventRecord(h->stage_ev[0], s);
  h->marked = 0;
}
void stage_begin(lmoe_handle* h, int i, cudaStream_t s) {
  if (!h->stage_on) return;
  while (h->marked < i) cudaEventRecord(h->stage_ev[++h->marked], s);
}
void stage_end(lmoe_handle* h, int i, cudaStream_t s) {
  if (!h->stage_on) return;
  stage_begin(h, i, s);
  cudaEventRecord(h->stage_ev[++h->marked], s);
}
void stages_finish(lmoe_handle* h, cudaStream_t s) { stage_begin(h, LMOE_NUM_STAGES, s); }

#define LMOE_TRY(expr)                          \
  do {                                          \
    cudaError_t e__ = (expr);                   \
    if (e__ != cudaSuccess) return LMOE_ERR_CUDA; \
  } while (0)

lmoe_status validate_config(const lmoe_config& c) {
  const bool identity = (c.flags & LMOE_FLAG_IDENTITY_EXPERTS) != 0;
  if (c.d <= 0 || c.latent <= 0 || c.num_experts < 1 || c.num_experts > 1024) return LMOE_ERR_INVALID_ARG;
  if (c.top_k < 1 || c.top_k > c.num_experts || c.top_k > 32) return LMOE_ERR_INVALID_ARG;
  if (c.num_shared < 0 || c.max_tokens < 1) return LMOE_ERR_INVALID_ARG;
  if (!identity && (c.hidden <= 0 || (c.num_shared > 0 && c.shared_hidden <= 0))) return LMOE_ERR_INVALID_ARG;
  if ((int64_t)c.max_tokens * c.top_k >= (int64_t)1 << 31) return LMOE_ERR_INVALID_ARG;
  if (c.act != LMOE_F32 && c.act != LMOE_BF16) return LMOE_ERR_INVALID_ARG;
  if (c.router_w != LMOE_F32 && c.router_w != LMOE_BF16) return LMOE_ERR_INVALID_ARG;
  if (c.routed_w != LMOE_F32 && c.routed_w != LMOE_BF16 && c.routed_w != LMOE_MXFP4) return LMOE_ERR_INVALID_ARG;
  if (!(c.rms_eps >= 0.0f)) return LMOE_ERR_INVALID_ARG;
  if (c.flags & ~(LMOE_FLAG_IDENTITY_EXPERTS | LMOE_FLAG_SINGLE_CTA_GEMM | LMOE_FLAG_MXFP4_DEQUANT |
                  LMOE_FLAG_MXFP8_ACT))
    return LMOE_ERR_INVALID_ARG;
  if ((c.flags & LMOE_FLAG_MXFP8_ACT) &&
      (c.routed_w != LMOE_MXFP4 || c.act != LMOE_BF16 || (c.flags & (LMOE_FLAG_MXFP4_DEQUANT | LMOE_FLAG_SINGLE_CTA_GEMM))))
    return LMOE_ERR_INVALID_ARG;
  // router GEMM and the CUDA-core path step K by 16; combine moves 16-byte vectors
  if (c.d % 16 || c.latent % 16) return LMOE_ERR_UNSUPPORTED;
  if (c.act == LMOE_F32) {
    if (!identity && c.routed_w != LMOE_F32) return LMOE_ERR_UNSUPPORTED;
    if (!identity && (c.hidden % 16 || (c.num_shared > 0 && c.shared_hidden % 16))) return LMOE_ERR_UNSUPPORTED;
    if (c.latent > 4096) return LMOE_ERR_UNSUPPORTED;
  } else {
    // tensor-core tiles: K steps of 64, output tiles of 256 columns (128 for GLU halves)
    if (c.d % 256 || c.latent % 256 || c.latent > 8192 || c.num_experts % 4) return LMOE_ERR_UNSUPPORTED;
    if (!identity) {
      if (c.routed_w == LMOE_F32) return LMOE_ERR_UNSUPPORTED;
      if (c.hidden % 128) return LMOE_ERR_UNSUPPORTED;
      if (c.num_shared > 0 && c.shared_hidden % 128) return LMOE_ERR_UNSUPPORTED;
      // MXFP4 experts: the converters read E8M0 scales 16 bytes (512 elements) at a time
      if (c.routed_w == LMOE_MXFP4 && (c.latent % 512 || c.hidden % 512)) return LMOE_ERR_UNSUPPORTED;
    }
  }
  return LMOE_OK;
}

// Carve the workspace.  With base == nullptr only computes the size.
size_t layout(lmoe_handle* h, uint8_t* base) {
  const lmoe_config& c = h->cfg;
  const bool identity = (c.flags & LMOE_FLAG_IDENTITY_EXPERTS) != 0;
  const size_t T = (size_t)c.max_tokens, E = (size_t)c.num_experts, k = (size_t)c.top_k;
  const size_t rows = T * k;
  const size_t nchunks = (T + kDispatchChunk - 1) / kDispatchChunk;
  const size_t ab = dtype_bytes(c.act);
  const size_t kcat = (size_t)c.num_shared * c.shared_hidden + c.latent;
  size_t off = 0;
  auto take = [&](size_t bytes) -> uint8_t* {
    uint8_t* p = base ? base + off : nullptr;
    off += round_up(bytes, 256);
    return p;
  };
  h->max_tiles = (int)(rows / kTileM + E + 1);
  h->status = reinterpret_cast<uint32_t*>(take(sizeof(uint32_t)));
  h->logits = reinterpret_cast<float*>(take(T * E * 4));
  h->refine_list = reinterpret_cast<int32_t*>(take(T * 4));
  h->refine_count = reinterpret_cast<int32_t*>(take(8));
  h->idx = reinterpret_cast<int32_t*>(take(rows * 4));
  h->p = reinterpret_cast<float*>(take(rows * 4));
  h->db.chunk_counts = reinterpret_cast<int32_t*>(take(nchunks * E * 4));
  h->db.chunk_base = reinterpret_cast<int32_t*>(take(nchunks * E * 4));
  h->db.offsets = reinterpret_cast<int32_t*>(take((E + 1) * 4));
  h->db.tiles = reinterpret_cast<int4*>(take((size_t)h->max_tiles * 16));
  h->db.num_tiles = reinterpret_cast<int32_t*>(take(4));
  h->max_tiles_s = (int)(rows / kTileS + E + 1);
  h->db.tiles_s = reinterpret_cast<int4*>(take((size_t)h->max_tiles_s * 16));
  h->db.num_tiles_s = reinterpret_cast<int32_t*>(take(4));
  h->max_tiles_p = (int)(rows / kTileP + E + 1);
  h->db.tiles_p = reinterpret_cast<int4*>(take((size_t)h->max_tiles_p * 16));
  h->db.num_tiles_p = reinterpret_cast<int32_t*>(take(4));
  h->max_tiles_m = (int)(rows / kTileMx + E + 1);
  h->db.tiles_m = reinterpret_cast<int4*>(take((size_t)h->max_tiles_m * 16));
  h->db.num_tiles_m = reinterpret_cast<int32_t*>(take(4));
  h->db.tok_of_row = reinterpret_cast<int32_t*>(take(rows * 4));
  h->db.row_of = reinterpret_cast<int32_t*>(take(rows * 4));
  h->db.p_row = reinterpret_cast<float*>(take(rows * 4));
  h->z = take(T * c.latent * ab);
  h->z_perm = take(rows * c.latent * ab);
  h->a = identity ? nullptr : take(rows * (size_t)c.hidden * ab);
  h->act_cat = identity ? nullptr : take(T * kcat * ab);
  h->x_stage = take(T * (size_t)c.d * ab);
  h->y_stage = take(T * (size_t)(identity ? c.latent : c.d) * ab);
  h->wr_split = (c.act == LMOE_BF16 && c.router_w == LMOE_F32) ? take(3 * E * (size_t)c.d * 2) : nullptr;
  h->splitk_bytes = c.act == LMOE_BF16 ? tc_splitk_partial_bytes(h->num_sms) : 0;
  h->splitk = h->splitk_bytes ? reinterpret_cast<float*>(take(h->splitk_bytes)) : nullptr;
  h->splitk_aux = h->splitk_bytes ? reinterpret_cast<float*>(take(h->splitk_bytes)) : nullptr;
  h->ep_plan = reinterpret_cast<int32_t*>(take(ep_plan_ints(E, kMaxEpRanks) * 4));
  h->ep_row_of = reinterpret_cast<int32_t*>(take(rows * 4));
  return off;
}

bool weights_ok(const lmoe_handle* h, const lmoe_weights* w, bool need_router) {
  const lmoe_config& c = h->cfg;
  const bool identity = (c.flags & LMOE_FLAG_IDENTITY_EXPERTS) != 0;
  if (!w) return false;
  if (need_router && (!w->w_router || !aligned16(w->w_router))) return false;
  if (w->router_bias && !aligned16(w->router_bias)) return false;
  if (!w->w_down_proj || !aligned16(w->w_down_proj)) return false;
  if (identity) return true;
  if (!w->rms_gain || !w->routed_gate_up || !w->routed_down || !w->w_up_proj) return false;
  if (!aligned16(w->rms_gain) || !aligned16(w->routed_gate_up) || !aligned16(w->routed_down) ||
      !aligned16(w->w_up_proj))
    return false;
  if (c.num_shared > 0) {
    if (!w->shared_gate_up || !w->shared_down || !aligned16(w->shared_gate_up) || !aligned16(w->shared_down))
      return false;
  }
  if (c.routed_w == LMOE_MXFP4) {
    if (!w->routed_gate_up_scale || !w->routed_down_scale || !aligned16(w->routed_gate_up_scale) ||
        !aligned16(w->routed_down_scale))
      return false;
  }
  return true;
}

// Storage type of the routed-expert activations (z, gathered rows, GLU outputs, expert outputs):
// fp16 next to MXFP4 weights (the converted weights are fp16), else the activation type.
int routed_act_dtype(const lmoe_config& c) { return c.routed_w == LMOE_MXFP4 ? kF16 : c.act; }

TcOperand op2d(const void* ptr, int64_t rows, int64_t cols) {
  return TcOperand{ptr, cols, rows, 1, cols, rows * cols};
}
TcOperand op3d(const void* ptr, int64_t depth, int64_t rows, int64_t cols) {
  return TcOperand{ptr, cols, rows, depth, cols, rows * cols};
}

// Routing into the handle's buffers: router + top-k unless the caller supplies idx/p.
lmoe_status run_routing(lmoe_handle* h, const void* x, int T, const lmoe_weights* w, const int32_t* ext_idx,
                        const float* ext_p, const int32_t** idx_out, const float** p_out, cudaStream_t s) {
  const lmoe_config& c = h->cfg;
  const int32_t* idx = ext_idx;
  const float* p = ext_p;
  if (!ext_idx) {
    stage_begin(h, kStRouter, s);
    // short batches: the top-k kernel adds the router GEMM's split-K sums itself
    SplitPartials part{nullptr, 0, 0, 0};
    LMOE_TRY(launch_router(x, c.act, w->w_router, c.router_w, h->logits, h->wr_split, T, c.num_experts, c.d,
                           h->status, h->timeout_ns, h->num_sms, &h->last_launches, s, h->splitk, h->splitk_bytes,
                           !(c.flags & LMOE_FLAG_SINGLE_CTA_GEMM), T <= kTopkFusedMaxT ? &part : nullptr));
    stage_end(h, kStRouter, s);
    const RouterSrc rs{x, c.act, w->w_router, c.router_w, c.d, kRouterLogitMargin};
    LMOE_TRY(launch_topk(h->logits, w->router_bias, rs, T, c.num_experts, c.top_k, h->idx, h->p, h->refine_list,
                         h->refine_count, h->status, h->num_sms, s, &part));
    stage_end(h, kStTopk, s);
    h->last_launches += T <= kTopkFusedMaxT ? 1 : 2;  // one kernel for short batches, else select + refine
    idx = h->idx;
    p = h->p;
  }
  stage_begin(h, kStDispatch, s);
  LMOE_TRY(launch_dispatch(idx, p, T, c.num_experts, c.top_k, h->db, h->status, &h->last_launches, s));
  stage_end(h, kStDispatch, s);
  *idx_out = idx;
  *p_out = p;
  return LMOE_OK;
}

// A tensor-core GEMM of the layer: dense GEMMs with at least 256 rows run on CTA pairs (256 x 256
// tiles), everything else on single CTAs (128-row tiles; dense ones with at most half as many
// output tiles as SMs split K).  Adds its launches to *launches.
cudaError_t run_tc_gemm(lmoe_handle* h, TcGemm g, int inject, int* launches, cudaStream_t s) {
  const bool on_aux = s == h->aux && h->aux != nullptr;
  const bool pair = !(h->cfg.flags & LMOE_FLAG_SINGLE_CTA_GEMM) && g.M >= kTileP && tc_pair_supported(g);
  if (pair) {
    *launches += 1;
    return launch_tc_pair(g, h->status, h->timeout_ns, s, inject);
  }
  // dense GEMMs of at most 128 rows may split K over the SMs (decode batches)
  if (!g.tiles) {
    g.partial = on_aux ? h->splitk_aux : h->splitk;  // each stream has its own partials
    g.partial_bytes = h->splitk_bytes;
  }
  g.launch_count = launches;
  return launch_tc_gemm(g, h->status, h->timeout_ns, inject, h->num_sms, s);
}

// While armed, makes the caller's stream wait for everything enqueued on the handle's second
// stream so far (used when a forward pass returns early after forking).
struct AuxJoin {
  lmoe_handle* h;
  cudaStream_t s;
  bool armed;
  ~AuxJoin() {
    if (armed && cudaEventRecord(h->ev_shared, h->aux) == cudaSuccess) cudaStreamWaitEvent(s, h->ev_shared, 0);
  }
};

lmoe_status run_forward(lmoe_handle* h, const void* x, int T, const lmoe_weights* w, const int32_t* ext_idx,
                        const float* ext_p, void* y, cudaStream_t s) {
  const lmoe_config& c = h->cfg;
  const bool identity = (c.flags & LMOE_FLAG_IDENTITY_EXPERTS) != 0;
  const bool tc = c.act == LMOE_BF16;
  const int k = c.top_k, l = c.latent, d = c.d, hdim = c.hidden;
  const int rows = T * k;
  const int ns = c.num_shared, hs = c.shared_hidden;
  const int kcat = ns * hs + l;
  const size_t ab = dtype_bytes(c.act);
  h->last_launches = 0;
  h->last_T = T;
  stages_start(h, s);

  // test hook (latentmoe_set_wait_limit): drop one pipeline signal in the first routed GEMM (1)
  // or in the W_down GEMM (2) of this call
  const int inject_routed = h->inject == 1 ? 1 : 0, inject_wdown = h->inject == 2 ? 1 : 0;
  h->inject = 0;
  const int rt = routed_act_dtype(c);
  // z = W_down x (tensor cores)
  auto launch_wdown = [&](cudaStream_t st) {
    TcGemm g = {};
    g.epi = rt == kF16 ? kEpiF16 : kEpiBF16;
    g.M = T; g.N = l; g.K = d;
    g.A = op2d(x, T, d);
    g.B0 = op2d(w->w_down_proj, l, d);
    g.k0_len = d; g.k0_per_group = d;
    g.C = h->z; g.ldc = l;
    return run_tc_gemm(h, g, inject_wdown, &h->last_launches, st);
  };
  // shared experts' SiLU(gate) * up into the head columns of act_cat (tensor cores)
  auto launch_shared = [&](cudaStream_t st) {
    TcGemm g = {};
    g.epi = kEpiGluBF16;
    g.M = T; g.N = ns * hs; g.K = d;
    g.A = op2d(x, T, d);
    g.B0 = op3d(w->shared_gate_up, ns, 2 * hs, d);
    g.k0_len = d; g.k0_per_group = d; g.glu_h = hs;
    g.C = h->act_cat; g.ldc = kcat;
    return run_tc_gemm(h, g, 0, &h->last_launches, st);
  };
  // Both depend on x alone: unless stages are being timed one by one, they go to the second
  // stream at once and the caller's stream waits for them where their results are read.
  const bool fork = tc && !h->stage_on && h->aux != nullptr;
  AuxJoin join{h, s, false};  // on an early return the caller's stream still waits for the second
  if (fork) {
    LMOE_TRY(cudaEventRecord(h->ev_fork, s));
    LMOE_TRY(cudaStreamWaitEvent(h->aux, h->ev_fork, 0));
    join.armed = true;
    LMOE_TRY(launch_wdown(h->aux));
    LMOE_TRY(cudaEventRecord(h->ev_wdown, h->aux));
    if (!identity && ns > 0) LMOE_TRY(launch_shared(h->aux));
    LMOE_TRY(cudaEventRecord(h->ev_shared, h->aux));
  }
  const int32_t* idx;
  const float* p;
  lmoe_status st = run_routing(h, x, T, w, ext_idx, ext_p, &idx, &p, s);
  if (st != LMOE_OK) return st;
  stage_begin(h, kStWDown, s);

  if (fork) {
    LMOE_TRY(cudaStreamWaitEvent(s, h->ev_wdown, 0));
  } else if (tc) {
    LMOE_TRY(launch_wdown(s));
  } else {
    SimtGemm g = {};
    g.A = x; g.lda = d; g.a_dtype = c.act; g.b_dtype = c.act;
    g.nseg = 1; g.seg[0] = SimtSegment{w->w_down_proj, d, 0, d, d};
    g.M = T; g.N = l; g.K = d;
    g.C = h->z; g.ldc = l; g.c_dtype = c.act;
    LMOE_TRY(launch_simt_gemm(g, s));
    h->last_launches += 1;
  }
  stage_end(h, kStWDown, s);
  // MXFP4 experts on the block-scaled MMA (CTA pairs): gathered rows and GLU activations as
  // three-term MXFP4 records (each no larger than the 16-bit row it replaces), expert outputs fp16
  const bool mx = tc && !identity && c.routed_w == LMOE_MXFP4 &&
                  !(c.flags & (LMOE_FLAG_MXFP4_DEQUANT | LMOE_FLAG_SINGLE_CTA_GEMM));
  // rows of z into expert-contiguous order (as MXFP4 records for the block-scaled expert GEMMs)
  const bool f8 = (c.flags & LMOE_FLAG_MXFP8_ACT) != 0;
  if (mx)
    LMOE_TRY(launch_scatter_mx3(h->z, rt, h->z_perm, h->db.row_of, T, k, l, h->status, h->timeout_ns, h->num_sms, s,
                                f8));
  else
    LMOE_TRY(launch_scatter_rows(h->z, h->z_perm, h->db.row_of, T, k, l, (int)ab, h->status, h->timeout_ns,
                                 h->num_sms, s));
  stage_end(h, kStScatter, s);
  h->last_launches += 1;

  if (identity) {  // the second stream (W_down only) was joined before the row scatter
    join.armed = false;
    stage_begin(h, kStCombine, s);
    LMOE_TRY(launch_combine(h->z_perm, c.act, c.act, h->db.row_of, p, nullptr, 0.f, T, k, l, y, l, s));
    stage_end(h, kStCombine, s);
    stages_finish(h, s);
    h->last_launches += 1;
    return LMOE_OK;
  }

  void* o = h->z_perm;  // the down projection overwrites the gathered rows it no longer needs
  uint8_t* n_out = static_cast<uint8_t*>(h->act_cat) + (size_t)ns * hs * ab;
  // few rows per expert (decode): weights on the M side of the MMA, tokens on the N side
  const bool swap = tc && (int64_t)T * k <= 32LL * c.num_experts;
  // many rows per expert, bf16 experts: swapped operands on CTA pairs (token tiles cut to fit)
  const bool pair_swap = tc && !swap && c.routed_w == LMOE_BF16 && !(c.flags & LMOE_FLAG_SINGLE_CTA_GEMM) &&
                         hdim % 128 == 0 && l % 256 == 0;
  if (mx) {
    // few rows per expert (decode): 16-row units and a deep weight ring; else 192-row tiles
    const int4* tl = swap ? h->db.tiles_s : h->db.tiles_m;
    const int32_t* ntl = swap ? h->db.num_tiles_s : h->db.num_tiles_m;
    const int max_tl = swap ? h->max_tiles_s : h->max_tiles_m;
    const int unit = swap ? kTileS : kTileMx;
    TcMx g = {};
    g.K = l; g.out_features = hdim; g.glu_h = hdim;
    g.w = op3d(w->routed_gate_up, c.num_experts, 2 * hdim, l);
    g.w_scale = w->routed_gate_up_scale;
    g.x = h->z_perm; g.rows = rows;
    g.C = h->a;
    g.f8 = f8;
    LMOE_TRY(launch_tc_mx(g, tl, ntl, max_tl, unit, h->status, h->timeout_ns, s, inject_routed));
    stage_end(h, kStGlu, s);

    TcMx dn = {};
    dn.K = hdim; dn.out_features = l; dn.glu_h = 0;
    dn.w = op3d(w->routed_down, c.num_experts, l, hdim);
    dn.w_scale = w->routed_down_scale;
    dn.x = h->a; dn.rows = rows;
    dn.C = o; dn.ldc = l; dn.row_scale = h->db.p_row;
    dn.f8 = f8;
    LMOE_TRY(launch_tc_mx(dn, tl, ntl, max_tl, unit, h->status, h->timeout_ns, s));
    stage_end(h, kStDown, s);
    h->last_launches += 2;
  } else if (pair_swap) {
    TcSwap g = {};
    g.epi = kEpiGluBF16;
    g.K = l; g.out_features = hdim; g.glu_h = hdim;
    g.act = op2d(h->z_perm, rows, l);
    g.w = op3d(w->routed_gate_up, c.num_experts, 2 * hdim, l);
    g.C = h->a; g.ldc = hdim;
    LMOE_TRY(launch_tc_pair_swap(g, h->db.tiles_p, h->db.num_tiles_p, h->max_tiles_p, h->status,
                                 h->timeout_ns, s, inject_routed));
    stage_end(h, kStGlu, s);

    TcSwap dn = {};
    dn.epi = kEpiScaleBF16;
    dn.K = hdim; dn.out_features = l;
    dn.act = op2d(h->a, rows, hdim);
    dn.w = op3d(w->routed_down, c.num_experts, l, hdim);
    dn.C = o; dn.ldc = l; dn.row_scale = h->db.p_row;
    LMOE_TRY(launch_tc_pair_swap(dn, h->db.tiles_p, h->db.num_tiles_p, h->max_tiles_p, h->status,
                                 h->timeout_ns, s));
    stage_end(h, kStDown, s);
    h->last_launches += 2;
  } else if (swap) {
    const bool fp4 = c.routed_w == LMOE_MXFP4;
    TcSwap g = {};
    g.epi = fp4 ? kEpiGluF16 : kEpiGluBF16;
    g.K = l; g.out_features = hdim; g.glu_h = hdim;
    g.act = op2d(h->z_perm, rows, l);
    g.w = op3d(w->routed_gate_up, c.num_experts, 2 * hdim, l);
    g.w_scale = fp4 ? w->routed_gate_up_scale : nullptr;
    g.ab_f16 = fp4;
    g.tiles_s = h->db.tiles_s; g.num_tiles_s = h->db.num_tiles_s; g.max_tiles_s = h->max_tiles_s;
    g.C = h->a; g.ldc = hdim;
    // MXFP4: units of at most kGemvMaxRows rows stream their weights through the CUDA cores,
    // larger ones go to the tensor cores
    g.skip_rows_upto = fp4 ? kGemvMaxRows : 0;
    if (fp4) LMOE_TRY(launch_gemv_fp4(g, h->status, h->timeout_ns, h->num_sms, s, inject_routed));
    LMOE_TRY(launch_tc_swap(g, h->status, h->timeout_ns, h->num_sms, s, inject_routed));
    stage_end(h, kStGlu, s);

    TcSwap dn = {};
    dn.epi = fp4 ? kEpiScaleF16 : kEpiScaleBF16;
    dn.K = hdim; dn.out_features = l;
    dn.act = op2d(h->a, rows, hdim);
    dn.w = op3d(w->routed_down, c.num_experts, l, hdim);
    dn.w_scale = fp4 ? w->routed_down_scale : nullptr;
    dn.ab_f16 = fp4;
    dn.tiles_s = h->db.tiles_s; dn.num_tiles_s = h->db.num_tiles_s; dn.max_tiles_s = h->max_tiles_s;
    dn.C = o; dn.ldc = l; dn.row_scale = h->db.p_row;
    dn.skip_rows_upto = fp4 ? kGemvMaxRows : 0;
    if (fp4) LMOE_TRY(launch_gemv_fp4(dn, h->status, h->timeout_ns, h->num_sms, s));
    LMOE_TRY(launch_tc_swap(dn, h->status, h->timeout_ns, h->num_sms, s));
    stage_end(h, kStDown, s);
    h->last_launches += fp4 ? 4 : 2;
  } else if (tc) {
    const bool fp4 = c.routed_w == LMOE_MXFP4;
    TcGemm g = {};
    g.epi = fp4 ? kEpiGluF16 : kEpiGluBF16;
    g.M = rows; g.N = hdim; g.K = l;
    g.A = op2d(h->z_perm, rows, l);
    g.B0 = op3d(w->routed_gate_up, c.num_experts, 2 * hdim, l);
    g.ab_f16 = fp4;
    g.b_scale = fp4 ? w->routed_gate_up_scale : nullptr;
    g.k0_len = l; g.k0_per_group = l; g.glu_h = hdim;
    g.tiles = h->db.tiles; g.num_tiles = h->db.num_tiles; g.offsets = h->db.offsets; g.max_tiles = h->max_tiles;
    g.C = h->a; g.ldc = hdim;
    LMOE_TRY(run_tc_gemm(h, g, inject_routed, &h->last_launches, s));
    stage_end(h, kStGlu, s);

    TcGemm dn = {};
    dn.epi = fp4 ? kEpiScaleF16 : kEpiScaleBF16;
    dn.M = rows; dn.N = l; dn.K = hdim;
    dn.A = op2d(h->a, rows, hdim);
    dn.B0 = op3d(w->routed_down, c.num_experts, l, hdim);
    dn.ab_f16 = fp4;
    dn.b_scale = fp4 ? w->routed_down_scale : nullptr;
    dn.k0_len = hdim; dn.k0_per_group = hdim;
    dn.tiles = h->db.tiles; dn.num_tiles = h->db.num_tiles; dn.offsets = h->db.offsets; dn.max_tiles = h->max_tiles;
    dn.C = o; dn.ldc = l; dn.row_scale = h->db.p_row;
    LMOE_TRY(run_tc_gemm(h, dn, 0, &h->last_launches, s));
    stage_end(h, kStDown, s);
  } else {
    SimtGemm g = {};
    g.A = h->z_perm; g.lda = l; g.a_dtype = c.act; g.b_dtype = c.routed_w;
    g.nseg = 1; g.seg[0] = SimtSegment{w->routed_gate_up, l, (int64_t)2 * hdim * l, l, l};
    g.M = rows; g.N = hdim; g.K = l; g.glu_h = hdim;
    g.tiles = h->db.tiles; g.num_tiles = h->db.num_tiles; g.offsets = h->db.offsets; g.max_tiles = h->max_tiles;
    g.C = h->a; g.ldc = hdim; g.c_dtype = c.act;
    LMOE_TRY(launch_simt_gemm(g, s));
    stage_end(h, kStGlu, s);

    SimtGemm dn = {};
    dn.A = h->a; dn.lda = hdim; dn.a_dtype = c.act; dn.b_dtype = c.routed_w;
    dn.nseg = 1; dn.seg[0] = SimtSegment{w->routed_down, hdim, (int64_t)l * hdim, hdim, hdim};
    dn.M = rows; dn.N = l; dn.K = hdim;
    dn.tiles = h->db.tiles; dn.num_tiles = h->db.num_tiles; dn.offsets = h->db.offsets; dn.max_tiles = h->max_tiles;
    dn.C = o; dn.ldc = l; dn.c_dtype = c.act; dn.row_scale = h->db.p_row;
    LMOE_TRY(launch_simt_gemm(dn, s));
    stage_end(h, kStDown, s);
    h->last_launches += 2;
  }
  // u = sum_j o_j (rank order), n = RMSNorm(u) into the tail columns of act_cat
  LMOE_TRY(launch_combine(o, rt, c.act, h->db.row_of, nullptr, w->rms_gain, c.rms_eps, T, k, l, n_out, kcat, s));
  stage_end(h, kStCombine, s);
  h->last_launches += 1;

  if (tc) {
    if (fork) {
      LMOE_TRY(cudaStreamWaitEvent(s, h->ev_shared, 0));
      join.armed = false;  // every launch of the second stream is now ordered before the rest
    } else if (ns > 0) {
      LMOE_TRY(launch_shared(s));
      stage_end(h, kStSharedGlu, s);
    }
    stage_begin(h, kStFinal, s);
    TcGemm f = {};
    f.epi = kEpiBF16;
    f.M = T; f.N = d; f.K = kcat;
    f.A = op2d(h->act_cat, T, kcat);
    if (ns > 0) {
      f.B0 = op3d(w->shared_down, ns, d, hs);
      f.k0_len = ns * hs; f.k0_per_group = hs;
      f.B1 = op2d(w->w_up_proj, d, l);
    } else {
      f.B0 = op2d(w->w_up_proj, d, l);
      f.k0_len = l; f.k0_per_group = l;
    }
    f.C = y; f.ldc = d;
    LMOE_TRY(run_tc_gemm(h, f, 0, &h->last_launches, s));
    stage_end(h, kStFinal, s);
  } else {
    if (ns > 0) {
      SimtGemm g = {};
      g.A = x; g.lda = d; g.a_dtype = c.act; g.b_dtype = c.act;
      g.nseg = 1; g.seg[0] = SimtSegment{w->shared_gate_up, d, (int64_t)2 * hs * d, d, d};
      g.M = T; g.N = ns * hs; g.K = d; g.glu_h = hs;
      g.C = h->act_cat; g.ldc = kcat; g.c_dtype = c.act;
      LMOE_TRY(launch_simt_gemm(g, s));
      stage_end(h, kStSharedGlu, s);
      h->last_launches += 1;
    }
    stage_begin(h, kStFinal, s);
    SimtGemm f = {};
    f.A = h->act_cat; f.lda = kcat; f.a_dtype = c.act; f.b_dtype = c.act;
    f.nseg = 0;
    if (ns > 0) f.seg[f.nseg++] = SimtSegment{w->shared_down, hs, (int64_t)d * hs, ns * hs, hs};
    f.seg[f.nseg++] = SimtSegment{w->w_up_proj, l, 0, l, l};
    f.M = T; f.N = d; f.K = kcat;
    f.C = y; f.ldc = d; f.c_dtype = c.act;
    LMOE_TRY(launch_simt_gemm(f, s));
    stage_end(h, kStFinal, s);
    h->last_launches += 1;
  }
  stages_finish(h, s);
  return LMOE_OK;
}

void release_streams(lmoe_handle* h) {
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_wdown) cudaEventDestroy(h->ev_wdown);
  if (h->ev_shared) cudaEventDestroy(h->ev_shared);
  if (h->aux) cudaStreamDestroy(h->aux);
  h->ev_fork = h->ev_wdown = h->ev_shared = nullptr;
  h->aux = nullptr;
}

lmoe_status check_call(lmoe_handle* h, const void* x, int32_t T) {
  if (!h) return LMOE_ERR_INVALID_ARG;
  if (T < 0 || T > h->cfg.max_tokens) return LMOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !aligned16(x))) return LMOE_ERR_INVALID_ARG;
  return LMOE_OK;
}

// Makes the handle's device current for one call and gives the caller's current device back
// when the call returns.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      prev = -1;
      return;
    }
    ok = prev == dev || cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

}  // namespace

extern "C" {

lmoe_status latentmoe_create(const lmoe_config* cfg, lmoe_handle** out) {
  if (!cfg || !out) return LMOE_ERR_INVALID_ARG;
  *out = nullptr;
  lmoe_status st = validate_config(*cfg);
  if (st != LMOE_OK) return st;
  lmoe_handle* h = new (std::nothrow) lmoe_handle();
  if (!h) return LMOE_ERR_OOM;
  h->cfg = *cfg;
  h->timeout_ns = kDefaultTimeoutNs;
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    delete h;
    return LMOE_ERR_CUDA;
  }
  h->ws_bytes = layout(h, nullptr);
  if (cudaMalloc(&h->ws, h->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return LMOE_ERR_OOM;
  }
  layout(h, h->ws);
  if (cudaMemset(h->status, 0, sizeof(uint32_t)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
      cudaStreamCreateWithFlags(&h->aux, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_wdown, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_shared, cudaEventDisableTiming) != cudaSuccess) {
    release_streams(h);
    cudaFree(h->ws);
    delete h;
    return LMOE_ERR_CUDA;
  }
  *out = h;
  return LMOE_OK;
}

lmoe_status latentmoe_destroy(lmoe_handle* h) {
  if (!h) return LMOE_OK;
  DeviceGuard dg(h->device);
  cudaError_t e = dg.ok ? cudaDeviceSynchronize() : cudaErrorInvalidDevice;
  release_streams(h);
  cudaFree(h->ws);
  delete h;
  return cuda_status(e);
}

lmoe_status latentmoe_route(lmoe_handle* h, const void* x, int32_t T, const lmoe_weights* w, int32_t* topk_idx,
                            float* topk_p, int32_t* expert_offsets, int32_t* tok_of_row, int32_t* row_of,
                            void* stream) {
  lmoe_status st = check_call(h, x, T);
  if (st != LMOE_OK) return st;
  DeviceGuard dg(h->device);
  if (!dg.ok) return LMOE_ERR_CUDA;
  if (!w || !w->w_router || !aligned16(w->w_router)) return LMOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const lmoe_config& c = h->cfg;
  h->last_launches = 0;
  const size_t rows = (size_t)T * c.top_k;
  if (T > 0) {
    const int32_t* idx;
    const float* p;
    stages_start(h, s);
    st = run_routing(h, x, T, w, nullptr, nullptr, &idx, &p, s);
    if (st != LMOE_OK) return st;
    stages_finish(h, s);
  }
  if (topk_idx && rows) LMOE_TRY(cudaMemcpyAsync(topk_idx, h->idx, rows * 4, cudaMemcpyDeviceToDevice, s));
  if (topk_p && rows) LMOE_TRY(cudaMemcpyAsync(topk_p, h->p, rows * 4, cudaMemcpyDeviceToDevice, s));
  if (expert_offsets) {
    if (T > 0)
      LMOE_TRY(cudaMemcpyAsync(expert_offsets, h->db.offsets, (c.num_experts + 1) * 4, cudaMemcpyDeviceToDevice, s));
    else
      LMOE_TRY(cudaMemsetAsync(expert_offsets, 0, (c.num_experts + 1) * 4, s));
  }
  if (tok_of_row && rows) LMOE_TRY(cudaMemcpyAsync(tok_of_row, h->db.tok_of_row, rows * 4, cudaMemcpyDeviceToDevice, s));
  if (row_of && rows) LMOE_TRY(cudaMemcpyAsync(row_of, h->db.row_of, rows * 4, cudaMemcpyDeviceToDevice, s));
  return LMOE_OK;
}

lmoe_status latentmoe_ep_emulate(lmoe_handle* h, const void* x, int32_t T, const lmoe_weights* w, int32_t ranks,
                                 int32_t full_width, void* send_buf, void* recv_buf, size_t buf_bytes, void* u,
                                 int32_t* cells, void* const* events, void* stream) {
  lmoe_status st = check_call(h, x, T);
  if (st != LMOE_OK) return st;
  DeviceGuard dg(h->device);
  if (!dg.ok) return LMOE_ERR_CUDA;
  const lmoe_config& c = h->cfg;
  const int E = c.num_experts, k = c.top_k, d = c.d, l = c.latent;
  if (!w || !w->w_router || !aligned16(w->w_router) || !w->w_down_proj || !aligned16(w->w_down_proj) ||
      (w->router_bias && !aligned16(w->router_bias)))
    return LMOE_ERR_INVALID_ARG;
  if (ranks < 1 || ranks > kMaxEpRanks || E % ranks || T % ranks || (full_width != 0 && full_width != 1))
    return LMOE_ERR_INVALID_ARG;
  const bool tc = c.act == LMOE_BF16;
  const int row_dtype = full_width ? c.act : routed_act_dtype(c);
  const int width = full_width ? d : l;
  const int row_bytes = width * (int)dtype_bytes(row_dtype);
  const int64_t rows = (int64_t)T * k;
  if (row_bytes % 16 || (T > 0 && (!send_buf || !recv_buf || !u || !aligned16(send_buf) || !aligned16(recv_buf) ||
                                   !aligned16(u) || buf_bytes < (size_t)rows * row_bytes)))
    return LMOE_ERR_INVALID_ARG;
  if (events)
    for (int i = 0; i < 6; ++i)
      if (!events[i]) return LMOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto mark = [&](int i) { return events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) : cudaSuccess; };
  h->last_launches = 0;
  h->last_T = T;
  if (T == 0) return LMOE_OK;
  LMOE_TRY(mark(0));
  const int32_t* idx;
  const float* p;
  st = run_routing(h, x, T, w, nullptr, nullptr, &idx, &p, s);
  if (st != LMOE_OK) return st;
  if (!full_width) {  // the latent rows z = W_down x
    if (tc) {
      TcGemm g = {};
      g.epi = row_dtype == kF16 ? kEpiF16 : kEpiBF16;
      g.M = T; g.N = l; g.K = d;
      g.A = op2d(x, T, d);
      g.B0 = op2d(w->w_down_proj, l, d);
      g.k0_len = d; g.k0_per_group = d;
      g.C = h->z; g.ldc = l;
      LMOE_TRY(run_tc_gemm(h, g, 0, &h->last_launches, s));
    } else {
      SimtGemm g = {};
      g.A = x; g.lda = d; g.a_dtype = c.act; g.b_dtype = c.act;
      g.nseg = 1; g.seg[0] = SimtSegment{w->w_down_proj, d, 0, d, d};
      g.M = T; g.N = l; g.K = d;
      g.C = h->z; g.ldc = l; g.c_dtype = c.act;
      LMOE_TRY(launch_simt_gemm(g, s));
      h->last_launches += 1;
    }
  }
  LMOE_TRY(mark(1));
  const void* src = full_width ? x : h->z;
  LMOE_TRY(launch_ep_plan(h->db.offsets, h->db.tok_of_row, T, E, ranks, h->ep_plan, s));
  LMOE_TRY(launch_ep_pack(src, row_bytes, row_bytes, h->idx, h->db.row_of, h->db.offsets, h->ep_plan, T, E, ranks, k,
                          send_buf, h->ep_row_of, h->num_sms, s));
  LMOE_TRY(mark(2));
  LMOE_TRY(launch_ep_exchange(send_buf, recv_buf, row_bytes, rows, h->ep_plan, E, ranks, 1, h->num_sms, s));
  LMOE_TRY(mark(3));
  // identity experts: the received rows return as the experts' outputs, into send order
  LMOE_TRY(launch_ep_exchange(recv_buf, send_buf, row_bytes, rows, h->ep_plan, E, ranks, 0, h->num_sms, s));
  LMOE_TRY(mark(4));
  LMOE_TRY(launch_combine(send_buf, row_dtype, c.act, h->ep_row_of, p, nullptr, 0.f, T, k, width, u, width, s));
  LMOE_TRY(mark(5));
  h->last_launches += 5;
  if (cells)
    LMOE_TRY(cudaMemcpyAsync(cells, h->ep_plan + (size_t)2 * E * ranks, (size_t)ranks * ranks * 4,
                             cudaMemcpyDeviceToDevice, s));
  return LMOE_OK;
}

lmoe_status latentmoe_forward(lmoe_handle* h, const void* x, int32_t T, const lmoe_weights* w, void* y,
                              void* stream) {
  lmoe_status st = check_call(h, x, T);
  if (st != LMOE_OK) return st;
  DeviceGuard dg(h->device);
  if (!dg.ok) return LMOE_ERR_CUDA;
  if (!weights_ok(h, w, true) || (T > 0 && (!y || !aligned16(y)))) return LMOE_ERR_INVALID_ARG;
  h->last_launches = 0;
  if (T == 0) return LMOE_OK;
  return run_forward(h, x, T, w, nullptr, nullptr, y, static_cast<cudaStream_t>(stream));
}

lmoe_status latentmoe_forward_routed(lmoe_handle* h, const void* x, int32_t T, const lmoe_weights* w,
                                     const int32_t* topk_idx, const float* topk_p, void* y, void* stream) {
  lmoe_status st = check_call(h, x, T);
  if (st != LMOE_OK) return st;
  DeviceGuard dg(h->device);
  if (!dg.ok) return LMOE_ERR_CUDA;
  if (!weights_ok(h, w, false) || (T > 0 && (!y || !aligned16(y) || !topk_idx || !topk_p)))
    return LMOE_ERR_INVALID_ARG;
  h->last_launches = 0;
  if (T == 0) return LMOE_OK;
  return run_forward(h, x, T, w, topk_idx, topk_p, y, static_cast<cudaStream_t>(stream));
}

lmoe_status latentmoe_forward_host(lmoe_handle* h, const void* x_host, int32_t T, const lmoe_weights* w,
                                   void* y_host, void* stream) {
  if (!h) return LMOE_ERR_INVALID_ARG;
  if (T < 0 || T > h->cfg.max_tokens || (T > 0 && (!x_host || !y_host))) return LMOE_ERR_INVALID_ARG;
  if (!weights_ok(h, w, true)) return LMOE_ERR_INVALID_ARG;
  DeviceGuard dg(h->device);
  if (!dg.ok) return LMOE_ERR_CUDA;
  h->last_launches = 0;
  if (T == 0) return LMOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const lmoe_config& c = h->cfg;
  const size_t ab = dtype_bytes(c.act);
  const bool identity = (c.flags & LMOE_FLAG_IDENTITY_EXPERTS) != 0;
  const size_t in_bytes = (size_t)T * c.d * ab;
  const size_t out_bytes = (size_t)T * (identity ? c.latent : c.d) * ab;
  LMOE_TRY(cudaMemcpyAsync(h->x_stage, x_host, in_bytes, cudaMemcpyHostToDevice, s));
  lmoe_status st = run_forward(h, h->x_stage, T, w, nullptr, nullptr, h->y_stage, s);
  if (st != LMOE_OK) return st;
  LMOE_TRY(cudaMemcpyAsync(y_host, h->y_stage, out_bytes, cudaMemcpyDeviceToHost, s));
  LMOE_TRY(cudaStreamSynchronize(s));
  return LMOE_OK;
}

lmoe_status latentmoe_status(lmoe_handle* h, void* stream) {
  if (!h) return LMOE_ERR_INVALID_ARG;
  DeviceGuard dg(h->device);
  if (!dg.ok) return LMOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  LMOE_TRY(cudaStreamSynchronize(s));
  LMOE_TRY(cudaMemcpy(&word, h->status, sizeof(word), cudaMemcpyDeviceToHost));
  LMOE_TRY(cudaMemset(h->status, 0, sizeof(word)));
  if (word & kStatusTimeout) return LMOE_ERR_TIMEOUT;
  if (word & kStatusDeviceCheck) return LMOE_ERR_DEVICE_CHECK;
  return LMOE_OK;
}

int32_t latentmoe_last_launch_count(const lmoe_handle* h) { return h ? h->last_launches : 0; }

size_t latentmoe_workspace_bytes(const lmoe_handle* h) { return h ? h->ws_bytes : 0; }

lmoe_status latentmoe_set_wait_limit(lmoe_handle* h, uint64_t timeout_ns, int32_t inject) {
  if (!h || timeout_ns == 0) return LMOE_ERR_INVALID_ARG;
  if (inject < 0 || inject > 2) return LMOE_ERR_INVALID_ARG;
  h->timeout_ns = timeout_ns;
  h->inject = inject;
  return LMOE_OK;
}

lmoe_status latentmoe_set_stage_events(lmoe_handle* h, void* const* events, int32_t n_events) {
  if (!h) return LMOE_ERR_INVALID_ARG;
  if (!events) {
    h->stage_on = false;
    return LMOE_OK;
  }
  if (n_events < LMOE_NUM_STAGES + 1) return LMOE_ERR_INVALID_ARG;
  for (int i = 0; i <= LMOE_NUM_STAGES; ++i) {
    if (!events[i]) return LMOE_ERR_INVALID_ARG;
    h->stage_ev[i] = static_cast<cudaEvent_t>(events[i]);
  }
  h->stage_on = true;
  return LMOE_OK;
}

lmoe_status latentmoe_debug_buffer(const lmoe_handle* h, const char* name, void** ptr, size_t* bytes) {
  if (!h || !name || !ptr || !bytes) return LMOE_ERR_INVALID_ARG;
  const lmoe_config& c = h->cfg;
  const size_t T = (size_t)h->last_T, k = (size_t)c.top_k, ab = dtype_bytes(c.act);
  const size_t kcat = (size_t)c.num_shared * c.shared_hidden + c.latent;
  void* p = nullptr;
  size_t n = 0;
  if (!strcmp(name, "logits")) { p = h->logits; n = T * c.num_experts * 4; }
  else if (!strcmp(name, "z")) { p = h->z; n = T * c.latent * ab; }
  else if (!strcmp(name, "gathered")) { p = h->z_perm; n = T * k * c.latent * ab; }
  else if (!strcmp(name, "act")) { p = h->a; n = T * k * (size_t)c.hidden * ab; }
  else if (!strcmp(name, "act_cat")) { p = h->act_cat; n = T * kcat * ab; }
  else if (!strcmp(name, "p_row")) { p = h->db.p_row; n = T * k * 4; }
  else if (!strcmp(name, "refine_count")) { p = h->refine_count; n = 2 * sizeof(int32_t); }
  if (!p) return LMOE_ERR_INVALID_ARG;
  *ptr = p;
  *bytes = n;
  return LMOE_OK;
}

const char* latentmoe_stage_name(int32_t i) {
  return (i >= 0 && i < LMOE_NUM_STAGES) ? kStageNames[i] : nullptr;
}

const char* latentmoe_status_string(lmoe_status s) {
  switch (s) {
    case LMOE_OK: return "ok";
    case LMOE_ERR_INVALID_ARG: return "invalid argument";
    case LMOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case LMOE_ERR_CUDA: return "CUDA error";
    case LMOE_ERR_OOM: return "out of device memory";
    case LMOE_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
    case LMOE_ERR_DEVICE_CHECK: return "a kernel rejected its input";
  }
  return "unknown status";
}

}  // extern "C"
