// Host-side launchers shared between the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace lmoe {

// ---------------------------------------------------------------- per-device launch setup
// A kernel's launch attributes (the dynamic shared-memory opt-in) and occupancy queries belong
// to a device: a launcher keeps one value per device, 0 until that device is set up.  Two
// threads setting up the same device at once only repeat idempotent runtime calls.
constexpr int kMaxSetupDevices = 64;
struct PerDeviceValue {
  std::atomic<int> v[kMaxSetupDevices];
  PerDeviceValue() {
    for (auto& x : v) x.store(0, std::memory_order_relaxed);
  }
  // The slot of the current device, or nullptr when there is none.
  std::atomic<int>* current() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxSetupDevices) return nullptr;
    return &v[d];
  }
};

// ---------------------------------------------------------------- routing (route.cu)
// Split-K partial sums of a GEMM left for the consumer to add: output [row][col] = sum over
// s = 0..splits-1, in that order, of part[s * split_stride + row * ldp + col].  splits == 0: the
// output was written whole (no split).
struct SplitPartials {
  const float* part;
  int splits;
  int64_t split_stride, ldp;
};
// logits[T][E] = x[T][d] . W_r[E][d]^T in fp32 (CUDA cores, fixed K order per output).
cudaError_t launch_router_logits(const void* x, int x_dtype, const void* w_router, int w_dtype, float* logits,
                                 int T, int E, int d, cudaStream_t s);
// Router logits for either activation type: bf16 activations use the tensor cores (an fp32 W_r
// is first split into three bf16 terms in `wr_split`, [3][E][d] bf16, then contracted over
// K = 3d), fp32 activations the CUDA-core GEMM.  Adds its kernel count to *launches.
// With `pair_ok`, a router GEMM of at least 256 rows whose 128-row tiles would more than half
// fill the SMs runs on CTA pairs; fewer tiles split K on single CTAs (`splitk` workspace).
// With `defer` (non-null) a split-K router GEMM leaves its partial sums unreduced and describes
// them there (the short-batch top-k adds them); defer->splits == 0 when logits were written.
cudaError_t launch_router(const void* x, int act, const void* w_router, int router_w, float* logits,
                          void* wr_split, int T, int E, int d, uint32_t* status, uint64_t timeout_ns, int num_sms,
                          int* launches, cudaStream_t s, float* splitk = nullptr, size_t splitk_bytes = 0,
                          bool pair_ok = false, SplitPartials* defer = nullptr);
// Exact split of fp32 W_r into three bf16 terms, out[t][e][c], t = hi, mid, lo:
// w = hi + mid + lo with each term the bf16 rounding of what the previous terms left.
cudaError_t launch_split_bf16x3(const float* w, int64_t n, void* out, cudaStream_t s);
// Operands of the router GEMM, for exact recomputation of logits near the top-k boundary.
struct RouterSrc {
  const void* x; int x_dtype;  // [T][d]
  const void* w; int w_dtype;  // [E][d]
  int d;
  float margin;                // bound on |logits[t][e] - exact logit|
};
// Logit error bound used for the router GEMMs (tensor cores with fp32 accumulation, or the
// fp32 CUDA-core GEMM): measured errors are below 1e-4 at d = 7168 (tested).
constexpr float kRouterLogitMargin = 1e-3f;
// s = sigmoid(logits), key = s + b, top-k by (key desc, index asc), p = s / sum(s over T_k);
// wherever two keys that decide the selected set or the rank order are within the key
// uncertainty the margin implies, they are compared as exact fp64 keys.
// Two kernels: a selection pass that appends tokens with an uncertain list to refine_list[T],
// and a refinement pass over that list.  refine_count[0] is the list length and refine_count[1]
// the number of near ties (exact k-th/(k+1)-th key gap below 1e-6); both are reset here.  A
// recomputed logit further than margin/2 from the GEMM's sets kStatusDeviceCheck |
// kStatusRouterMargin in *status (may be null).
// Batches of at most kTopkFusedMaxT tokens run both passes in one kernel; there `part` (when its
// splits > 0) holds the router GEMM's unreduced split-K sums, which the kernel adds in split order
// (the arithmetic of the split-K reduction) and writes to `logits`.
constexpr int kTopkFusedMaxT = 512;
cudaError_t launch_topk(float* logits, const float* bias, const RouterSrc& src, int T, int E, int k, int32_t* idx,
                        float* p, int32_t* refine_list, int32_t* refine_count, uint32_t* status, int num_sms,
                        cudaStream_t s, const SplitPartials* part = nullptr);
// Deterministic expert batches: per-chunk counts, scan, stable (expert, token) rows, the
// grouped-GEMM M-tile list, and per-row weights.  idx entries outside [0,E) are reported.
struct DispatchBuffers {
  int32_t* chunk_counts;  // [nchunks][E]
  int32_t* chunk_base;    // [nchunks][E]
  int32_t* offsets;       // [E+1]
  int4* tiles;            // [max_tiles]: {expert, first m-tile of expert, rows of expert, first row}
  int32_t* num_tiles;     // [1]
  int4* tiles_s;          // [T*k/16 + E + 1]: {expert, first row, rows (<= 16), 0}
  int32_t* num_tiles_s;   // [1]
  int4* tiles_p;          // [T*k/256 + E + 1]: 256-row tiles, same layout as `tiles` (or nullptr)
                          // (one load gives a work item everything: the tile count is ceil(rows / tile))
  int32_t* num_tiles_p;   // [1]
  int4* tiles_m;          // [T*k/192 + E + 1]: 192-row tiles of the block-scaled kernel, same layout (or nullptr)
  int32_t* num_tiles_m;   // [1]
  int32_t* tok_of_row;    // [T*k]
  int32_t* row_of;        // [T][k]
  float* p_row;           // [T*k]
};
cudaError_t launch_dispatch(const int32_t* idx, const float* p, int T, int E, int k, const DispatchBuffers& b,
                            uint32_t* status, int* launches, cudaStream_t s);
// dst[row_of[t][j]] = src[t] for every (t, j) with row_of[t][j] >= 0: rows of `width` elements of
// `elem_bytes` (a multiple of 16 bytes, at most 16 KB; 16-byte aligned buffers; k <= 32).
cudaError_t launch_scatter_rows(const void* src, void* dst, const int32_t* row_of, int T, int k, int width,
                                int elem_bytes, uint32_t* status, uint64_t timeout_ns, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------- combine (combine.cu)
// u_t = sum_j o[row_of[t][j]] (rank order, fp32) [times p[t][j] when p != nullptr];
// with gain != nullptr writes n_t = u_t * g / sqrt(mean(u_t^2) + eps), else u_t.
// in_dtype: kF32, kBF16 or kF16 (expert rows); out_dtype: kF32 or kBF16.
cudaError_t launch_combine(const void* o, int in_dtype, int out_dtype, const int32_t* row_of, const float* p,
                           const float* gain, float eps, int T, int k, int width, void* out, int64_t ld_out,
                           cudaStream_t s);

// ---------------------------------------------------------------- expert-parallel emulation (ep_emulate.cu)
// R virtual ranks over T/R tokens and E/R experts each (T % R == 0, E % R == 0, R <= kMaxEpRanks).
constexpr int kMaxEpRanks = 64;
size_t ep_plan_ints(int E, int R);
// Plan from the dispatch's expert offsets and expert-sorted tokens (one CTA).
cudaError_t launch_ep_plan(const int32_t* offsets, const int32_t* tok_of_row, int T, int E, int R, int32_t* plan,
                           cudaStream_t s);
// Token rows (src + t * src_ld_bytes, row_bytes each, a multiple of 16) into the send buffer
// ordered (source rank, destination rank, expert, token); ep_row_of[t][j] = send position.
cudaError_t launch_ep_pack(const void* src, int64_t src_ld_bytes, int row_bytes, const int32_t* idx,
                           const int32_t* row_of, const int32_t* offsets, const int32_t* plan, int T, int E, int R,
                           int k, void* send, int32_t* ep_row_of, int num_sms, cudaStream_t s);
// forward: send -> recv (destination rank, source rank) order; backward: recv -> send order.
cudaError_t launch_ep_exchange(const void* from, void* to, int row_bytes, int64_t rows, const int32_t* plan, int E,
                               int R, int forward, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------- fp32 CUDA-core GEMM (simt.cu)
struct SimtSegment {
  const void* ptr;        // B segment: element (group g, row n, col c) at ptr + g*group_stride + n*ld + c
  int64_t ld;
  int64_t group_stride;
  int k_len;              // K extent of this segment
  int k_per_group;        // K columns per group inside the segment (segment spans k_len/k_per_group groups)
};
struct SimtGemm {
  const void* A; int64_t lda; int a_dtype;
  int b_dtype;
  int nseg; SimtSegment seg[6];
  int M, N, K;            // N = output columns
  int glu_h;              // > 0: gate rows j, up rows j + glu_h of the group; out = SiLU(gate)*up
  const int4* tiles; const int32_t* num_tiles; const int32_t* offsets; int max_tiles;  // grouped mode
  void* C; int64_t ldc; int c_dtype;
  const float* row_scale; // per output row multiplier (or nullptr)
};
cudaError_t launch_simt_gemm(const SimtGemm& g, cudaStream_t s);

// ---------------------------------------------------------------- tcgen05 GEMM (gemm_tc.cu)
enum TcEpilogue : int {
  kEpiF32 = 0,        // fp32 store (router logits)
  kEpiBF16 = 1,       // bf16 store
  kEpiGluBF16 = 2,    // SiLU(gate) * up, bf16
  kEpiScaleBF16 = 3,  // row_scale[r] * acc, bf16
  kEpiF16 = 4,        // fp16 variants of the above
  kEpiGluF16 = 5,
  kEpiScaleF16 = 6
};
struct TcOperand {        // a 16-bit (or packed E2M1) tensor viewed as [depth][rows][cols], cols = K contiguous
  const void* ptr;
  int64_t cols, rows, depth;
  int64_t row_stride;     // elements
  int64_t depth_stride;   // elements
};
struct TcGemm {
  int epi;
  int M, N, K;            // N = output columns (GLU: hidden outputs); K multiple of 64
  TcOperand A;            // [1][rows][K]
  TcOperand B0, B1;       // B1.ptr == nullptr when K has a single segment
  int k0_len;             // K columns served by B0 (multiple of 64)
  int k0_per_group;       // B0 K columns per depth slice (K-concatenated groups), else k0_len
  int a_k_period;         // A's K coordinate wraps every a_k_period columns (0 = K: no wrap)
  int glu_h;              // GLU: rows of B between gate and up; output column j -> (j / glu_h, j % glu_h)
  const int4* tiles; const int32_t* num_tiles; const int32_t* offsets; int max_tiles;  // grouped mode
  void* C; int64_t ldc;
  const float* row_scale;
  int ab_f16;                // operands are fp16 (with MXFP4 B) instead of bf16
  const uint8_t* b_scale;    // non-null: B0 holds packed E2M1 bytes, b_scale E8M0 [depth][rows][K/32]
  float* partial;            // split-K workspace (dense GEMMs of few tiles) or nullptr: no split
  size_t partial_bytes;      // its size (tc_splitk_partial_bytes)
  SplitPartials* defer;      // non-null (fp32 epilogue): leave split-K sums unreduced, described here
  int* launch_count;         // incremented by the number of kernels launched (or nullptr)
};
// Workspace the split-K path needs at most (splits x tiles <= SMs, 128 rows x 256 fp32 columns each).
size_t tc_splitk_partial_bytes(int num_sms);
cudaError_t launch_tc_gemm(const TcGemm& g, uint32_t* status, uint64_t timeout_ns, int inject_fault, int num_sms,
                           cudaStream_t s);

// The same GEMM on CTA pairs (gemm_pair.cu): 256 x 256 tiles, tcgen05.mma.cta_group::2.  Dense
// (not grouped), bf16 operands, bf16, GLU or fp32 epilogue; tc_pair_supported says whether `g`
// qualifies.
// inject != 0 (test hook): the first pair skips its first ring stage, so that its MMA's bounded
// wait runs out and reports a timeout.
bool tc_pair_supported(const TcGemm& g);
cudaError_t launch_tc_pair(const TcGemm& g, uint32_t* status, uint64_t timeout_ns, cudaStream_t s, int inject = 0);

// Swapped-operand grouped GEMM for experts with few rows (gemm_swap.cu): weights are the
// 128-row M operand, the tile's token rows (up to 128) the N operand.
struct TcSwap {
  int epi;                  // kEpiGlu{BF16,F16} (output h features) or kEpiScale{BF16,F16}
  int K;                    // reduction width
  int out_features;         // h for gate/up, l for down
  TcOperand act;            // [rows][K] 16-bit token rows (expert-contiguous)
  TcOperand w;              // [E][w_rows][K] weights (16-bit, or packed E2M1 when w_scale)
  const uint8_t* w_scale;   // E8M0 [E][w_rows][K/32] or nullptr
  int ab_f16;
  int glu_h;
  const int4* tiles_s; const int32_t* num_tiles_s; int max_tiles_s;  // 16-row units
  int skip_rows_upto;       // units with at most this many rows are left to the CUDA-core kernel
  void* C; int64_t ldc;
  const float* row_scale;   // down: routing weight per row
};
cudaError_t launch_tc_swap(const TcSwap& g, uint32_t* status, uint64_t timeout_ns, int num_sms, cudaStream_t s,
                           int inject = 0);
// MXFP4 routed experts for units of at most 4 rows on the CUDA cores (gemv_fp4.cu): the same
// descriptor as launch_tc_swap (kEpiGluF16 or kEpiScaleF16, fp16 activations, K % 512 == 0,
// K <= 4096); units with more rows are skipped (run launch_tc_swap with skip_rows_upto = 4).
constexpr int kGemvMaxRows = 4;
cudaError_t launch_gemv_fp4(const TcSwap& g, uint32_t* status, uint64_t timeout_ns, int num_sms, cudaStream_t s,
                            int inject = 0);

// The same swapped-operand grouped GEMM on CTA pairs for experts with many rows
// (gemm_pair_swap.cu): 256 weight rows x up to 256 token rows per tile, each expert's rows cut
// into ceil(rows/256) equal token tiles (tiles_p: the dispatch's 256-row tile list).  bf16 only
// (kEpiGluBF16 with glu_h % 128 == 0, or kEpiScaleBF16 with out_features % 256 == 0).
cudaError_t launch_tc_pair_swap(const TcSwap& g, const int4* tiles_p, const int32_t* num_tiles_p, int max_tiles_p,
                                uint32_t* status, uint64_t timeout_ns, cudaStream_t s, int inject = 0);

// ---------------------------------------------------------------- block-scaled MXFP4 experts
// Three-term MXFP4 records of token rows (mx.cuh): rows of z in expert-contiguous order.  z
// [T][K] fp16 or bf16 (K % 512 == 0); dst[row_of[t][j]] = record of z[t] for every (t, j) with
// row_of[t][j] >= 0.  k <= 32.  f8: MXFP8 records (mx8_row_bytes) instead.
size_t scatter_mx3_smem_bytes(int K, int in_elem_bytes, bool f8 = false);
cudaError_t launch_scatter_mx3(const void* src, int src_dtype, void* dst, const int32_t* row_of, int T, int k, int K,
                               uint32_t* status, uint64_t timeout_ns, int num_sms, cudaStream_t s, bool f8 = false);
// Grouped expert GEMM on tcgen05.mma.cta_group::2.kind::mxf4 (gemm_mx.cu): E2M1 weights with E8M0
// scales per 32 along K against token records.  unit_rows 192: the dispatch's 192-row tile list
// (tiles_m; prefill); unit_rows 16: its 16-row unit list (tiles_s; decode, a deep weight ring).
//   glu_h > 0: gate/up weights [E][2h][K] (out_features == glu_h, multiple of 512); C receives
//              the records of SiLU(gate) * up ([rows][mx3_row_bytes(h)]).
//   glu_h == 0: down weights [E][out_features][K]; C receives fp16 rows [rows][ldc], each scaled
//              by row_scale[row].
struct TcMx {
  int K;                    // reduction width (multiple of 512)
  int out_features;
  int glu_h;
  TcOperand w;              // [E][w_rows][K] in elements (packed E2M1 bytes)
  const uint8_t* w_scale;   // E8M0 [E][w_rows][K/32]
  const void* x;            // token records [rows][mx3_row_bytes(K)]
  int64_t rows;             // rows of x
  void* C;
  int64_t ldc;              // down: fp16 elements per output row
  const float* row_scale;
  bool f8;                  // token records are MXFP8 (kind::mxf8f6f4) instead of three-term MXFP4
};
cudaError_t launch_tc_mx(const TcMx& g, const int4* tiles, const int32_t* num_tiles, int max_tiles, int unit_rows,
                         uint32_t* status, uint64_t timeout_ns, cudaStream_t s, int inject = 0);

}  // namespace lmoe
