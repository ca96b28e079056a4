/*
 * latentmoe.h - C ABI of the LatentMoE layer forward pass on one GB300 GPU (sm_103a).
 *
 * The layer (page "Lesson 6 - LatentMoE", kimi-k3-course.pages.dev, section
 * "show me the actual equation", eq. 11 and eq. 13, quoting the K3 report section 2.3):
 *
 *   s    = Sigmoid(W_r x)                       router scores, one per routed expert
 *   T_k  = argtopk(s + b)                       b steers selection only (eq. 13)
 *   p_i  = s_i / sum_{r in T_k} s_r             weights over the selected set (eq. 13)
 *   z    = W_down x                             d -> latent width l, before dispatch
 *   u    = sum_{i in T_k} p_i E_i(z)            routed GLU experts in latent space (eq. 11)
 *   y    = sum_{j<N_s} S_j(x) + W_up RMSNorm(u) shared full-width GLU experts + up-projection
 *
 * with E(v) = D( SiLU(G v) * (U v) ) for every expert, and
 * RMSNorm(u) = u * g / sqrt(mean(u^2) + eps) (section "What extreme sparsity breaks":
 * the norm sits between aggregation and W_up).
 *
 * Conventions for every entry point
 *  - Matrices are row-major [out][in] (K contiguous).  All tensor pointers are DEVICE
 *    pointers unless the name ends in _host; device pointers must be 16-byte aligned.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *    default stream).  A handle must not be used from two streams at once and is not
 *    thread-safe.  A handle's calls run on the device that was current at create time
 *    (stream and buffers must belong to it); the caller's current device is restored
 *    before each call returns.
 *  - The caller owns x, y, the weights and any routing buffers; the handle owns its
 *    workspace (sized at create time for cfg.max_tokens) and a device status word.
 *  - Every call returns an lmoe_status and never throws across the ABI.  Argument errors
 *    are detected on the host before any launch and leave outputs untouched.  Errors a
 *    kernel detects (a bounded wait that ran out, an out-of-range routing index) are sticky
 *    in the device status word and are reported by latentmoe_status().
 */
#ifndef LATENTMOE_H
#define LATENTMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LMOE_OK = 0,
  LMOE_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or config field           */
  LMOE_ERR_UNSUPPORTED = 2,   /* valid but not implemented (shape/dtype combination)     */
  LMOE_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed                       */
  LMOE_ERR_OOM = 4,           /* workspace allocation failed                             */
  LMOE_ERR_TIMEOUT = 5,       /* a kernel's bounded wait ran out (device status word)    */
  LMOE_ERR_DEVICE_CHECK = 6   /* a kernel rejected its input (e.g. routing index >= E),  */
                              /* or a router logit recomputed exactly was further from   */
                              /* the GEMM's than half the error margin selection assumes */
} lmoe_status;

typedef enum {
  LMOE_F32 = 0,               /* IEEE fp32                                               */
  LMOE_BF16 = 1,              /* bfloat16                                                */
  LMOE_MXFP4 = 2,             /* OCP MXFP4: E2M1 pairs per byte (element 2i in the low    */
                              /* nibble) + one E8M0 scale byte per 32 elements along K   */
  LMOE_F16 = 3                /* IEEE fp16 (latentmoe_mx3_quantize input only)           */
} lmoe_dtype;

/* Routed experts are the identity map: forward() returns u = sum_i p_i z (width l) and
 * stops there (no RMSNorm, W_up or shared experts).  Used by the routing/dispatch
 * stress workload. */
#define LMOE_FLAG_IDENTITY_EXPERTS 0x1u
/* Run every tensor-core GEMM on single CTAs (128-row tiles) instead of CTA pairs (256-row
 * tiles, tcgen05 cta_group::2) where the latter would apply.  Same results up to fp32
 * accumulation order; for comparison and testing. */
#define LMOE_FLAG_SINGLE_CTA_GEMM 0x2u
/* MXFP4 routed experts: decode the E2M1 weights to fp16 in shared memory and run fp16 MMAs
 * (kind::f16), or a CUDA-core GEMV for decode units of at most 4 rows, instead of the default
 * block-scaled kind::mxf4 MMAs on three-term MXFP4 activations.  For comparison and testing. */
#define LMOE_FLAG_MXFP4_DEQUANT 0x4u
/* MXFP4 experts with MXFP8 activations (bf16 layers only): the expert inputs and the GLU
 * activations become MXFP8 records (E4M3 elements, one E8M0 scale per 32, round to nearest
 * even, the smallest power-of-two scale that keeps every element within 448) and the expert
 * GEMMs run tcgen05.mma kind::mxf8f6f4 (E2M1 x E4M3) -- K3's quantisation-aware-training
 * numerics (page "What K3 actually is", srikanthmalla.com: MXFP4 weights with MXFP8
 * activations).  A different numerics mode: it is compared with the oracle's MXFP8 mode, not
 * with the bf16 evaluation. */
#define LMOE_FLAG_MXFP8_ACT 0x8u

typedef struct {
  int32_t d;             /* model width                                                 */
  int32_t latent;        /* l, routed-expert width                                      */
  int32_t hidden;        /* h, routed-expert GLU hidden width (ignored with identity)   */
  int32_t num_experts;   /* E, 1..1024                                                  */
  int32_t top_k;         /* k, 1..min(E, 32)                                            */
  int32_t num_shared;    /* N_s >= 0                                                    */
  int32_t shared_hidden; /* shared-expert GLU hidden width                              */
  int32_t max_tokens;    /* largest T any call will pass (sizes the workspace)          */
  int32_t act;           /* lmoe_dtype of x, y, W_down, W_up, shared experts: F32|BF16 */
  int32_t router_w;      /* lmoe_dtype of W_r: F32|BF16                                 */
  int32_t routed_w;      /* lmoe_dtype of routed experts: F32|BF16|MXFP4 (MXFP4 needs bf16
                            act, l and h multiples of 512, E8M0 scale exponents in
                            [-24, 13]; others set LMOE_ERR_DEVICE_CHECK)                 */
  float rms_eps;         /* RMSNorm epsilon                                             */
  uint32_t flags;        /* LMOE_FLAG_*                                                 */
} lmoe_config;

/* Weight pointers (device, row-major [out][in]); types per lmoe_config. */
typedef struct {
  const void *w_router;                 /* W_r [E][d]                                   */
  const float *router_bias;             /* b [E] fp32, or NULL (= 0); selection only    */
  const void *w_down_proj;              /* W_down [l][d]                                */
  const float *rms_gain;                /* g [l] fp32                                   */
  const void *routed_gate_up;           /* [E][2h][l]: gate rows 0..h-1, up rows h..2h-1;
                                           MXFP4: bytes [E][2h][l/2]                    */
  const uint8_t *routed_gate_up_scale;  /* MXFP4 only: E8M0 [E][2h][l/32]               */
  const void *routed_down;              /* [E][l][h]; MXFP4: bytes [E][l][h/2]          */
  const uint8_t *routed_down_scale;     /* MXFP4 only: E8M0 [E][l][h/32]                */
  const void *w_up_proj;                /* W_up [d][l]                                  */
  const void *shared_gate_up;           /* [N_s][2h_s][d]: gate rows then up rows       */
  const void *shared_down;              /* [N_s][d][h_s]                                */
} lmoe_weights;

typedef struct lmoe_handle lmoe_handle;

/* Validate `cfg`, allocate the workspace for cfg->max_tokens tokens on the current
 * device, and return a handle in *out.  Synchronous.  Errors: INVALID_ARG (bad field),
 * UNSUPPORTED (e.g. widths that do not tile), OOM, CUDA. */
lmoe_status latentmoe_create(const lmoe_config *cfg, lmoe_handle **out);

/* Free the workspace and the handle.  Synchronises the device first.  NULL is a no-op. */
lmoe_status latentmoe_destroy(lmoe_handle *h);

/* Router and dispatch only (eq. 13 and the conversion of selections into expert batches).
 *   x              [T][d] act dtype
 *   topk_idx       [T][k] int32, out: selected experts in rank order (largest s+b first,
 *                  equal keys -> lower expert index first).  Keys closer together than the
 *                  router GEMM's error bound are compared exactly (fp64 from a ~44-bit logit),
 *                  so set and order equal those of an exact evaluation except where the k-th
 *                  and (k+1)-th keys differ by less than 1e-6 (near ties; counted, see
 *                  latentmoe_debug_buffer "refine_count").
 *   topk_p         [T][k] fp32, out: p = s / sum of s over the selected set
 *   expert_offsets [E+1] int32, out: exclusive prefix sum of per-expert row counts
 *   tok_of_row     [T*k] int32, out: token of each row, rows ordered by (expert, token)
 *   row_of         [T][k] int32, out: the row holding (token t, rank j)
 * Any output pointer may be NULL (not written).  0 <= T <= max_tokens. */
lmoe_status latentmoe_route(lmoe_handle *h, const void *x, int32_t T, const lmoe_weights *w,
                            int32_t *topk_idx, float *topk_p, int32_t *expert_offsets,
                            int32_t *tok_of_row, int32_t *row_of, void *stream);

/* The whole layer: y [T][d] act dtype (with LMOE_FLAG_IDENTITY_EXPERTS: u [T][l]).
 * 0 <= T <= max_tokens; T == 0 returns LMOE_OK without launching anything.
 * With bf16 activations, W_down and the shared experts' GLU (they read x only) run on a second
 * stream that the handle owns: it waits for an event recorded on `stream` at the start of the
 * call, and `stream` waits for its events before the expert-row scatter and before the final
 * GEMM, so the call stays ordered on `stream` like a single-stream launch sequence (and can be
 * captured into a CUDA graph from `stream`).  While stage events are set
 * (latentmoe_set_stage_events) every stage runs on `stream`, one after another.  Concurrent calls
 * on one handle are not supported (they share the workspace). */
lmoe_status latentmoe_forward(lmoe_handle *h, const void *x, int32_t T, const lmoe_weights *w,
                              void *y, void *stream);

/* As latentmoe_forward, but with the routing supplied by the caller instead of the
 * router: topk_idx [T][k] int32 (distinct experts per token, each in [0,E)) and topk_p
 * [T][k] fp32.  An index outside [0,E) sets LMOE_ERR_DEVICE_CHECK in the status word and
 * its row is skipped. */
lmoe_status latentmoe_forward_routed(lmoe_handle *h, const void *x, int32_t T, const lmoe_weights *w,
                                     const int32_t *topk_idx, const float *topk_p, void *y,
                                     void *stream);

/* End to end from HOST memory: copies x_host [T][d] to the device, runs the layer, and
 * copies the result back to y_host ([T][d], or [T][l] with identity experts), all on
 * `stream`; returns after the stream has finished.  Weights stay device pointers.
 * Page-locked host buffers give full copy bandwidth. */
lmoe_status latentmoe_forward_host(lmoe_handle *h, const void *x_host, int32_t T, const lmoe_weights *w,
                                   void *y_host, void *stream);

/* Synchronise `stream`, read and clear the device status word, and return the first
 * sticky error (TIMEOUT before DEVICE_CHECK), or LMOE_OK. */
lmoe_status latentmoe_status(lmoe_handle *h, void *stream);

/* Number of kernels the last route/forward call enqueued. */
int32_t latentmoe_last_launch_count(const lmoe_handle *h);

/* Device workspace bytes held by the handle. */
size_t latentmoe_workspace_bytes(const lmoe_handle *h);

/* Test hook: bound every in-kernel wait of later calls to `timeout_ns` nanoseconds
 * (default 4e9).  With inject = 1 the next forward's first routed GEMM kernel(s), with
 * inject = 2 its W_down GEMM, skip the loads and the signal of one pipeline stage in their first
 * CTA (or CTA pair), so that the consumer's bounded wait runs out and reports LMOE_ERR_TIMEOUT;
 * the kernel waits (bounded) for its own loads and MMAs in flight before it exits.  No fault,
 * trap or hang results; other tiles complete normally.  inject outside 0..2: INVALID_ARG. */
lmoe_status latentmoe_set_wait_limit(lmoe_handle *h, uint64_t timeout_ns, int32_t inject);

/* Stage timing.  With `events` non-NULL (n_events >= LMOE_NUM_STAGES + 1 cudaEvent_t
 * handles created by the caller, passed as void*), later route/forward calls record
 * events[0] on `stream` before their first launch and events[i+1] after stage i, so that
 * cudaEventElapsedTime(events[i], events[i+1]) is the device time of stage i on the
 * launching stream.  Stages a call does not run are recorded back to back (zero time).
 * NULL switches recording off.  The handle does not own the events. */
#define LMOE_NUM_STAGES 10
lmoe_status latentmoe_set_stage_events(lmoe_handle *h, void *const *events, int32_t n_events);

/* Name of stage i (0 <= i < LMOE_NUM_STAGES): router_logits, topk, dispatch, w_down,
 * scatter_rows, routed_gate_up_glu, routed_down, combine_rmsnorm, shared_gate_up_glu,
 * final_gemm; NULL otherwise. */
const char *latentmoe_stage_name(int32_t i);

/* Expert-parallel dispatch and combine emulated on one GPU, to measure the all-to-all payload
 * at the latent width against the full width (page "What K3 actually is", srikanthmalla.com,
 * opening section: a routed token crosses the expert-parallel all-to-all at the experts' input
 * width; page "Lesson 6 - LatentMoE", kimi-k3-course.pages.dev, table "What scales with what").
 * `ranks` virtual ranks: rank r owns tokens [r T/ranks, (r+1) T/ranks) and experts
 * [r E/ranks, (r+1) E/ranks) (T % ranks == 0, E % ranks == 0, 1 <= ranks <= 64).  The call
 * routes x (router, top-k, dispatch), forms one row per selected (token, expert) pair -- the
 * latent row z = W_down x (full_width 0: l values of the routed-expert activation dtype, fp16
 * with MXFP4 experts) or x itself (full_width 1: d values, act dtype) -- packs each source
 * rank's rows into send_buf ordered (destination rank, expert, token), exchanges them
 * (send_buf -> recv_buf, the all-to-all), returns them unchanged as the outputs of identity
 * experts (recv_buf -> send_buf) and combines each token's k rows in rank order weighted by p:
 *   u [T][width] act dtype = sum_j p_(t,j) row(t, j)   (= z, resp. x, up to rounding: sum p = 1).
 *   send_buf, recv_buf  device buffers of at least T*k*width*elem bytes each (buf_bytes)
 *   cells     [ranks][ranks] int32 device, out (or NULL): rows sent from rank src to rank dst
 *             (row-major by src); the payload of the all-to-all is sum over src != dst
 *   events    6 cudaEvent_t (or NULL), recorded on `stream`: start, routed (and W_down done),
 *             packed, exchanged, returned, combined.
 * Errors: INVALID_ARG (sizes, alignment, ranks), CUDA. */
lmoe_status latentmoe_ep_emulate(lmoe_handle *h, const void *x, int32_t T, const lmoe_weights *w,
                                 int32_t ranks, int32_t full_width, void *send_buf, void *recv_buf,
                                 size_t buf_bytes, void *u, int32_t *cells, void *const *events,
                                 void *stream);

/* Test hook: device address and byte size of an intermediate of the last call inside the
 * handle's workspace, by name: "logits" [T][E] fp32, "z" [T][l], "gathered" [T*k][l] (the
 * expert-contiguous rows; after a full forward it holds the p-scaled expert outputs), "act"
 * [T*k][h] (routed GLU activations), "act_cat" [T][N_s*h_s + l] (shared activations and
 * RMSNorm(u)), "p_row" [T*k] fp32, "refine_count" [2] int32 (tokens of the last routing whose
 * list was settled on exact keys, and among them the near ties: exact k-th/(k+1)-th key gap
 * below 1e-6).  Activations use the act dtype, except that "z", "gathered" and "act" are fp16
 * when routed_w is MXFP4 and the dequantizing kernels run; on the block-scaled path "gathered"
 * holds three-term MXFP4 records of z's rows (3*l/2 packed E2M1 bytes, then 3*l/32 E8M0 scales)
 * until the down projection overwrites it with fp16 rows, and "act" the records of the GLU
 * activations (3*h/2 + 3*h/32 bytes per row); T is the last call's T.
 * The pointers stay valid until latentmoe_destroy.  Unknown name or absent buffer:
 * LMOE_ERR_INVALID_ARG. */
lmoe_status latentmoe_debug_buffer(const lmoe_handle *h, const char *name, void **ptr, size_t *bytes);

/* Router and dispatch without any device allocation, for callers that must not allocate
 * (for example a plugin whose host framework owns all device memory and forbids allocation
 * while it executes, or a serving loop that plans every byte ahead).  The paper has no
 * counterpart to this entry point; it computes exactly what latentmoe_route computes.
 *
 * No handle: `cfg` supplies d, num_experts, top_k, act and router_w (other fields are
 * ignored).  Outputs are as for latentmoe_route, but all five must be non-NULL when T > 0.
 * Scratch lives in one fixed 16 MiB device array inside the library, held on every GPU that
 * loads the library until the process exits; a call needs
 *   256*ceil(T*E*4/256) + 2*256*ceil(ceil(T/256)*E*4/256) + 256*ceil((T*k/128+E+1)*16/256)
 *   + 256*ceil(T*4/256) + 512
 * bytes of it, plus 256*ceil(3*E*d*2/256) when act is BF16 and router_w is F32 (the three bf16
 * terms of W_r), plus 256 for a status word; with k=16 and a bf16 W_r, T up to 32,133 for E=128
 * and up to 4,631 for E=896; a larger need returns LMOE_ERR_INVALID_ARG before any launch.  The
 * first call on a device (T == 0 included) looks up the array's device address
 * (cudaGetSymbolAddress), which also loads the library's kernels and the array on that device:
 * make one such call, e.g. with T = 0, at start-up, before any stream capture.  A device reset
 * invalidates the looked-up address: use a new process after one.  Calls that overlap on the GPU
 * share the array and race: serialise them.  Returned errors: INVALID_ARG (bad field, pointer or
 * size), CUDA.  Errors the kernels detect (a bounded wait that ran out, an index out of range, a
 * router logit outside the error margin) are ORed into a status word inside the array and are
 * reported by latentmoe_route_noalloc_status(). */
lmoe_status latentmoe_route_noalloc(const lmoe_config *cfg, const void *x, int32_t T, const lmoe_weights *w,
                                    int32_t *topk_idx, float *topk_p, int32_t *expert_offsets,
                                    int32_t *tok_of_row, int32_t *row_of, void *stream);

/* Test hook: the three-term MXFP4 records the block-scaled expert GEMMs read, for `rows` rows of
 * K values (src [rows][K], src_dtype LMOE_BF16 or LMOE_F16; K % 512 == 0).  Row r of dst (rows x
 * (3*K/2 + 3*K/32) bytes) holds terms q_0, q_1, q_2 (K/2 bytes each, element 2i in the low nibble
 * of byte i), then their E8M0 scales (K/32 bytes each): per 32-element block, q_t rounds what the
 * earlier terms left to nearest on the E2M1 grid (ties to the even code) with the smallest
 * power-of-two scale that leaves no element above 6.  Asynchronous on `stream`; allocates nothing.
 * Errors: INVALID_ARG, CUDA. */
lmoe_status latentmoe_mx3_quantize(const void *src, int32_t src_dtype, int64_t rows, int32_t K, void *dst,
                                   void *stream);

/* Test hook: the MXFP8 records (LMOE_FLAG_MXFP8_ACT) of rows x K values, K % 512 == 0:
 * dst [rows][K + K/32] bytes = K E4M3 codes (element i in byte i), then K/32 scale bytes. */
lmoe_status latentmoe_mx8_quantize(const void *src, int32_t src_dtype, int64_t rows, int32_t K, void *dst,
                                   void *stream);

/* Measurement hook: the dense tensor-core rate of this GPU, in TFLOP/s, for the instruction shape
 * the expert GEMMs issue (tcgen05.mma.cta_group::2, M = N = 256 per CTA pair, back to back on
 * every SM pair from shared-memory operands, fp32 accumulation in TMEM): kind 0 = kind::f16 (bf16
 * operands, K = 16 per instruction), kind 1 = kind::mxf4 (E2M1 operands with E8M0 scales per 32,
 * K = 64).  Synchronises `stream`; takes a few milliseconds.  Errors: INVALID_ARG, CUDA, TIMEOUT. */
lmoe_status latentmoe_mma_peak(int32_t kind, double *tflops, void *stream);

/* For callers of latentmoe_route_noalloc: synchronise `stream`, then read and clear the status
 * word its kernels report into on the current device (shared by every no-allocation call on
 * that device since the last read), and return the first sticky error (TIMEOUT before
 * DEVICE_CHECK) or LMOE_OK.  Allocates nothing. */
lmoe_status latentmoe_route_noalloc_status(void *stream);

/* Static description of a status code. */
const char *latentmoe_status_string(lmoe_status s);

#ifdef __cplusplus
}
#endif
#endif /* LATENTMOE_H */
