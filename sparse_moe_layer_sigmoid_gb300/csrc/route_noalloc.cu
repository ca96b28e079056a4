// latentmoe_route_noalloc: the router and dispatch of latentmoe_route for callers that may
// not allocate device memory, with every scratch buffer inside one fixed file-scope array.
//
// Who needs it: code that runs where cudaMalloc/cudaFree (or any allocating library call) is
// not allowed or not wanted at run time, e.g. a plugin whose host framework owns all device
// memory and forbids allocation in its execute step, or a latency-critical serving loop that
// plans every byte up front.  Such a caller cannot create a handle (latentmoe_create allocates
// a workspace), so this entry point takes the configuration directly and needs only the
// caller's inputs and outputs.
//
// Scratch: kScratchBytes in `g_route_scratch`, present on every GPU that loads the library
// until the process exits.  All calls share it, so calls that overlap on the GPU (different
// streams, or different host threads without ordering) race and must be serialised by the
// caller.  Its first 256 bytes hold a status word: errors the kernels detect (a bounded wait
// that ran out, an out-of-range index, a router logit outside the error margin) are ORed into
// it and stay there until latentmoe_route_noalloc_status() reads and clears it (the array
// starts zeroed).  The refinement-list counters are reset (cudaMemsetAsync, no allocation) at
// the start of every call; every other scratch word a kernel reads is written earlier in the
// same call.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "latentmoe.h"

namespace {

constexpr size_t kScratchBytes = (size_t)16 << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_route_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

struct ScratchLayout {
  size_t status, logits, chunk_counts, chunk_base, tiles, num_tiles, refine_list, refine_count, wr_split, total;
};

ScratchLayout scratch_layout(int T, int E, int k, size_t wr_split_bytes) {
  const size_t nchunks = ((size_t)T + lmoe::kDispatchChunk - 1) / lmoe::kDispatchChunk;
  const size_t max_tiles = (size_t)T * k / lmoe::kTileM + E + 1;
  ScratchLayout s;
  s.status = 0;  // sticky status word (uint32)
  s.logits = 256;
  s.chunk_counts = s.logits + round256((size_t)T * E * sizeof(float));
  s.chunk_base = s.chunk_counts + round256(nchunks * E * sizeof(int32_t));
  s.tiles = s.chunk_base + round256(nchunks * E * sizeof(int32_t));
  s.num_tiles = s.tiles + round256(max_tiles * sizeof(int4));
  s.refine_list = s.num_tiles + 256;
  s.refine_count = s.refine_list + round256((size_t)T * sizeof(int32_t));
  s.wr_split = s.refine_count + 256;
  s.total = s.wr_split + round256(wr_split_bytes);
  return s;
}

// Device address of the scratch array on the current device, looked up once per device.
lmoe_status scratch_for_current_device(uint8_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LMOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LMOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess || p == nullptr) return LMOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_scratch_addr[dev]);
  return LMOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" lmoe_status latentmoe_route_noalloc(const lmoe_config* cfg, const void* x, int32_t T,
                                               const lmoe_weights* w, int32_t* topk_idx, float* topk_p,
                                               int32_t* expert_offsets, int32_t* tok_of_row, int32_t* row_of,
                                               void* stream) {
  if (!cfg || !w) return LMOE_ERR_INVALID_ARG;
  const int E = cfg->num_experts, k = cfg->top_k, d = cfg->d;
  if (E < 1 || E > 1024 || k < 1 || k > E || k > 32 || d <= 0 || d % 16) return LMOE_ERR_INVALID_ARG;
  if (cfg->act == LMOE_BF16 && (d % 64 || E % 4)) return LMOE_ERR_INVALID_ARG;  // tensor-core router tiles
  if ((cfg->act != LMOE_F32 && cfg->act != LMOE_BF16) || (cfg->router_w != LMOE_F32 && cfg->router_w != LMOE_BF16))
    return LMOE_ERR_INVALID_ARG;
  if (T < 0) return LMOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !aligned16(x) || !w->w_router || !aligned16(w->w_router) || !topk_idx || !topk_p ||
                !expert_offsets || !tok_of_row || !row_of))
    return LMOE_ERR_INVALID_ARG;
  if (w->router_bias && !aligned16(w->router_bias)) return LMOE_ERR_INVALID_ARG;
  // bf16 activations with an fp32 W_r contract three bf16 terms of W_r (3*E*d*2 bytes)
  const size_t wr_split_bytes = (cfg->act == LMOE_BF16 && cfg->router_w == LMOE_F32) ? (size_t)3 * E * d * 2 : 0;
  const ScratchLayout L = scratch_layout(T, E, k, wr_split_bytes);
  if (L.total > kScratchBytes) return LMOE_ERR_INVALID_ARG;  // beyond the fixed scratch

  // the set-up of this device (the array's address) happens here even for T == 0, so that a
  // T == 0 call made at start-up does it ahead of any stream capture
  uint8_t* base = nullptr;
  lmoe_status st = scratch_for_current_device(&base);
  if (st != LMOE_OK || T == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* status = reinterpret_cast<uint32_t*>(base + L.status);
  float* logits = reinterpret_cast<float*>(base + L.logits);
  lmoe::DispatchBuffers db;
  db.chunk_counts = reinterpret_cast<int32_t*>(base + L.chunk_counts);
  db.chunk_base = reinterpret_cast<int32_t*>(base + L.chunk_base);
  db.offsets = expert_offsets;
  db.tiles = reinterpret_cast<int4*>(base + L.tiles);
  db.num_tiles = reinterpret_cast<int32_t*>(base + L.num_tiles);
  db.tiles_s = nullptr;  // the 16-row list serves only the expert GEMMs
  db.num_tiles_s = nullptr;
  db.tiles_p = nullptr;
  db.num_tiles_p = nullptr;
  db.tiles_m = nullptr;
  db.num_tiles_m = nullptr;
  db.tok_of_row = tok_of_row;
  db.row_of = row_of;
  db.p_row = nullptr;
  int dev = 0, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return LMOE_ERR_CUDA;
  if (lmoe::launch_router(x, cfg->act, w->w_router, cfg->router_w, logits,
                          wr_split_bytes ? base + L.wr_split : nullptr, T, E, d, status, 4000000000ull, num_sms,
                          nullptr, s) != cudaSuccess)
    return LMOE_ERR_CUDA;
  const lmoe::RouterSrc rs{x, cfg->act, w->w_router, cfg->router_w, d, lmoe::kRouterLogitMargin};
  if (lmoe::launch_topk(logits, w->router_bias, rs, T, E, k, topk_idx, topk_p,
                        reinterpret_cast<int32_t*>(base + L.refine_list),
                        reinterpret_cast<int32_t*>(base + L.refine_count), status, num_sms, s) != cudaSuccess)
    return LMOE_ERR_CUDA;
  if (lmoe::launch_dispatch(topk_idx, topk_p, T, E, k, db, status, nullptr, s) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

// Reads and clears the status word the no-allocation route's kernels report into, after
// `stream` has finished; allocates nothing either.
extern "C" lmoe_status latentmoe_route_noalloc_status(void* stream) {
  uint8_t* base = nullptr;
  lmoe_status st = scratch_for_current_device(&base);
  if (st != LMOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, base, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(base, 0, sizeof(word), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return LMOE_ERR_CUDA;
  if (word & lmoe::kStatusTimeout) return LMOE_ERR_TIMEOUT;
  if (word & lmoe::kStatusDeviceCheck) return LMOE_ERR_DEVICE_CHECK;
  return LMOE_OK;
}
