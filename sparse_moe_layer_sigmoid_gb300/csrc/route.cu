// Router, top-k selection and expert dispatch (page "Lesson 6 - LatentMoE",
// kimi-k3-course.pages.dev, section "show me the actual equation", eq. 13; and
// "Kimi K3 architectural innovations", manishklach.github.io, section "A router decision is
// also a scheduling decision": selections become expert batches).
//
// Everything here is integer or per-token fp32 work on CUDA cores; the router GEMM itself runs on
// the tensor cores (bf16 activations) or the fp32 CUDA-core GEMM of simt.cu.  All results are
// deterministic: no reduction depends on thread scheduling (counts use atomicOr on bit masks,
// which commute exactly).
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace lmoe {
namespace {

__device__ __forceinline__ uint32_t orderable(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float from_orderable(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// Double-float accumulator (hi + lo, |lo| <= ulp(hi)/2): products of bf16/fp32 operands are
// split exactly with an FMA (TwoProd) and added with Knuth's TwoSum, so the sum of d products
// keeps about 44 significant bits: far below the spacing of the decisions it settles.
struct DF {
  float hi, lo;
};
__device__ __forceinline__ void df_add_prod(DF& a, float x, float w) {
  const float p = x * w;
  const float pe = fmaf(x, w, -p);  // exact: p + pe == x * w
  const float s = a.hi + p;
  const float bb = s - a.hi;
  const float se = (a.hi - (s - bb)) + (p - bb);  // exact: s + se == a.hi + p
  a.hi = s;
  a.lo += se + pe;
}
__device__ __forceinline__ DF df_add(DF a, DF b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  const float se = (a.hi - (s - bb)) + (b.hi - bb);
  DF r;
  r.lo = se + a.lo + b.lo;
  r.hi = s + r.lo;  // renormalise
  r.lo = r.lo - (r.hi - s);
  return r;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&f)[8]) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float (&f)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

constexpr int kCandBatch = 8;  // boundary candidates evaluated per pass over d

// Partial dot products x . W_r[e_m] in double-float for up to kCandBatch candidates, one warp
// over the 256-element blocks part, part + nparts, ... of d: each step loads 8 elements of x once
// and 8 elements of every candidate row (independent loads in flight).  Every lane receives the
// warp's partial sums.
template <typename TX, typename TW>
__device__ void dots_df_part(const TX* x, const TW* w, int64_t d, const int (&ce)[kCandBatch], int nc, int part,
                             int nparts, int lane, DF (&out)[kCandBatch]) {
  DF acc[kCandBatch];
#pragma unroll
  for (int m = 0; m < kCandBatch; ++m) acc[m] = DF{0.f, 0.f};
#pragma unroll 2
  for (int64_t c = (int64_t)part * 256 + lane * 8; c < d; c += (int64_t)nparts * 256) {  // d % 16 == 0
    float xf[8];
    load8(x + c, xf);
#pragma unroll
    for (int m = 0; m < kCandBatch; ++m) {
      if (m < nc) {
        float wf[8];
        load8(w + ce[m] * d + c, wf);
#pragma unroll
        for (int i = 0; i < 8; ++i) df_add_prod(acc[m], xf[i], wf[i]);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < kCandBatch; ++m) {
    DF a = acc[m];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      DF o;
      o.hi = __shfl_xor_sync(0xffffffffu, a.hi, off);
      o.lo = __shfl_xor_sync(0xffffffffu, a.lo, off);
      a = df_add(a, o);
    }
    out[m] = a;
  }
}

// Partial logits of the candidate experts ce[0..nc) for token t (see dots_df_part).
__device__ void exact_logit_parts(const RouterSrc& r, int t, const int (&ce)[kCandBatch], int nc, int part,
                                  int nparts, int lane, DF (&out)[kCandBatch]) {
  const int64_t xo = (int64_t)t * r.d;
  if (r.x_dtype == kBF16 && r.w_dtype == kBF16)
    dots_df_part(static_cast<const __nv_bfloat16*>(r.x) + xo, static_cast<const __nv_bfloat16*>(r.w), r.d, ce, nc,
                 part, nparts, lane, out);
  else if (r.x_dtype == kBF16)
    dots_df_part(static_cast<const __nv_bfloat16*>(r.x) + xo, static_cast<const float*>(r.w), r.d, ce, nc, part,
                 nparts, lane, out);
  else if (r.w_dtype == kBF16)
    dots_df_part(static_cast<const float*>(r.x) + xo, static_cast<const __nv_bfloat16*>(r.w), r.d, ce, nc, part,
                 nparts, lane, out);
  else
    dots_df_part(static_cast<const float*>(r.x) + xo, static_cast<const float*>(r.w), r.d, ce, nc, part, nparts,
                 lane, out);
}

// One warp per token.  Lane l holds experts l, l + 32, ... (NPL slots).  The selection finds the
// k-th largest key by bisection over the order-preserving 32-bit image of the fp32 keys (a warp
// count per probe), keeps every key above it and, among keys equal to it, the lowest indices
// (eq. 13's tie rule), then sorts the k winners by (key descending, index ascending) with a
// 32-lane bitonic network; after the pass, lane j < k holds the rank-j winner.  `sk` / `ss` are
// 32-entry scratch arrays private to the warp.
//
// The logits come from a GEMM whose error is bounded by `src.margin`, so a key is known to
// within eta (token_eta: margin times the largest sigmoid' among the token's contenders, + fp32
// rounding), and two keys further apart than 2*eta are ordered correctly.  A token is settled exactly (second pass) when the order of its list is not certain:
// when the k-th and (k+1)-th keys are closer than 2*eta (the selected set itself), or when two
// neighbouring ranks are (the rank order).  There every expert whose key lies in the band around
// an uncertain boundary, and every selected expert with a neighbour closer than 2*eta, has its
// logit recomputed to ~44 bits and its key evaluated in fp64; the k winners are then the
// contenders (the selected experts and the band) in descending order of their keys, exact where
// recomputed, else the fp32 key (which is at least 2*eta away from every other contender's).
template <int NPL>
struct TopkState {
  float kf[NPL], sv[NPL];  // keys and scores of this lane's experts
  int my_e;                // lane j < k: expert of rank j
  float my_s, my_kf;       // its score and key
  float a_k, a_k1;         // k-th and (k+1)-th keys
};

// Bound on |key - exact key| for any expert: a logit error of at most `margin` moves s = sigmoid(l)
// by at most margin * max sigmoid' = margin / 4 (+ fp32 rounding of s and s + b).
__device__ __forceinline__ float key_eta(const RouterSrc& src) { return 0.25f * src.margin + 1e-6f; }

// The key uncertainty of one token's contenders.  Expert e's key moves by at most margin *
// max sigmoid'(l) over [l_e - margin, l_e + margin] <= margin * (s_e (1 - s_e) + 1e-4) (sigmoid''
// is at most 0.1 in size), + 1e-6 for rounding.  Every expert whose key could reach the boundary
// lies within the widest band (2 key_eta around the k-th and (k+1)-th keys), so the largest bound
// over that band and the selected experts bounds every comparison the selection and the rank
// order make; near the top of 896 experts sigmoid' is ~0.08, a third of the worst case.
template <int NPL>
__device__ __forceinline__ float token_eta(const float (&kf)[NPL], const float (&sv)[NPL], float a_k1,
                                           const RouterSrc& src) {
  const float lo = a_k1 - 2.0f * key_eta(src);
  float d = 0.0f;
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (kf[i] >= lo) d = fmaxf(d, sv[i] * (1.0f - sv[i]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) d = fmaxf(d, __shfl_xor_sync(0xffffffffu, d, off));
  return src.margin * (d + 1e-4f) + 1e-6f;
}

template <int NPL>
__device__ __forceinline__ int count_at_least(const uint32_t (&ko)[NPL], uint32_t v) {
  int c = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) c += ko[i] >= v ? 1 : 0;
  return (int)__reduce_add_sync(0xffffffffu, (unsigned)c);
}

// Score s = sigmoid(logit) and key s + b of expert e of token t (fp32, the same arithmetic
// wherever a key is needed).
__device__ __forceinline__ void expert_key(const float* __restrict__ logits, const float* __restrict__ bias, int t,
                                           int E, int e, float& s, float& key) {
  s = 1.0f / (1.0f + expf(-logits[(size_t)t * E + e]));
  key = bias ? s + bias[e] : s;
}

// Keys and scores of this lane's experts (-inf / 0 past E).  All of the lane's logits and biases
// are loaded before any is used, so the loads are in flight together (one memory latency per
// token instead of one per expert slot).
template <int NPL>
__device__ __forceinline__ void topk_keys(const float* __restrict__ logits, const float* __restrict__ bias, int t,
                                          int E, int lane, TopkState<NPL>& st) {
  const float* row = logits + (size_t)t * E;
  float lg[NPL], bs[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    lg[i] = e < E ? __ldg(row + e) : 0.f;
    bs[i] = bias && e < E ? __ldg(bias + e) : 0.f;
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const bool in = lane + 32 * i < E;
    const float s = 1.0f / (1.0f + expf(-lg[i]));  // the arithmetic of expert_key
    st.sv[i] = in ? s : 0.f;
    st.kf[i] = in ? (bias ? s + bs[i] : s) : -INFINITY;
  }
}

template <int NPL>
__device__ __forceinline__ void topk_pass(const float* __restrict__ logits, const float* __restrict__ bias, int t,
                                          int E, int k, int lane, TopkState<NPL>& st, uint64_t* sk, float* ss,
                                          bool keys_ready = false) {
  if (!keys_ready) topk_keys<NPL>(logits, bias, t, E, lane, st);  // else st.kf / st.sv are filled
  uint32_t ko[NPL];  // orderable keys; 0 (below every key) for slots past E
  uint32_t kmax = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    ko[i] = lane + 32 * i < E ? orderable(st.kf[i]) : 0u;
    kmax = ko[i] > kmax ? ko[i] : kmax;
  }
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  // K = the k-th largest key: the largest v with at least k keys >= v (every key is >= 1)
  uint32_t lo = 1, hi = kmax;
  while (lo < hi) {
    const uint32_t mid = lo + ((hi - lo + 1u) >> 1);
    if (count_at_least<NPL>(ko, mid) >= k)
      lo = mid;
    else
      hi = mid - 1u;
  }
  const uint32_t K = lo;
  const int n_gt = K == 0xFFFFFFFFu ? 0 : count_at_least<NPL>(ko, K + 1u);
  // keys equal to K: the lowest indices (slot-major, then lane) fill the k - n_gt open ranks
  int need = k - n_gt;
  bool sel[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const bool eq = ko[i] == K;
    const uint32_t m = __ballot_sync(0xffffffffu, eq);
    const int before = __popc(m & ((1u << lane) - 1u));
    sel[i] = ko[i] > K || (eq && before < need);
    const int n_eq = __popc(m);
    need -= need < n_eq ? need : n_eq;
  }
  st.a_k = from_orderable(K);
  st.a_k1 = -INFINITY;
  if (k < E) {
    uint32_t below = 0;  // largest key not selected
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (!sel[i] && ko[i] > below) below = ko[i];
    st.a_k1 = from_orderable(__reduce_max_sync(0xffffffffu, below));
  }
  // compact the k winners into the scratch: key, then (1023 - expert) << 5, then the slot of its score
  int c = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) c += sel[i] ? 1 : 0;
  int base = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, base, off);
    if (lane >= off) base += o;
  }
  base -= c;
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (sel[i]) {
      const uint32_t e = (uint32_t)(lane + 32 * i);
      sk[base] = ((uint64_t)ko[i] << 32) | ((1023u - e) << 5) | (uint32_t)base;
      ss[base] = st.sv[i];
      ++base;
    }
  __syncwarp();
  uint64_t v = lane < k ? sk[lane] : 0ull;
  // bitonic sort, descending over the 32 lanes
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
    }
  st.my_e = 0;
  st.my_s = 0.f;
  st.my_kf = 0.f;
  if (lane < k) {
    st.my_e = 1023 - (int)((v >> 5) & 1023u);
    st.my_kf = from_orderable((uint32_t)(v >> 32));
    st.my_s = ss[v & 31u];
  }
  __syncwarp();  // the scratch is rewritten by the warp's next token
}

// Bitonic sort of 64 (key, aux) entries held two per lane (entry j = 2 lane + h in key[h],
// aux[h]) into descending key order, equal keys by ascending aux; afterwards entry j is rank j.
__device__ __forceinline__ bool sorts_before(uint64_t ka, uint32_t aa, uint64_t kb, uint32_t ab) {
  return ka > kb || (ka == kb && aa < ab);
}
__device__ __forceinline__ void sort64_desc(uint64_t (&key)[2], uint32_t (&aux)[2], int lane) {
#pragma unroll
  for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride == 1) {  // entries 2 lane and 2 lane + 1: in the lane
        const bool desc = ((2 * lane) & size) == 0;
        const bool swap = desc ? sorts_before(key[1], aux[1], key[0], aux[0])
                               : sorts_before(key[0], aux[0], key[1], aux[1]);
        if (swap) {
          const uint64_t tk = key[0];
          key[0] = key[1];
          key[1] = tk;
          const uint32_t ta = aux[0];
          aux[0] = aux[1];
          aux[1] = ta;
        }
      } else {  // partner entry j ^ stride sits in lane ^ (stride / 2), same h
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = 2 * lane + h;
          const uint64_t ok = __shfl_xor_sync(0xffffffffu, key[h], stride >> 1);
          const uint32_t oa = __shfl_xor_sync(0xffffffffu, aux[h], stride >> 1);
          const bool keep_first = ((j & stride) == 0) == ((j & size) == 0);
          const bool other_first = sorts_before(ok, oa, key[h], aux[h]);
          if (keep_first ? other_first : !other_first) {
            key[h] = ok;
            aux[h] = oa;
          }
        }
      }
    }
  }
}

// Entry r (0 <= r < 64) of a sort64_desc result, in every lane.
__device__ __forceinline__ uint64_t entry_key(const uint64_t (&key)[2], int r) {
  const uint64_t a = __shfl_sync(0xffffffffu, key[0], r >> 1), b = __shfl_sync(0xffffffffu, key[1], r >> 1);
  return (r & 1) ? b : a;
}
__device__ __forceinline__ uint32_t entry_aux(const uint32_t (&aux)[2], int r) {
  const uint32_t a = __shfl_sync(0xffffffffu, aux[0], r >> 1), b = __shfl_sync(0xffffffffu, aux[1], r >> 1);
  return (r & 1) ? b : a;
}

// Pass 1 by candidates: the k-th largest of the 32 lane maxima bounds the k-th largest key from
// below (those k lanes hold k keys at least that large), so only keys at or above it can be
// selected.  When at most 64 keys qualify (k <= 32) they are compacted into the warp's scratch
// and sorted by (key, lower index first) in one 64-entry bitonic network, which gives the
// selection, its rank order and the (k+1)-th key at once: about 1.5 K warp instructions and a
// few dozen dependent steps instead of a 32-step bisection.  Returns false (state untouched
// but for the keys) when more than 64 keys qualify: topk_pass then selects by bisection.
// `sk` / `ss`: 64-entry scratch private to the warp.
template <int NPL>
__device__ __forceinline__ bool topk_pass_sorted(const float* __restrict__ logits, const float* __restrict__ bias,
                                                 int t, int E, int k, int lane, TopkState<NPL>& st, uint64_t* sk,
                                                 float* ss) {
  topk_keys<NPL>(logits, bias, t, E, lane, st);
  if (k > 32) return false;
  uint32_t ko[NPL];
  uint32_t lm = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    ko[i] = lane + 32 * i < E ? orderable(st.kf[i]) : 0u;
    lm = ko[i] > lm ? ko[i] : lm;
  }
  // k-th largest lane maximum: bitonic sort of the 32 maxima, descending
  uint32_t v = lm;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
    }
  const uint32_t lb = __shfl_sync(0xffffffffu, v, k - 1);
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) cnt += __popc(__ballot_sync(0xffffffffu, ko[i] >= lb && ko[i] != 0u));
  if (cnt > 64) return false;
  // candidates into the scratch: key, then 0xFFFF - expert (lower index first), then the position
  const uint32_t lt = (1u << lane) - 1u;
  int base = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const bool c = ko[i] >= lb && ko[i] != 0u;
    const uint32_t m = __ballot_sync(0xffffffffu, c);
    if (c) {
      const int pos = base + __popc(m & lt);
      sk[pos] = ((uint64_t)ko[i] << 32) | ((uint64_t)(0xFFFFu - (uint32_t)(lane + 32 * i)) << 16) | (uint64_t)pos;
      ss[pos] = st.sv[i];
    }
    base += __popc(m);
  }
  __syncwarp();
  uint64_t key[2];
  uint32_t aux[2] = {0u, 0u};
  key[0] = 2 * lane < cnt ? sk[2 * lane] : 0ull;
  key[1] = 2 * lane + 1 < cnt ? sk[2 * lane + 1] : 0ull;
  sort64_desc(key, aux, lane);
  const uint64_t mine = entry_key(key, lane < k ? lane : 0);
  st.my_e = 0;
  st.my_s = 0.f;
  st.my_kf = 0.f;
  if (lane < k) {
    st.my_e = (int)(0xFFFFu - (uint32_t)((mine >> 16) & 0xFFFFu));
    st.my_kf = from_orderable((uint32_t)(mine >> 32));
    st.my_s = ss[mine & 0xFFFFu];
  }
  st.a_k = from_orderable((uint32_t)(entry_key(key, k - 1) >> 32));
  st.a_k1 = -INFINITY;
  if (k < E) {
    if (cnt > k) {
      st.a_k1 = from_orderable((uint32_t)(entry_key(key, k) >> 32));
    } else {  // exactly k candidates: the (k+1)-th key is the largest below the bound
      uint32_t below = 0;
#pragma unroll
      for (int i = 0; i < NPL; ++i)
        if (ko[i] < lb && ko[i] > below) below = ko[i];
      st.a_k1 = from_orderable(__reduce_max_sync(0xffffffffu, below));
    }
  }
  __syncwarp();  // the scratch is rewritten by the warp's next token
  return true;
}

// p = s / sum(s over the selected set), summed in rank order; lanes j < k store rank j.
__device__ __forceinline__ void topk_write(int t, int k, int my_e, float my_s, int32_t* __restrict__ idx,
                                           float* __restrict__ p, int lane) {
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, my_s, j);  // rank order
  if (lane < k) {
    idx[(size_t)t * k + lane] = my_e;
    p[(size_t)t * k + lane] = my_s / sum;
  }
}

// Pass 1: one warp per token; tokens whose boundary is uncertain go to the refinement list.
template <int NPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                                                   RouterSrc src, int T, int E, int k, int32_t* __restrict__ idx,
                                                   float* __restrict__ p, int32_t* __restrict__ refine_list,
                                                   int32_t* __restrict__ refine_count) {
  __shared__ uint64_t s_sk[8][64];
  __shared__ float s_ss[8][64];
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (t >= T) return;
  TopkState<NPL> st;
  if (!topk_pass_sorted<NPL>(logits, bias, t, E, k, lane, st, s_sk[warp], s_ss[warp]))
    topk_pass<NPL>(logits, bias, t, E, k, lane, st, s_sk[warp], s_ss[warp]);
  const float eta2 = 2.0f * token_eta<NPL>(st.kf, st.sv, st.a_k1, src);
  const float next = __shfl_down_sync(0xffffffffu, st.my_kf, 1);
  const bool close = lane + 1 < k && st.my_kf - next < eta2;  // rank order of lanes j, j+1 uncertain
  if ((k < E && st.a_k - st.a_k1 < eta2) || __any_sync(0xffffffffu, close)) {
    // the ranked list stays in idx for the refinement, which rewrites idx and p
    if (lane < k) idx[(size_t)t * k + lane] = st.my_e;
    if (lane == 0) refine_list[atomicAdd(refine_count, 1)] = t;  // list order is irrelevant: tokens are independent
    return;
  }
  topk_write(t, k, st.my_e, st.my_s, idx, p, lane);
}

constexpr int kRefineWarps = 4;  // warps of a refinement CTA
constexpr int kMaxCont = 64;     // contenders of one token: its selected experts and the band

// Shared memory of one refinement group (a warp, or the whole CTA): the token's contenders.
struct RefineSmem {
  int* ce;          // [kMaxCont] contender experts
  uint64_t* key;    // [kMaxCont] sort keys (order-preserving images of the fp64 keys)
  float* s;         // [kMaxCont] scores
  int* exa;         // [kMaxCont] 1: key and score recomputed exactly
  int* cand;        // [kMaxCont] positions (in ce) of the contenders to recompute
  float2* part;     // [G][kMaxCont] partial logits (double-float) of the G warps
  int* n;           // [2]: contenders, contenders to recompute
};

template <int G>
__device__ __forceinline__ void group_sync() {
  if (G == 1)
    __syncwarp();
  else
    __syncthreads();
}

// fp64 key -> unsigned integer of the same order (0 stays below every key), and back.
__device__ __forceinline__ uint64_t orderable64(double d) {
  const uint64_t u = (uint64_t)__double_as_longlong(d);
  return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}
__device__ __forceinline__ double from_orderable64(uint64_t u) {
  return __longlong_as_double((long long)((u >> 63) ? (u & 0x7FFFFFFFFFFFFFFFull) : ~u));
}

// Gap between the k-th and (k+1)-th keys below which a token is a near tie (its selected set may
// differ from the fp64 evaluation's; such tokens are counted).
constexpr double kNearTieGap = 1e-6;

// Settle the list of token t exactly: G warps (gw = 0..G-1) cooperate.  Warp 0 lists the
// token's contenders in shared memory (build_contenders): the selected experts and, when the
// boundary is uncertain, the band of experts that may cross it; those whose order is uncertain
// (the band; selected experts with a neighbouring rank closer than the key uncertainty) are
// recomputed.  The G warps compute their logits to ~44 bits, warp gw over the 256-element blocks
// gw, gw + G, ... of d; warp 0 sums the G partials in a fixed order, takes fp64 keys, checks each
// recomputed logit against the GEMM's (an error above half the margin is reported) and ranks the
// contenders by key, exact where recomputed (refine_finish).  A token whose exact k-th and
// (k+1)-th keys differ by less than kNearTieGap is counted in *near_ties.  More than kMaxCont
// contenders (dozens of experts within the key uncertainty of the boundary) is reported as a
// device check and ranks the first kMaxCont.

// Warp 0: the contender list of a token from its keys (st.kf, st.sv), its ranked list (st.my_e /
// my_kf on lanes < k), the k-th / (k+1)-th keys and 2 eta.
template <int NPL>
__device__ __forceinline__ void build_contenders(const TopkState<NPL>& st, float eta2, int E, int k, int lane,
                                                 const RefineSmem& sm, uint32_t* status) {
  const uint32_t lt_mask = (1u << lane) - 1u;
  const bool uncertain = k < E && st.a_k - st.a_k1 < eta2;
  // ranks whose order against a neighbouring rank (or, for the last, against the experts below
  // an uncertain boundary) is not certain
  const float prev = __shfl_up_sync(0xffffffffu, st.my_kf, 1);
  const float next = __shfl_down_sync(0xffffffffu, st.my_kf, 1);
  const int close = lane < k && ((lane > 0 && prev - st.my_kf < eta2) || (lane + 1 < k && st.my_kf - next < eta2) ||
                                 (lane == k - 1 && uncertain));
  uint32_t sel = 0, pend = 0;  // bit i: expert lane + 32 i is selected / awaits recomputation
  for (int j = 0; j < k; ++j) {
    const int e = __shfl_sync(0xffffffffu, st.my_e, j);
    const int c = __shfl_sync(0xffffffffu, close, j);
    if ((e & 31) == lane) {
      sel |= 1u << (e >> 5);
      if (c) pend |= 1u << (e >> 5);
    }
  }
  if (uncertain) {  // the band: every expert that may cross the boundary
    const float hi = st.a_k + eta2, lo = st.a_k1 - eta2;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && st.kf[i] >= lo && st.kf[i] <= hi) pend |= 1u << i;
    }
  }
  // contenders into shared memory (slot-major, then lane: a fixed order)
  int cnt = 0, nrc = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const bool c = ((sel | pend) >> i) & 1u;
    const uint32_t m = __ballot_sync(0xffffffffu, c);
    const int at = cnt + __popc(m & lt_mask);
    const bool in = c && at < kMaxCont;
    const bool r = in && ((pend >> i) & 1u);
    const uint32_t mr = __ballot_sync(0xffffffffu, r);
    if (in) {
      sm.ce[at] = lane + 32 * i;
      sm.key[at] = orderable64((double)st.kf[i]);
      sm.s[at] = st.sv[i];
      sm.exa[at] = 0;
      if (r) sm.cand[nrc + __popc(mr & lt_mask)] = at;
    }
    cnt += __popc(m);
    nrc += __popc(mr);
  }
  if (cnt > kMaxCont) {  // the first kMaxCont are ranked; the result is not exact
    if (lane == 0) report(status, kStatusDeviceCheck);
    cnt = kMaxCont;
  }
  if (lane == 0) {
    sm.n[0] = cnt;
    sm.n[1] = nrc;
  }
}

// 16-byte asynchronous copies of `bytes` (a multiple of 16) from global to shared memory by the
// `n` threads of the group, thread `i` taking chunks i, i + n, ...
__device__ __forceinline__ void cp_async_bytes(uint8_t* dst, const uint8_t* src, int64_t bytes, int i, int n) {
#pragma unroll 4
  for (int64_t o = (int64_t)i * 16; o < bytes; o += (int64_t)n * 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ptx::smem_addr(dst + o)),
                 "l"(__cvta_generic_to_global(src + o))
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// This thread's part of x . w over staged rows: elements i*8 .. i*8+7, + 8n, + 16n, ... in
// double-float (the arithmetic of dots_df_part).
template <typename TX, typename TW>
__device__ __forceinline__ DF dot_staged(const uint8_t* sx, const uint8_t* sw, int d, int i, int n) {
  const TX* x = reinterpret_cast<const TX*>(sx);
  const TW* w = reinterpret_cast<const TW*>(sw);
  DF a{0.f, 0.f};
#pragma unroll 1
  for (int c = i * 8; c < d; c += n * 8) {
    float xf[8], wf[8];
    load8(x + c, xf);
    load8(w + c, wf);
#pragma unroll
    for (int j = 0; j < 8; ++j) df_add_prod(a, xf[j], wf[j]);
  }
  return a;
}

// Shared-memory staging of the exact logits (short-batch selection): x's row and up to
// `rows` router rows per batch, `bytes_x` / `bytes_w` each.
struct RefineStage {
  uint8_t* mem;  // nullptr: the logits are recomputed from global memory (dots_df_part)
  int rows;
};

// All G warps: recompute the listed logits, then warp 0 ranks the contenders and writes the list.
// `lrow`: the token's logits from the router GEMM (global or shared memory).  With a stage (G warps = the whole CTA) the CTA copies x's row and a batch of router rows into
// shared memory in one round of asynchronous copies and every thread sums its elements of each
// row; warp gw's partial covers its lanes' elements.  Without, warp gw sums the 256-element blocks
// gw, gw + G, ... of d straight from global memory.
template <int NPL, int G>
__device__ __forceinline__ void refine_finish(const float* lrow, const float* __restrict__ bias,
                                              const RouterSrc& src, int t, int E, int k, int32_t* __restrict__ idx,
                                              float* __restrict__ p, int gw, int lane, const RefineSmem& sm,
                                              uint32_t* status, int32_t* near_ties, RefineStage stage = {nullptr, 0}) {
  group_sync<G>();
  const int n_cont = sm.n[0], n_rc = sm.n[1];
  if (stage.mem) {
    const int tid = gw * 32 + lane, nthr = 32 * G;
    const int64_t bx = (int64_t)src.d * (src.x_dtype == kBF16 ? 2 : 4);
    const int64_t bw = (int64_t)src.d * (src.w_dtype == kBF16 ? 2 : 4);
    uint8_t* sx = stage.mem;
    uint8_t* sw = stage.mem + bx;
#pragma unroll 1
    for (int b0 = 0; b0 < n_rc; b0 += stage.rows) {
      const int nc = n_rc - b0 < stage.rows ? n_rc - b0 : stage.rows;
      if (b0 == 0) cp_async_bytes(sx, static_cast<const uint8_t*>(src.x) + (int64_t)t * bx, bx, tid, nthr);
#pragma unroll 1
      for (int m = 0; m < nc; ++m)
        cp_async_bytes(sw + m * bw, static_cast<const uint8_t*>(src.w) + (int64_t)sm.ce[sm.cand[b0 + m]] * bw, bw,
                       tid, nthr);
      cp_async_wait_all();
      group_sync<G>();
#pragma unroll 1
      for (int m = 0; m < nc; ++m) {
        const uint8_t* wr = sw + m * bw;
        DF a;
        if (src.x_dtype == kBF16 && src.w_dtype == kBF16)
          a = dot_staged<__nv_bfloat16, __nv_bfloat16>(sx, wr, src.d, tid, nthr);
        else if (src.x_dtype == kBF16)
          a = dot_staged<__nv_bfloat16, float>(sx, wr, src.d, tid, nthr);
        else if (src.w_dtype == kBF16)
          a = dot_staged<float, __nv_bfloat16>(sx, wr, src.d, tid, nthr);
        else
          a = dot_staged<float, float>(sx, wr, src.d, tid, nthr);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          DF o;
          o.hi = __shfl_xor_sync(0xffffffffu, a.hi, off);
          o.lo = __shfl_xor_sync(0xffffffffu, a.lo, off);
          a = df_add(a, o);
        }
        if (lane == 0) sm.part[gw * kMaxCont + b0 + m] = make_float2(a.hi, a.lo);
      }
      group_sync<G>();  // the stage is rewritten by the next batch
    }
  }
  for (int b0 = 0; !stage.mem && b0 < n_rc; b0 += kCandBatch) {
    int ce[kCandBatch];
    const int nc = n_rc - b0 < kCandBatch ? n_rc - b0 : kCandBatch;
#pragma unroll
    for (int m = 0; m < kCandBatch; ++m) ce[m] = m < nc ? sm.ce[sm.cand[b0 + m]] : 0;
    DF part[kCandBatch];
    exact_logit_parts(src, t, ce, nc, gw, G, lane, part);
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < kCandBatch; ++m)
        if (m < nc) sm.part[gw * kMaxCont + b0 + m] = make_float2(part[m].hi, part[m].lo);
    }
  }
  group_sync<G>();
  if (gw == 0) {
    for (int c = lane; c < n_rc; c += 32) {
      DF a{sm.part[c].x, sm.part[c].y};
#pragma unroll
      for (int q = 1; q < G; ++q) a = df_add(a, DF{sm.part[q * kMaxCont + c].x, sm.part[q * kMaxCont + c].y});
      const int at = sm.cand[c];
      const int e = sm.ce[at];
      const double l64 = (double)a.hi + (double)a.lo;
      // the margin the selection relies on, checked on every logit recomputed here
      if (fabs((double)lrow[e] - l64) > 0.5 * (double)src.margin)
        report(status, kStatusDeviceCheck | kStatusRouterMargin);
      const double s64 = 1.0 / (1.0 + exp(-l64));
      sm.key[at] = orderable64(s64 + (bias ? (double)bias[e] : 0.0));
      sm.s[at] = (float)s64;
      sm.exa[at] = 1;
    }
    __syncwarp();
    // ranks 0..k-1 by (key descending, index ascending) over the contenders: one 64-entry sort
    // (aux = expert << 8 | position); entry k is the (k+1)-th contender, for the near-tie count
    uint64_t key[2];
    uint32_t aux[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = 2 * lane + h;
      key[h] = c < n_cont ? sm.key[c] : 0ull;  // 0: below every key
      aux[h] = c < n_cont ? ((uint32_t)sm.ce[c] << 8) | (uint32_t)c : 0xFFFFFFFFu;
    }
    sort64_desc(key, aux, lane);
    const uint32_t mine = entry_aux(aux, lane < k ? lane : 0);
    const int my_e = lane < k ? (int)(mine >> 8) : 0;
    const float my_s = lane < k ? sm.s[mine & 0xFFu] : 0.f;
    if (k < n_cont) {
      const uint64_t key_k = entry_key(key, k - 1), key_k1 = entry_key(key, k);
      const uint32_t pos_k = entry_aux(aux, k - 1) & 0xFFu, pos_k1 = entry_aux(aux, k) & 0xFFu;
      if (lane == 0 && sm.exa[pos_k] && sm.exa[pos_k1] &&
          from_orderable64(key_k) - from_orderable64(key_k1) < kNearTieGap)
        atomicAdd(near_ties, 1);
    }
    topk_write(t, k, my_e, my_s, idx, p, lane);
  }
  group_sync<G>();  // the contender list of this token is read by every warp before the next token's
}

// Pass 2 for one listed token: warp 0 reloads its keys and pass 1's ranked list from idx.
template <int NPL, int G>
__device__ __forceinline__ void refine_token(const float* __restrict__ logits, const float* __restrict__ bias,
                                             const RouterSrc& src, int t, int E, int k, int32_t* __restrict__ idx,
                                             float* __restrict__ p, int gw, int lane, const RefineSmem& sm,
                                             uint32_t* status, int32_t* near_ties) {
  if (gw == 0) {
    TopkState<NPL> st;
    topk_keys<NPL>(logits, bias, t, E, lane, st);
    st.my_e = lane < k ? idx[(size_t)t * k + lane] : 0;
    st.my_s = 0.f;
    st.my_kf = 0.f;
    if (lane < k) expert_key(logits, bias, t, E, st.my_e, st.my_s, st.my_kf);
    // k-th key: the last rank's; (k+1)-th: equal to it if more than k keys reach it, else the
    // largest key below it
    st.a_k = __shfl_sync(0xffffffffu, st.my_kf, k - 1);
    int n_ge = 0;
    float below = -INFINITY;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      n_ge += st.kf[i] >= st.a_k ? 1 : 0;
      if (st.kf[i] < st.a_k && st.kf[i] > below) below = st.kf[i];
    }
    n_ge = (int)__reduce_add_sync(0xffffffffu, (unsigned)n_ge);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) below = fmaxf(below, __shfl_xor_sync(0xffffffffu, below, off));
    st.a_k1 = n_ge > k ? st.a_k : below;
    build_contenders<NPL>(st, 2.0f * token_eta<NPL>(st.kf, st.sv, st.a_k1, src), E, k, lane, sm, status);
  }
  refine_finish<NPL, G>(logits + (size_t)t * E, bias, src, t, E, k, idx, p, gw, lane, sm, status, near_ties);
}

// Pass 2: the listed tokens.  With at least one token per warp each warp settles its own tokens;
// otherwise the 4 warps of a CTA split d for one token at a time (short lists: decode batches).
// refine_count[0] is the list length, refine_count[1] the near-tie counter.
template <int NPL>
__global__ void __launch_bounds__(32 * kRefineWarps, 4) topk_refine_kernel(
    const float* __restrict__ logits, const float* __restrict__ bias, RouterSrc src, int E, int k,
    int32_t* __restrict__ idx, float* __restrict__ p, const int32_t* __restrict__ refine_list,
    int32_t* __restrict__ refine_count, uint32_t* status) {
  __shared__ int s_ce[kRefineWarps][kMaxCont];
  __shared__ uint64_t s_key[kRefineWarps][kMaxCont];
  __shared__ float s_s[kRefineWarps][kMaxCont];
  __shared__ int s_exa[kRefineWarps][kMaxCont];
  __shared__ int s_cand[kRefineWarps][kMaxCont];
  __shared__ float2 s_part[kRefineWarps][kMaxCont];
  __shared__ int s_n[kRefineWarps][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = refine_count[0];
  int32_t* near_ties = refine_count + 1;
  if (n >= (int)gridDim.x * kRefineWarps) {  // at least one token per warp
    const RefineSmem sm{s_ce[warp], s_key[warp], s_s[warp], s_exa[warp], s_cand[warp], s_part[warp], s_n[warp]};
    for (int w = blockIdx.x * kRefineWarps + warp; w < n; w += gridDim.x * kRefineWarps)
      refine_token<NPL, 1>(logits, bias, src, refine_list[w], E, k, idx, p, 0, lane, sm, status, near_ties);
  } else {
    const RefineSmem sm{s_ce[0], s_key[0], s_s[0], s_exa[0], s_cand[0], &s_part[0][0], s_n[0]};
    for (int w = blockIdx.x; w < n; w += gridDim.x)
      refine_token<NPL, kRefineWarps>(logits, bias, src, refine_list[w], E, k, idx, p, warp, lane, sm, status,
                                      near_ties);
  }
}

// Both passes in one kernel for short batches (decode): one CTA of kSmallWarps warps per token.
// A token's selection runs once per CTA, so the instructions it executes are fetched once, mostly
// from memory; the kernel therefore keeps its code short: the keys live in shared memory (and four
// per thread in registers), each step is a short loop shared by the CTA's threads, and only the
// rare fallback (more than 64 keys at or above the bound) runs the one-warp selection of
// topk_pass.  Steps:
//   bound     lb = the k-th largest of 32 group maxima (group g: the keys of threads g, g + 32,
//             ..., 28 of E = 896), a 32-entry sort in warp 0: k groups hold keys at least that
//             large, so every selected key is >= lb;
//   rank      the keys >= lb (at most 64) sorted by (key descending, index ascending) in warp 0:
//             ranks 0..k-1 and the (k+1)-th key (or the largest key below lb);
//   settle    as topk_refine_kernel: when the list's order is not certain within the key
//             uncertainty, the contenders (the selected experts and, at an uncertain boundary,
//             the band) are listed in ascending expert order and the CTA's warps settle them
//             with refine_finish, from x's row and the router rows staged in shared memory
//             (`stage_rows` rows per batch; 0: straight from global memory).
// refine_count[0] counts the settled tokens, refine_count[1] the near ties.
constexpr int kSmallWarps = 8;
constexpr int kSmallThreads = 32 * kSmallWarps;
constexpr int kSmallSlots = 4;  // keys per thread: E <= kSmallSlots * kSmallThreads
constexpr int kSmallStageRows = 4;                   // router rows staged per batch
constexpr size_t kSmallStageMax = 100 * 1024;        // staging budget (two CTAs per SM fit)

// Dynamic shared memory: keys, scores and flags of the E experts, then the staging area.
__device__ __forceinline__ size_t topk_small_keys_bytes_dev(int E) {
  return ((size_t)E * (3 * sizeof(float) + 1) + 15) / 16 * 16;
}
size_t topk_small_keys_bytes(int E) { return ((size_t)E * (3 * sizeof(float) + 1) + 15) / 16 * 16; }
int topk_small_stage_rows(const RouterSrc& src) {
  const size_t bx = (size_t)src.d * (src.x_dtype == kBF16 ? 2 : 4);
  const size_t bw = (size_t)src.d * (src.w_dtype == kBF16 ? 2 : 4);
  for (int r = kSmallStageRows; r > 0; --r)
    if (bx + r * bw <= kSmallStageMax) return r;
  return 0;
}
size_t topk_small_smem(int E, const RouterSrc& src) {
  const int r = topk_small_stage_rows(src);
  const size_t bx = (size_t)src.d * (src.x_dtype == kBF16 ? 2 : 4);
  const size_t bw = (size_t)src.d * (src.w_dtype == kBF16 ? 2 : 4);
  return topk_small_keys_bytes(E) + (r > 0 ? bx + r * bw : 0);
}

template <int NPL>
__global__ void __launch_bounds__(kSmallThreads, 2) topk_small_kernel(
    float* logits, const float* __restrict__ bias, RouterSrc src, int T, int E, int k, int32_t* __restrict__ idx,
    float* __restrict__ p, int32_t* __restrict__ refine_count, uint32_t* status, int stage_rows,
    SplitPartials part) {
  extern __shared__ __align__(16) float s_dyn[];
  float* s_sv = s_dyn;                                           // [E] scores
  float* s_kf = s_dyn + E;                                       // [E] keys
  float* s_lg = s_dyn + 2 * E;                                   // [E] logits
  uint8_t* s_flag = reinterpret_cast<uint8_t*>(s_dyn + 3 * E);  // [E] 1: selected, 2: recompute
  const RefineStage stage{stage_rows > 0 ? reinterpret_cast<uint8_t*>(s_dyn) + topk_small_keys_bytes_dev(E) : nullptr,
                          stage_rows};
  __shared__ uint64_t s_ck[64];  // candidates: orderable key << 32 | (0xFFFF - expert) << 16
  __shared__ float s_ss[64];     // topk_pass scratch
  __shared__ int s_ce[kMaxCont];
  __shared__ uint64_t s_key[kMaxCont];
  __shared__ float s_s[kMaxCont];
  __shared__ int s_exa[kMaxCont];
  __shared__ int s_cand[kMaxCont];
  __shared__ float2 s_part[kSmallWarps][kMaxCont];
  __shared__ int s_n[2];
  __shared__ uint32_t s_cnt, s_below, s_dmax;
  __shared__ float s_ak, s_ak1;
  __shared__ int s_need, s_unc;
  __shared__ int s_wc[kSmallWarps], s_wr[kSmallWarps];
  __shared__ uint32_t s_tmax[kSmallThreads];
  __shared__ uint32_t s_lb;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const RefineSmem sm{s_ce, s_key, s_s, s_exa, s_cand, &s_part[0][0], s_n};
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    if (tid == 0) {
      s_cnt = 0;
      s_below = 0;
      s_dmax = 0;
    }
    // keys and scores (every load in flight at once), this thread's largest key
    float kf[kSmallSlots], sv[kSmallSlots];
    uint32_t ko[kSmallSlots];
    {
      float lg[kSmallSlots], bs[kSmallSlots];
      if (part.splits > 0) {
        // the router GEMM's split-K sums, added in split order from zero (the arithmetic of the
        // split-K reduction), eight splits of every slot in flight at a time; then written out
#pragma unroll
        for (int i = 0; i < kSmallSlots; ++i) lg[i] = 0.f;
        const float* pr = part.part + (int64_t)t * part.ldp;
#pragma unroll 1
        for (int s0 = 0; s0 < part.splits; s0 += 8) {
          float a[kSmallSlots][8];
#pragma unroll
          for (int i = 0; i < kSmallSlots; ++i)
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int e = tid + kSmallThreads * i;
              a[i][q] = e < E && s0 + q < part.splits ? pr[(int64_t)(s0 + q) * part.split_stride + e] : 0.f;
            }
#pragma unroll
          for (int i = 0; i < kSmallSlots; ++i)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (s0 + q < part.splits) lg[i] += a[i][q];
        }
#pragma unroll
        for (int i = 0; i < kSmallSlots; ++i) {
          const int e = tid + kSmallThreads * i;
          if (e < E) logits[(size_t)t * E + e] = lg[i];
        }
      } else {
#pragma unroll
        for (int i = 0; i < kSmallSlots; ++i) {
          const int e = tid + kSmallThreads * i;
          lg[i] = e < E ? logits[(size_t)t * E + e] : 0.f;
        }
      }
#pragma unroll
      for (int i = 0; i < kSmallSlots; ++i) {
        const int e = tid + kSmallThreads * i;
        bs[i] = bias && e < E ? __ldg(bias + e) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < kSmallSlots; ++i) {
        const int e = tid + kSmallThreads * i;
        const float s = 1.0f / (1.0f + expf(-lg[i]));  // the arithmetic of expert_key
        sv[i] = e < E ? s : 0.f;
        kf[i] = e < E ? (bias ? s + bs[i] : s) : -INFINITY;
        ko[i] = e < E ? orderable(kf[i]) : 0u;
        if (e < E) {
          s_sv[e] = s;
          s_kf[e] = kf[i];
          s_lg[e] = lg[i];
          s_flag[e] = 0;
        }
      }
    }
    uint32_t tmax = 0;
#pragma unroll
    for (int i = 0; i < kSmallSlots; ++i) tmax = ko[i] > tmax ? ko[i] : tmax;
    s_tmax[tid] = tmax;
    __syncthreads();
    // bound (warp 0): the k-th largest group maximum, by a 32-entry bitonic sort (descending)
    if (warp == 0) {
      uint32_t v = 0;
#pragma unroll
      for (int j = 0; j < kSmallThreads / 32; ++j) v = s_tmax[lane + 32 * j] > v ? s_tmax[lane + 32 * j] : v;
#pragma unroll
      for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          const uint32_t o = __shfl_xor_sync(0xffffffffu, v, stride);
          const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
          v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
        }
      const uint32_t lb_w = __shfl_sync(0xffffffffu, v, k - 1);
      if (lane == 0) s_lb = lb_w;
    }
    __syncthreads();
    const uint32_t lb = s_lb;
    uint32_t below = 0;
#pragma unroll
    for (int i = 0; i < kSmallSlots; ++i) {
      const int e = tid + kSmallThreads * i;
      if (ko[i] >= lb && ko[i] != 0u) {
        const uint32_t pos = atomicAdd(&s_cnt, 1u);
        if (pos < 64) s_ck[pos] = ((uint64_t)ko[i] << 32) | ((uint64_t)(0xFFFFu - (uint32_t)e) << 16);
      } else if (ko[i] > below) {
        below = ko[i];
      }
    }
    if (below) atomicMax(&s_below, below);
    __syncthreads();
    const int cnt = (int)s_cnt;
    // rank (warp 0): ranks 0..k-1 on lanes 0..k-1, the k-th and (k+1)-th keys
    int my_e = 0;
    float my_s = 0.f, my_kf = 0.f;
    if (warp == 0) {
      float a_k, a_k1 = -INFINITY;
      if (cnt <= 64) {
        uint64_t key[2];
        uint32_t aux[2] = {0u, 0u};
        key[0] = 2 * lane < cnt ? s_ck[2 * lane] : 0ull;
        key[1] = 2 * lane + 1 < cnt ? s_ck[2 * lane + 1] : 0ull;
        sort64_desc(key, aux, lane);
        const uint64_t mine = entry_key(key, lane < k ? lane : 0);
        if (lane < k) {
          my_e = (int)(0xFFFFu - (uint32_t)((mine >> 16) & 0xFFFFu));
          my_kf = from_orderable((uint32_t)(mine >> 32));
          my_s = s_sv[my_e];
        }
        a_k = from_orderable((uint32_t)(entry_key(key, k - 1) >> 32));
        if (k < E) a_k1 = from_orderable(cnt > k ? (uint32_t)(entry_key(key, k) >> 32) : s_below);
      } else {  // many keys tie at or near the bound: the one-warp selection by bisection
        TopkState<NPL> st;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
          const int e = lane + 32 * i;
          st.kf[i] = e < E ? s_kf[e] : -INFINITY;
          st.sv[i] = e < E ? s_sv[e] : 0.f;
        }
        topk_pass<NPL>(logits, bias, t, E, k, lane, st, s_ck, s_ss, true);
        my_e = st.my_e;
        my_s = st.my_s;
        my_kf = st.my_kf;
        a_k = st.a_k;
        a_k1 = st.a_k1;
      }
      if (lane == 0) {
        s_ak = a_k;
        s_ak1 = a_k1;
      }
    }
    __syncthreads();
    const float a_k = s_ak, a_k1 = s_ak1;
    // the key uncertainty of the token's contenders (token_eta over the CTA)
    {
      const float lo_eta = a_k1 - 2.0f * key_eta(src);
      float dm = 0.0f;
#pragma unroll
      for (int i = 0; i < kSmallSlots; ++i)
        if (kf[i] >= lo_eta) dm = fmaxf(dm, sv[i] * (1.0f - sv[i]));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dm = fmaxf(dm, __shfl_xor_sync(0xffffffffu, dm, off));
      if (lane == 0) atomicMax(&s_dmax, __float_as_uint(dm));  // dm >= 0: bit order is value order
    }
    __syncthreads();
    const float eta2 = 2.0f * (src.margin * (__uint_as_float(s_dmax) + 1e-4f) + 1e-6f);
    if (warp == 0) {
      const bool unc = k < E && a_k - a_k1 < eta2;
      const float prev = __shfl_up_sync(0xffffffffu, my_kf, 1);
      const float next = __shfl_down_sync(0xffffffffu, my_kf, 1);
      const bool close_next = lane + 1 < k && my_kf - next < eta2;
      const bool need = unc || __any_sync(0xffffffffu, close_next);
      if (need) {
        // ranks whose order against a neighbouring rank (or an uncertain boundary) is not certain
        const bool close = lane < k && ((lane > 0 && prev - my_kf < eta2) || close_next || (lane == k - 1 && unc));
        if (lane < k) s_flag[my_e] = close ? 3 : 1;
        if (lane == 0) atomicAdd(refine_count, 1);
      } else {
        topk_write(t, k, my_e, my_s, idx, p, lane);
      }
      if (lane == 0) {
        s_need = need ? 1 : 0;
        s_unc = unc ? 1 : 0;
      }
    }
    __syncthreads();
    if (s_need) {  // uniform over the CTA
      // contenders in ascending expert order: the selected experts and the band
      const bool unc = s_unc != 0;
      const float band_hi = a_k + eta2, band_lo = a_k1 - eta2;
      int n_cont = 0, n_rc = 0;
#pragma unroll 1
      for (int i = 0; i < kSmallSlots; ++i) {
        const int e = tid + kSmallThreads * i;
        int f = 0;
        float kfe = 0.f;
        if (e < E) {
          f = s_flag[e];
          kfe = s_kf[e];
          if (unc && kfe >= band_lo && kfe <= band_hi) f |= 2;
        }
        const uint32_t mc = __ballot_sync(0xffffffffu, f != 0);
        if (lane == 0) s_wc[warp] = __popc(mc);
        __syncthreads();
        int before = 0, total = 0;
        for (int w = 0; w < kSmallWarps; ++w) {
          const int c = s_wc[w];
          before += w < warp ? c : 0;
          total += c;
        }
        const int at = n_cont + before + __popc(mc & lt_mask);
        const bool in = f != 0 && at < kMaxCont;
        const bool r = in && (f & 2);
        const uint32_t mr = __ballot_sync(0xffffffffu, r);
        if (lane == 0) s_wr[warp] = __popc(mr);
        __syncthreads();
        int before_r = 0, total_r = 0;
        for (int w = 0; w < kSmallWarps; ++w) {
          const int c = s_wr[w];
          before_r += w < warp ? c : 0;
          total_r += c;
        }
        if (in) {
          s_ce[at] = e;
          s_key[at] = orderable64((double)kfe);
          s_s[at] = s_sv[e];
          s_exa[at] = 0;
          if (r) s_cand[n_rc + before_r + __popc(mr & lt_mask)] = at;
        }
        n_cont += total;
        n_rc += total_r;
        __syncthreads();  // s_wc / s_wr are rewritten by the next slot
      }
      if (tid == 0) {
        if (n_cont > kMaxCont) report(status, kStatusDeviceCheck);  // the first kMaxCont are ranked
        s_n[0] = n_cont < kMaxCont ? n_cont : kMaxCont;
        s_n[1] = n_rc;
      }
      refine_finish<NPL, kSmallWarps>(s_lg, bias, src, t, E, k, idx, p, warp, lane, sm, status,
                                      refine_count + 1, stage);
    }
    __syncthreads();  // shared memory is reused by the next token
  }
}

__global__ void split_bf16x3_kernel(const float* __restrict__ w, int64_t n, __nv_bfloat16* __restrict__ out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float v = w[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);  // exact in fp32
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    out[i] = hi;
    out[n + i] = mid;
    out[2 * n + i] = __float2bfloat16_rn(r2);
  }
}

constexpr int kMaskWords = kDispatchChunk / 32;

// Per-chunk bit mask of the tokens that selected each expert.  Returns false (and reports)
// for an index outside [0,E) or an expert listed twice for one token.
__device__ __forceinline__ void build_masks(const int32_t* __restrict__ idx, int T, int E, int k, uint32_t* mask,
                                            uint32_t* status) {
  for (int i = threadIdx.x; i < E * kMaskWords; i += blockDim.x) mask[i] = 0;
  __syncthreads();
  const int t = blockIdx.x * kDispatchChunk + threadIdx.x;
  if (t < T) {
    // the token's expert ids eight at a time, each batch's loads in flight together
    for (int j0 = 0; j0 < k; j0 += 8) {
      int ex[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) ex[u] = j0 + u < k ? __ldg(idx + (size_t)t * k + j0 + u) : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + u >= k) break;
        const int e = ex[u];
        if (e < 0 || e >= E) {
          report(status, kStatusDeviceCheck);
          continue;
        }
        const uint32_t bit = 1u << (threadIdx.x & 31);
        const uint32_t old = atomicOr(&mask[e * kMaskWords + (threadIdx.x >> 5)], bit);
        if (old & bit) report(status, kStatusDeviceCheck);
      }
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kDispatchChunk) dispatch_count_kernel(const int32_t* __restrict__ idx, int T,
                                                                        int E, int k,
                                                                        int32_t* __restrict__ chunk_counts,
                                                                        uint32_t* status) {
  extern __shared__ uint32_t mask[];
  build_masks(idx, T, E, k, mask, status);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < kMaskWords; ++w) c += __popc(mask[e * kMaskWords + w]);
    chunk_counts[(size_t)blockIdx.x * E + e] = c;
  }
}

// Per-expert row offsets, chunk bases and the four tile lists from thread e's expert total
// (1024 threads, E <= 1024): inclusive scans over the 1024 entries, within each warp by shuffles
// and then over the 32 warp totals (integer: exact).  Returns the expert's first row.
struct ScanSmem {
  int *cnt, *tiles, *tiles_s, *tiles_p, *tiles_m;  // [1024] each
};
__device__ __forceinline__ int scan_experts(int e, int total, int E, const ScanSmem& sh, int32_t* __restrict__ offsets,
                                            int4* __restrict__ tiles, int32_t* __restrict__ num_tiles,
                                            int4* __restrict__ tiles_s, int32_t* __restrict__ num_tiles_s,
                                            int4* __restrict__ tiles_p, int32_t* __restrict__ num_tiles_p,
                                            int4* __restrict__ tiles_m, int32_t* __restrict__ num_tiles_m) {
  const int nt = (total + kTileM - 1) / kTileM;
  const int nts = (total + kTileS - 1) / kTileS;
  const int ntp = (total + kTileP - 1) / kTileP;
  const int ntm = (total + kTileMx - 1) / kTileMx;
  int* const arr[5] = {sh.cnt, sh.tiles, sh.tiles_s, sh.tiles_p, sh.tiles_m};  // [32] warp totals each
  int v[5] = {total, nt, nts, ntp, ntm};
  const int lane = e & 31, w = e >> 5;
#pragma unroll
  for (int q = 0; q < 5; ++q)
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v[q], off);
      if (lane >= off) v[q] += o;
    }
  if (lane == 31)
#pragma unroll
    for (int q = 0; q < 5; ++q) arr[q][w] = v[q];
  __syncthreads();
  if (w == 0) {
#pragma unroll
    for (int q = 0; q < 5; ++q) {
      int x = arr[q][lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += o;
      }
      arr[q][lane] = x;  // inclusive over warps 0..lane
    }
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < 5; ++q) v[q] += w > 0 ? arr[q][w - 1] : 0;  // inclusive over entries 0..e
  __syncthreads();  // the warp totals may be rewritten by the caller
  const int row0 = v[0] - total;
  const int tile0 = v[1] - nt;
  const int tile0s = v[2] - nts;
  const int tile0p = v[3] - ntp;
  const int tile0m = v[4] - ntm;
  if (e < E) {
    offsets[e] = row0;
    for (int j = 0; j < nt; ++j) tiles[tile0 + j] = make_int4(e, tile0, total, row0);
    if (tiles_s)
      for (int j = 0; j < nts; ++j) tiles_s[tile0s + j] = make_int4(e, row0 + kTileS * j, min(kTileS, total - kTileS * j), 0);
    if (tiles_p)
      for (int j = 0; j < ntp; ++j) tiles_p[tile0p + j] = make_int4(e, tile0p, total, row0);
    if (tiles_m)
      for (int j = 0; j < ntm; ++j) tiles_m[tile0m + j] = make_int4(e, tile0m, total, row0);
  }
  if (e == E - 1) {
    offsets[E] = v[0];
    *num_tiles = v[1];
    if (num_tiles_s) *num_tiles_s = v[2];
    if (num_tiles_p) *num_tiles_p = v[3];
    if (num_tiles_m) *num_tiles_m = v[4];
  }
  return row0;
}

__global__ void __launch_bounds__(1024) dispatch_scan_kernel(const int32_t* __restrict__ chunk_counts,
                                                             int nchunks, int E, int32_t* __restrict__ chunk_base,
                                                             int32_t* __restrict__ offsets, int4* __restrict__ tiles,
                                                             int32_t* __restrict__ num_tiles,
                                                             int4* __restrict__ tiles_s,
                                                             int32_t* __restrict__ num_tiles_s,
                                                             int4* __restrict__ tiles_p,
                                                             int32_t* __restrict__ num_tiles_p,
                                                             int4* __restrict__ tiles_m,
                                                             int32_t* __restrict__ num_tiles_m) {
  __shared__ int s_cnt[1024], s_tiles[1024], s_tiles_s[1024], s_tiles_p[1024], s_tiles_m[1024];
  const ScanSmem sh{s_cnt, s_tiles, s_tiles_s, s_tiles_p, s_tiles_m};
  const int e = threadIdx.x;
  int total = 0;
  if (e < E)
    for (int c = 0; c < nchunks; ++c) total += chunk_counts[(size_t)c * E + e];
  const int row0 = scan_experts(e, total, E, sh, offsets, tiles, num_tiles, tiles_s, num_tiles_s, tiles_p,
                                num_tiles_p, tiles_m, num_tiles_m);
  if (e < E) {
    int run = row0;
    for (int c = 0; c < nchunks; ++c) {
      chunk_base[(size_t)c * E + e] = run;
      run += chunk_counts[(size_t)c * E + e];
    }
  }
}

// Batches of one dispatch chunk (T <= 256, E <= 1024): count, scan and scatter in one CTA, the
// same arithmetic as the three-kernel path (masks of the chunk's tokens per expert, stable ranks).
__global__ void __launch_bounds__(1024) dispatch_small_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ p, int T, int E, int k, int32_t* __restrict__ offsets,
    int4* __restrict__ tiles, int32_t* __restrict__ num_tiles, int4* __restrict__ tiles_s,
    int32_t* __restrict__ num_tiles_s, int4* __restrict__ tiles_p, int32_t* __restrict__ num_tiles_p,
    int4* __restrict__ tiles_m, int32_t* __restrict__ num_tiles_m, int32_t* __restrict__ tok_of_row,
    int32_t* __restrict__ row_of, float* __restrict__ p_row, uint32_t* status) {
  extern __shared__ uint32_t mask[];  // [E][kMaskWords]
  __shared__ int s_cnt[1024], s_tiles[1024], s_tiles_s[1024], s_tiles_p[1024], s_tiles_m[1024], s_row0[1024];
  const ScanSmem sh{s_cnt, s_tiles, s_tiles_s, s_tiles_p, s_tiles_m};
  build_masks(idx, T, E, k, mask, status);  // thread t < T is token t
  const int e = threadIdx.x;
  int total = 0;
  if (e < E)
#pragma unroll
    for (int w = 0; w < kMaskWords; ++w) total += __popc(mask[e * kMaskWords + w]);
  s_row0[e] = scan_experts(e, total, E, sh, offsets, tiles, num_tiles, tiles_s, num_tiles_s, tiles_p, num_tiles_p,
                           tiles_m, num_tiles_m);
  __syncthreads();
  const int t = threadIdx.x;
  if (t >= T) return;
  const int w = t >> 5;
  const uint32_t below = (1u << (t & 31)) - 1u;
  for (int j0 = 0; j0 < k; j0 += 8) {  // eight selections at a time, their loads in flight together
    int exs[8];
    float ps[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      exs[u] = j0 + u < k ? __ldg(idx + (size_t)t * k + j0 + u) : 0;
      ps[u] = p && j0 + u < k ? __ldg(p + (size_t)t * k + j0 + u) : 1.0f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u;
      if (j >= k) break;
      const int ex = exs[u];
      if (ex < 0 || ex >= E) {
        if (row_of) row_of[(size_t)t * k + j] = -1;
        continue;
      }
      const uint32_t* m = mask + ex * kMaskWords;
      int rank = __popc(m[w] & below);
      for (int q = 0; q < w; ++q) rank += __popc(m[q]);
      const int row = s_row0[ex] + rank;
      if (row_of) row_of[(size_t)t * k + j] = row;
      if (tok_of_row) tok_of_row[row] = t;
      if (p_row) p_row[row] = ps[u];
    }
  }
}

__global__ void __launch_bounds__(kDispatchChunk) dispatch_scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ p, int T, int E, int k,
    const int32_t* __restrict__ chunk_base, int32_t* __restrict__ tok_of_row, int32_t* __restrict__ row_of,
    float* __restrict__ p_row) {
  extern __shared__ uint32_t mask[];
  build_masks(idx, T, E, k, mask, nullptr);
  const int t = blockIdx.x * kDispatchChunk + threadIdx.x;
  if (t >= T) return;
  const int w = threadIdx.x >> 5;
  const uint32_t below = (1u << (threadIdx.x & 31)) - 1u;
  for (int j = 0; j < k; ++j) {
    const int e = idx[(size_t)t * k + j];
    if (e < 0 || e >= E) {
      if (row_of) row_of[(size_t)t * k + j] = -1;
      continue;
    }
    const uint32_t* m = mask + e * kMaskWords;
    int rank = __popc(m[w] & below);
    for (int q = 0; q < w; ++q) rank += __popc(m[q]);
    const int row = chunk_base[(size_t)blockIdx.x * E + e] + rank;
    if (row_of) row_of[(size_t)t * k + j] = row;
    if (tok_of_row) tok_of_row[row] = t;
    if (p_row) p_row[row] = p ? p[(size_t)t * k + j] : 1.0f;
  }
}

// Rows of z into expert-contiguous order with bulk copies: one warp per CTA keeps kScatterSlots
// token rows in shared memory.  Lane 0 loads rows kScatterAhead tokens ahead of their use; lane j
// writes the slot to the token's j-th destination row (k <= 32), one bulk group per token and lane.
// A slot is reloaded once every lane's stores from it have finished reading.
constexpr int kScatterSlots = 4, kScatterAhead = 2;

__global__ void __launch_bounds__(32) scatter_rows_kernel(const char* __restrict__ src, char* __restrict__ dst,
                                                          const int32_t* __restrict__ row_of, int T, int k,
                                                          uint32_t row_bytes, uint32_t* status, uint64_t timeout_ns) {
  extern __shared__ __align__(128) unsigned char slot_mem[];
  __shared__ __align__(8) uint64_t full[kScatterSlots];
  __shared__ int abort_flag;
  const int lane = threadIdx.x;
  const int first = blockIdx.x, stride = gridDim.x;
  const int n = first < T ? (T - first + stride - 1) / stride : 0;  // tokens first, first + stride, ...
  if (lane == 0) {
    for (int i = 0; i < kScatterSlots; ++i) ptx::mbar_init(&full[i], 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncwarp();
  auto load = [&](int i) {
    uint64_t* bar = &full[i % kScatterSlots];
    ptx::mbar_arrive_expect_tx(bar, row_bytes);
    ptx::bulk_load(slot_mem + (size_t)(i % kScatterSlots) * row_bytes, src + (size_t)(first + i * stride) * row_bytes,
                   row_bytes, bar);
  };
  int issued = n < kScatterAhead ? n : kScatterAhead;
  if (lane == 0)
    for (int i = 0; i < issued; ++i) load(i);
  int i = 0;
  for (; i < n; ++i) {
    if (i + kScatterAhead < n) {
      // the slot of token i + ahead last held token i + ahead - slots: its stores are the
      // (slots - ahead)-th most recent bulk group of every lane
      ptx::bulk_wait_read<kScatterSlots - kScatterAhead - 1>();
      __syncwarp();
      if (lane == 0) load(i + kScatterAhead);
      ++issued;
    }
    const int t = first + i * stride;
    const int r = lane < k ? row_of[(size_t)t * k + lane] : -1;
    const bool ok = ptx::mbar_wait_bounded(&full[i % kScatterSlots], (uint32_t)(i / kScatterSlots) & 1u, &abort_flag,
                                           status, timeout_ns);
    if (!__all_sync(0xffffffffu, ok)) break;
    if (r >= 0) ptx::bulk_store(dst + (size_t)r * row_bytes, slot_mem + (size_t)(i % kScatterSlots) * row_bytes, row_bytes);
    ptx::bulk_commit();
  }
  if (lane == 0)  // after a wait gave up: let the loads still in flight land before the CTA exits
    for (int j = i; j < issued; ++j) {
      const uint32_t bar = ptx::smem_addr(&full[j % kScatterSlots]);
      const uint64_t t0 = globaltimer_ns();
      while (!ptx::mbar_try_wait(bar, (uint32_t)(j / kScatterSlots) & 1u) && globaltimer_ns() - t0 < timeout_ns) {
      }
    }
  ptx::bulk_wait_all();
}

}  // namespace

cudaError_t launch_router_logits(const void* x, int x_dtype, const void* w_router, int w_dtype, float* logits,
                                 int T, int E, int d, cudaStream_t s) {
  SimtGemm g = {};
  g.A = x;
  g.lda = d;
  g.a_dtype = x_dtype;
  g.b_dtype = w_dtype;
  g.nseg = 1;
  g.seg[0] = SimtSegment{w_router, d, 0, d, d};
  g.M = T;
  g.N = E;
  g.K = d;
  g.C = logits;
  g.ldc = E;
  g.c_dtype = kF32;
  return launch_simt_gemm(g, s);
}

cudaError_t launch_router(const void* x, int act, const void* w_router, int router_w, float* logits,
                          void* wr_split, int T, int E, int d, uint32_t* status, uint64_t timeout_ns, int num_sms,
                          int* launches, cudaStream_t s, float* splitk, size_t splitk_bytes, bool pair_ok,
                          SplitPartials* defer) {
  if (defer) defer->splits = 0;
  if (act != kBF16) {
    if (launches) *launches += 1;
    return launch_router_logits(x, act, w_router, router_w, logits, T, E, d, s);
  }
  const void* wr = w_router;
  int terms = 1;
  if (router_w == kF32) {
    if (!wr_split) return cudaErrorInvalidValue;
    cudaError_t e = launch_split_bf16x3(static_cast<const float*>(w_router), (int64_t)E * d, wr_split, s);
    if (e != cudaSuccess) return e;
    if (launches) *launches += 1;
    wr = wr_split;
    terms = 3;
  }
  TcGemm g = {};
  g.epi = kEpiF32;
  g.M = T;
  g.N = E;
  g.K = terms * d;
  g.A = TcOperand{x, d, T, 1, d, (int64_t)T * d};
  g.B0 = TcOperand{wr, d, E, terms, d, (int64_t)E * d};
  g.k0_len = terms * d;
  g.k0_per_group = d;
  g.a_k_period = d;
  g.C = logits;
  g.ldc = E;
  g.partial = splitk;
  g.partial_bytes = splitk_bytes;
  g.defer = defer;
  g.launch_count = launches;
  const long long single_tiles = (long long)((T + 127) / 128) * ((E + 255) / 256);
  if (pair_ok && T >= 256 && single_tiles * 2 > num_sms && tc_pair_supported(g)) {
    if (launches) *launches += 1;
    return launch_tc_pair(g, status, timeout_ns, s);
  }
  return launch_tc_gemm(g, status, timeout_ns, 0, num_sms, s);
}

cudaError_t launch_split_bf16x3(const float* w, int64_t n, void* out, cudaStream_t s) {
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  split_bf16x3_kernel<<<(int)(blocks < 4096 ? blocks : 4096), threads, 0, s>>>(w, n,
                                                                              static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

cudaError_t launch_topk(float* logits, const float* bias, const RouterSrc& src, int T, int E, int k, int32_t* idx,
                        float* p, int32_t* refine_list, int32_t* refine_count, uint32_t* status, int num_sms,
                        cudaStream_t s, const SplitPartials* part) {
  cudaError_t e = cudaMemsetAsync(refine_count, 0, 2 * sizeof(int32_t), s);
  if (e != cudaSuccess || T <= 0) return e;
  const int warps_per_block = 8;
  dim3 grid((T + warps_per_block - 1) / warps_per_block), block(32 * warps_per_block);
  const int rgrid = 4 * num_sms;  // the residency the launch bounds give
  // short batches: both passes in one kernel, a CTA per token (the latency of one token's
  // selection and refinement, not the throughput of many, sets the time)
  const bool fused = T <= kTopkFusedMaxT;
  const SplitPartials sp = part ? *part : SplitPartials{nullptr, 0, 0, 0};
  if (sp.splits > 0 && !fused) return cudaErrorInvalidValue;  // only the short-batch kernel adds partials
  const int npl = (E + 31) / 32;
#define LMOE_TOPK(N)                                                                                     \
  do {                                                                                                   \
    if (fused) {                                                                                         \
      const size_t smem = topk_small_smem(E, src);                                                       \
      if (smem > 48 * 1024) {                                                                            \
        const cudaError_t ea = cudaFuncSetAttribute(topk_small_kernel<N>,                                \
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
        if (ea != cudaSuccess) return ea;                                                                \
      }                                                                                                  \
      topk_small_kernel<N><<<T, kSmallThreads, smem, s>>>(logits, bias, src, T, E, k, idx, p, refine_count, \
                                                          status, topk_small_stage_rows(src), sp);        \
    } else {                                                                                             \
      topk_kernel<N><<<grid, block, 0, s>>>(logits, bias, src, T, E, k, idx, p, refine_list, refine_count); \
      topk_refine_kernel<N><<<rgrid, 128, 0, s>>>(logits, bias, src, E, k, idx, p, refine_list, refine_count, \
                                                   status);                                                       \
    }                                                                                                    \
  } while (0)
  if (npl <= 1) LMOE_TOPK(1);
  else if (npl <= 2) LMOE_TOPK(2);
  else if (npl <= 4) LMOE_TOPK(4);
  else if (npl <= 8) LMOE_TOPK(8);
  else if (npl <= 16) LMOE_TOPK(16);
  else if (npl <= 28) LMOE_TOPK(28);
  else LMOE_TOPK(32);
#undef LMOE_TOPK
  return cudaGetLastError();
}

cudaError_t launch_dispatch(const int32_t* idx, const float* p, int T, int E, int k, const DispatchBuffers& b,
                            uint32_t* status, int* launches, cudaStream_t s) {
  const int nchunks = (T + kDispatchChunk - 1) / kDispatchChunk;
  const size_t smem = (size_t)E * kMaskWords * sizeof(uint32_t);
  if (nchunks == 1 && E <= 1024) {  // one chunk: one CTA does the three steps
    // 24 KB of static scan arrays next to the masks: above 48 KB in all the opt-in is needed
    if (smem > 16 * 1024) {
      const cudaError_t ea =
          cudaFuncSetAttribute(dispatch_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (ea != cudaSuccess) return ea;
    }
    dispatch_small_kernel<<<1, 1024, smem, s>>>(idx, p, T, E, k, b.offsets, b.tiles, b.num_tiles, b.tiles_s,
                                                b.num_tiles_s, b.tiles_p, b.num_tiles_p, b.tiles_m, b.num_tiles_m,
                                                b.tok_of_row, b.row_of, b.p_row, status);
    if (launches) *launches += 1;
    return cudaGetLastError();
  }
  dispatch_count_kernel<<<nchunks, kDispatchChunk, smem, s>>>(idx, T, E, k, b.chunk_counts, status);
  dispatch_scan_kernel<<<1, 1024, 0, s>>>(b.chunk_counts, nchunks, E, b.chunk_base, b.offsets, b.tiles,
                                          b.num_tiles, b.tiles_s, b.num_tiles_s, b.tiles_p, b.num_tiles_p,
                                          b.tiles_m, b.num_tiles_m);
  dispatch_scatter_kernel<<<nchunks, kDispatchChunk, smem, s>>>(idx, p, T, E, k, b.chunk_base, b.tok_of_row,
                                                                b.row_of, b.p_row);
  if (launches) *launches += 3;
  return cudaGetLastError();
}

cudaError_t launch_scatter_rows(const void* src, void* dst, const int32_t* row_of, int T, int k, int width,
                                int elem_bytes, uint32_t* status, uint64_t timeout_ns, int num_sms, cudaStream_t s) {
  const int64_t row_bytes = (int64_t)width * elem_bytes;
  if (T <= 0) return cudaSuccess;
  if (k < 1 || k > 32 || row_bytes % 16 || row_bytes > 16384 || (reinterpret_cast<uintptr_t>(src) & 15u) ||
      (reinterpret_cast<uintptr_t>(dst) & 15u))
    return cudaErrorInvalidValue;
  const int smem = kScatterSlots * (int)row_bytes;  // <= 64 KB
  if (smem > 48 * 1024) {  // the opt-in limit is a per-device function attribute: set it where it is needed
    cudaError_t e = cudaFuncSetAttribute(scatter_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  const int per_sm = smem <= 32768 ? 6 : 3;
  const int grid = T < per_sm * num_sms ? T : per_sm * num_sms;
  scatter_rows_kernel<<<grid, 32, smem, s>>>(static_cast<const char*>(src), static_cast<char*>(dst), row_of, T, k,
                                             (uint32_t)row_bytes, status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace lmoe
