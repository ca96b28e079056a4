"""Oracle for the LatentMoE layer forward pass.  TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct CPU evaluation in fp64 of what the layer computes.
Only the test suite, the package's smoke check and the benchmark's CPU-baseline leg
may import it; the GPU library never calls it and shares no code with it.

Sources ("Lesson 6 - LatentMoE", kimi-k3-course.pages.dev):
  * section "show me the actual equation", eq. 11 (quoted from the K3 report section 2.3):
        u = sum_{i in T_k(x)} p_i * E_i^routed(W_down x)          (in R^l)
        y = sum_{j=1..N_s} E_j^shared(x) + W_up RMSNorm(u)        (in R^d)
    The extracted text lost the placement of the summation limits; the glossary right
    below the equation (T_k(x) = selected top-16, N_s = 2 shared experts) fixes them.
  * same section, eq. 13 (K3 report section 2.3.3):
        s_i = Sigmoid(W_r x_i);  T_i = argtopk(s_i + b);  p_ij = s_ij / sum_{r in T_i} s_ir
    with the bias b used for selection only.
  * section "Deriving the headline number": a routed expert is a GLU holding three
    matrices gate, up, down of sizes latent x hidden.
  * section "What extreme sparsity breaks": RMSNorm sits between aggregation and W_up.

Readings where the pages are silent (each listed in the design notes):
  * GLU composition: down( SiLU(gate v) * (up v) ), SiLU(v) = v / (1 + e^-v); the pages name
    the routed activation "SiTU-GLU" without defining it, the workload spec fixes SiLU.
  * RMSNorm: n = u * g / sqrt(mean(u^2) + eps), elementwise gain g, no bias.
  * Top-k ties: the lower expert index wins.  Ranks are kept: idx[:, 0] is the largest key.
  * No residual "+x": eq. 11 has no x term; the layer output is the sum of the two branches.
  * Identity experts (routing/dispatch stress workload): E_i(v) = v, output is u itself.

Storage formats accepted (widened exactly to fp64): float32/float64 arrays; uint16 arrays
holding bf16 bit patterns; MXFP4 = uint8 packed E2M1 pairs (element 2i in the low nibble)
plus one uint8 E8M0 scale per 32 elements along K (OCP Microscaling v1.0).

Pins (all in the CPU test suite): MXFP4 decode against the OCP E2M1 table for all 16 codes
x 255 scales; router/selection closed forms and a brute-force full sort; the pages'
parameter and dispatch arithmetic; a dense all-experts-under-a-0/1-mask evaluation; scalar
closed forms of the GLU and RMSNorm; identity-expert, zero-routed-weight and N_s=0
reductions; token-permutation invariance.  MXFP8 activation mode (K3's quantisation-aware
numerics, page "What K3 actually is", srikanthmalla.com: MXFP4 weights with MXFP8 activations):
the E4M3 codec against a library float8 conversion for all 256 codes, its rounding at every
midpoint, the power-of-two block scale rule at its boundaries.
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------------------------------
# Exact widening of stored values
# ----------------------------------------------------------------------------------------

def widen(a) -> np.ndarray:
    """Exact fp64 value of a stored array (bf16 bits as uint16, or float32/float64)."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if a.dtype in (np.float32, np.float64):
        return a.astype(np.float64)
    raise TypeError(f"unsupported stored dtype {a.dtype}")


def e2m1_value(nib) -> np.ndarray:
    """Value of 4-bit E2M1 codes: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.

    Exponent field 0 is subnormal: value = mantissa * 0.5.  Otherwise
    value = 2^(exp-1) * (1 + mantissa/2).  (OCP Microscaling v1.0, FP4 E2M1.)
    """
    nib = np.asarray(nib, dtype=np.int64)
    sign = np.where((nib >> 3) & 1, -1.0, 1.0)
    ex = (nib >> 1) & 3
    man = nib & 1
    mag = np.where(ex == 0, 0.5 * man, np.ldexp(1.0 + 0.5 * man, ex - 1))
    return sign * mag


def e8m0_value(e) -> np.ndarray:
    """Value of E8M0 scale bytes: 2^(e-127); 255 is NaN."""
    e = np.asarray(e, dtype=np.int64)
    return np.where(e == 255, np.nan, np.ldexp(1.0, e - 127))


def mxfp4_decode(packed, scales) -> np.ndarray:
    """Exact fp64 values of an MXFP4 array: packed [..., K/2] uint8, scales [..., K/32] uint8."""
    packed = np.asarray(packed, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    K = packed.shape[-1] * 2
    nib = np.empty(packed.shape[:-1] + (K,), dtype=np.uint8)
    nib[..., 0::2] = packed & 0x0F
    nib[..., 1::2] = packed >> 4
    assert scales.shape[-1] * 32 == K
    # the 16 code values from the bit-field definition, then looked up per element
    values = e2m1_value(np.arange(16))[nib]
    values *= np.repeat(e8m0_value(scales), 32, axis=-1)
    return values


def e4m3_value(code) -> np.ndarray:
    """Value of 8-bit E4M3 codes (OCP 8-bit floating point, E4M3): bit 7 sign, bits 6..3
    exponent (bias 7), bits 2..0 mantissa; exponent 0 is subnormal (mantissa * 2^-9); exponent
    15 with mantissa 7 is NaN (no infinities; largest finite 448)."""
    code = np.asarray(code, dtype=np.int64)
    sign = np.where((code >> 7) & 1, -1.0, 1.0)
    ex = (code >> 3) & 15
    man = code & 7
    mag = np.where(ex == 0, np.ldexp(man.astype(np.float64), -9), np.ldexp(1.0 + man / 8.0, ex - 7))
    mag = np.where((ex == 15) & (man == 7), np.nan, mag)
    return sign * mag


def e4m3_round(v) -> np.ndarray:
    """v rounded to the nearest E4M3 value, ties to the even code, |result| <= 448."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), 448.0)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # grid spacing: 2^-9 in the subnormal range (below 2^-6), else 2^(e-3) (3 mantissa bits)
    step = np.where(a < 2.0 ** -6, 2.0 ** -9, np.ldexp(1.0, (np.maximum(e, -6) - 3).astype(np.int64)))
    q = np.round(a / step) * step  # numpy rounds halves to even: the even multiple is the even code
    return np.sign(v) * np.minimum(q, 448.0)


def mxfp8_quantize(v) -> np.ndarray:
    """Values of the MXFP8 encoding of rows v [..., K] (K % 32 == 0): per 32-element block the
    scale is the smallest power of two s with max|v| <= 448 s (E8M0 exponent clamped to
    [-126, 126]; an all-zero block gives zeros), each element E4M3(v / s) * s."""
    v = np.asarray(v, dtype=np.float64)
    blk = v.reshape(v.shape[:-1] + (v.shape[-1] // 32, 32))
    amax = np.max(np.abs(blk), axis=-1, keepdims=True)
    with np.errstate(divide="ignore"):
        ex = np.ceil(np.log2(np.where(amax > 0, amax / 448.0, 1.0)))
    ex = np.clip(ex, -126, 126)
    s = np.ldexp(1.0, ex.astype(np.int64))
    q = e4m3_round(blk / s) * s
    q = np.where(amax > 0, q, 0.0)
    return q.reshape(v.shape)


def weight_values(w, scale=None) -> np.ndarray:
    """fp64 values of one stored weight matrix (MXFP4 when a scale array is given)."""
    if scale is not None:
        return mxfp4_decode(w, scale)
    return widen(w)


# ----------------------------------------------------------------------------------------
# Router: eq. 13
# ----------------------------------------------------------------------------------------

def sigmoid(v):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-v))


def router_logits(x, w_router) -> np.ndarray:
    """W_r x for each token row of x: [n, E]."""
    return x @ w_router.T


def router_scores(x, w_router) -> np.ndarray:
    """s = Sigmoid(W_r x) for each token row of x: [n, E]."""
    return sigmoid(router_logits(x, w_router))


def select_topk(s, bias, k):
    """T = argtopk(s + b): the k largest keys per row, ties to the lower index, in rank order.

    Returns (idx [n, k] int64, gap [n]) where gap = key_(k) - key_(k+1) (inf when k == E).
    """
    keys = s if bias is None else s + bias[None, :]
    n, E = keys.shape
    idx = np.empty((n, k), dtype=np.int64)
    gap = np.full(n, np.inf)
    order_index = np.arange(E)
    for t in range(n):
        # primary key: larger key first; secondary: smaller expert index first
        order = np.lexsort((order_index, -keys[t]))
        idx[t] = order[:k]
        if k < E:
            gap[t] = keys[t, order[k - 1]] - keys[t, order[k]]
    return idx, gap


def route_weights(s, idx) -> np.ndarray:
    """p_j = s_{idx_j} / sum_{r in T} s_r: normalised over the selected set, bias-free."""
    sel = np.take_along_axis(s, idx, axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


# ----------------------------------------------------------------------------------------
# Dispatch: selections converted into expert-contiguous batches
# ----------------------------------------------------------------------------------------

def dispatch(idx, num_experts):
    """Canonical expert batches for a routing table idx [T, k].

    counts[e]  = number of (t, j) with idx[t, j] == e
    offsets    = exclusive prefix sum of counts, length E+1
    tok_of_row = token of each row when rows are ordered by (expert, token)
    row_of     = [T, k] row that holds (t, j)
    """
    T, k = idx.shape
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=num_experts).astype(np.int64)
    offsets = np.zeros(num_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    order = np.argsort(flat, kind="stable")  # (t, j) flattened t-major: stable => token order
    tok_of_row = order // k
    row_of = np.empty(T * k, dtype=np.int64)
    row_of[order] = np.arange(T * k)
    return counts, offsets, tok_of_row, row_of.reshape(T, k)


# ----------------------------------------------------------------------------------------
# Experts and normalisation
# ----------------------------------------------------------------------------------------

def silu(v):
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def expert_matrix_shapes(width, hidden):
    """Shapes of the three matrices of one GLU expert acting on ``width`` channels."""
    return {"gate": (hidden, width), "up": (hidden, width), "down": (width, hidden)}


def glu_expert(v, gate_up, down, hidden):
    """E(v) = down( SiLU(gate v) * (up v) ) for rows v [n, width].

    gate_up holds gate in rows 0..hidden-1 and up in rows hidden..2*hidden-1.
    """
    width = v.shape[1]
    shapes = expert_matrix_shapes(width, hidden)
    gate, up = gate_up[:hidden], gate_up[hidden:]
    assert gate.shape == shapes["gate"] and up.shape == shapes["up"] and down.shape == shapes["down"]
    a = silu(v @ gate.T) * (v @ up.T)
    return a @ down.T


def glu_expert_mxfp8(v, gate_up, down, hidden):
    """The GLU expert with MXFP8 activations: its input rows and its GLU activations are
    quantised (mxfp8_quantize) before the products that read them."""
    gate, up = gate_up[:hidden], gate_up[hidden:]
    vq = mxfp8_quantize(v)
    a = silu(vq @ gate.T) * (vq @ up.T)
    return mxfp8_quantize(a) @ down.T


def rmsnorm(u, gain, eps):
    """n = u * g / sqrt(mean(u^2) + eps), per row."""
    ms = np.mean(u * u, axis=1, keepdims=True)
    return u * gain[None, :] / np.sqrt(ms + eps)


# ----------------------------------------------------------------------------------------
# The layer: eq. 11 with eq. 13 routing
# ----------------------------------------------------------------------------------------

def layer_forward(inp, cfg, tokens=None, routing=None, act_quant=None):
    """Evaluate the layer for the token rows ``tokens`` (all rows when None).

    ``inp`` holds stored arrays as produced by the input generator's host copy (routed
    weights may be any object indexable by expert).  ``cfg`` supplies top_k, hidden,
    shared_hidden, n_shared, rms_eps and identity_experts.  ``routing`` optionally forces
    (idx, p) for the evaluated rows instead of the router's choice.  ``act_quant="mxfp8"``:
    the routed experts take MXFP8 activations (glu_expert_mxfp8).

    Returns a dict with s, idx, p, gap, z, u, and (unless identity experts) n and y.
    Rows are independent given routing, so a row subset is an exact sub-problem.
    """
    X = inp["x"] if tokens is None else np.asarray(inp["x"])[tokens]
    x = widen(X)
    k = cfg.top_k
    w_r = widen(inp["w_router"])
    bias = None if inp.get("router_bias") is None else widen(inp["router_bias"])
    s = router_scores(x, w_r)
    idx, gap = select_topk(s, bias, k)
    p = route_weights(s, idx)
    if routing is not None:
        idx = np.asarray(routing[0], dtype=np.int64)
        p = np.asarray(routing[1], dtype=np.float64)
    z = x @ widen(inp["w_down_proj"]).T                      # W_down x, in R^l
    n_tok = x.shape[0]
    out_rows = np.zeros((n_tok, k, z.shape[1]))              # E_i(z) for each (t, j)
    if cfg.identity_experts:
        out_rows[:] = z[:, None, :]
    else:
        gu_w, gu_s = inp["routed_gate_up"], inp.get("routed_gate_up_scale")
        dn_w, dn_s = inp["routed_down"], inp.get("routed_down_scale")
        for e in np.unique(idx):
            t_sel, j_sel = np.nonzero(idx == e)
            gate_up = weight_values(gu_w[e], None if gu_s is None else gu_s[e])
            down = weight_values(dn_w[e], None if dn_s is None else dn_s[e])
            expert = glu_expert_mxfp8 if act_quant == "mxfp8" else glu_expert
            out_rows[t_sel, j_sel] = expert(z[t_sel], gate_up, down, cfg.hidden)
    u = np.zeros_like(z)
    for j in range(k):                                       # sum in rank order
        u += p[:, j:j + 1] * out_rows[:, j, :]
    res = {"s": s, "idx": idx, "p": p, "gap": gap, "z": z, "u": u}
    if cfg.identity_experts:
        return res
    n = rmsnorm(u, widen(inp["rms_gain"]), cfg.rms_eps)
    y = n @ widen(inp["w_up_proj"]).T                        # W_up RMSNorm(u)
    for i in range(cfg.n_shared):
        y += glu_expert(x, widen(inp["shared_gate_up"][i]), widen(inp["shared_down"][i]),
                        cfg.shared_hidden)
    res["n"] = n
    res["y"] = y
    return res
