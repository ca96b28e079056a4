"""Pins of the oracle to facts outside itself (CPU only).

Each test checks an oracle function against something the pages or mathematics fix:
printed arithmetic, closed forms, a published encoding table, a library routine in a
special case, brute force on tiny inputs, or an invariant.
"""
import json
import math
import os
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from sparse_moe_layer_sigmoid_gb300 import configs, inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    with open(os.path.join(GOLDEN, "pages_arithmetic.json")) as f:
        return json.load(f)


# -------------------------------------------------------------------------------------
# MXFP4 decode: OCP Microscaling v1.0 E2M1 table, all 16 codes x all 255 finite scales
# -------------------------------------------------------------------------------------

OCP_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_e8m0_exhaustive():
    codes = np.arange(16)
    vals = oracle.e2m1_value(codes)
    assert list(vals) == OCP_E2M1
    for e in range(255):
        got = oracle.e2m1_value(codes) * oracle.e8m0_value(e)
        want = np.array([v * 2.0 ** (e - 127) for v in OCP_E2M1])
        assert np.array_equal(got, want), e
    assert np.isnan(oracle.e8m0_value(255))


def test_mxfp4_nibble_order_and_scale_blocks():
    # byte 0x21: element 0 = low nibble 1 -> 0.5, element 1 = high nibble 2 -> 1.0
    packed = np.zeros((1, 32), dtype=np.uint8)
    packed[0, 0] = 0x21
    packed[0, 16] = 0x7F          # elements 32, 33: -6.0, 6.0
    scales = np.array([[127, 129]], dtype=np.uint8)  # block 0: x1, block 1: x4
    v = oracle.mxfp4_decode(packed, scales)
    assert v.shape == (1, 64)
    assert v[0, 0] == 0.5 and v[0, 1] == 1.0
    assert v[0, 32] == -6.0 * 4 and v[0, 33] == 6.0 * 4
    assert np.count_nonzero(v) == 4


def test_generator_mx_encoding_roundtrip_and_nearest():
    g = torch.Generator().manual_seed(7)
    # on-grid values with per-block power-of-two scales encode and decode exactly
    grid = torch.tensor(OCP_E2M1[:8] + [-v for v in OCP_E2M1[1:8]] + [6.0])
    pick = torch.randint(0, grid.numel(), (4, 256), generator=g)
    vals = grid[pick].reshape(4, 8, 32)
    vals[..., 0] = 6.0                                   # make amax = 6 in every block
    exps = torch.randint(-20, 20, (4, 8, 1), generator=g).float()
    w = (vals * torch.exp2(exps)).reshape(4, 256)
    packed, scales = inputs.encode_mxfp4(w)
    dec = oracle.mxfp4_decode(packed.numpy(), scales.numpy())
    assert np.array_equal(dec, w.double().numpy())
    # random values: each decoded element is a nearest grid point of the scaled value
    w = torch.randn(16, 64, generator=g)
    packed, scales = inputs.encode_mxfp4(w)
    dec = oracle.mxfp4_decode(packed.numpy(), scales.numpy())
    sc = np.repeat(oracle.e8m0_value(scales.numpy()), 32, axis=-1)
    mags = np.array(OCP_E2M1[:8])
    target = np.clip(w.double().numpy() / sc, -6, 6)
    best = np.min(np.abs(np.abs(target)[..., None] - mags), axis=-1)
    assert np.allclose(np.abs(np.abs(dec / sc) - np.abs(target)), best, atol=0)


# -------------------------------------------------------------------------------------
# Pages' arithmetic: shapes used by the oracle reproduce the printed figures
# -------------------------------------------------------------------------------------

def _expert_params(width, hidden):
    return sum(a * b for a, b in oracle.expert_matrix_shapes(width, hidden).values())


def test_pages_parameter_arithmetic():
    gd = _golden()
    w = gd["k3_widths"]
    d, l, h, E, k, Ns, L = w["d"], w["latent"], w["hidden"], w["experts"], w["top_k"], w["n_shared"], w["moe_layers"]
    per_expert = _expert_params(l, h)
    assert per_expert == 33_030_144
    assert abs(per_expert - gd["params_per_routed_expert"]["value"]) <= gd["params_per_routed_expert"]["rounding"]
    pool = per_expert * E
    assert abs(pool - gd["routed_pool_per_layer"]["value"]) <= gd["routed_pool_per_layer"]["rounding"]
    assert abs(pool * L - gd["routed_pool_all_layers"]["value"]) <= gd["routed_pool_all_layers"]["rounding"]
    full = _expert_params(d, h) * E * L
    assert abs(full - gd["routed_pool_full_width"]["value"]) <= gd["routed_pool_full_width"]["rounding"]
    # W_down [l][d] and W_up [d][l] as the oracle applies them
    proj = (l * d + d * l) * L
    assert abs(proj - gd["projections_all_layers"]["value"]) <= gd["projections_all_layers"]["rounding"]
    shared = _expert_params(d, h) * Ns * L
    assert abs(shared - gd["shared_experts_all_layers"]["value"]) <= gd["shared_experts_all_layers"]["rounding"]
    active = per_expert * k * L
    assert abs(active - gd["activated_routed_all_layers"]["value"]) <= gd["activated_routed_all_layers"]["rounding"]


def test_pages_dispatch_and_sparsity():
    gd = _golden()
    w = gd["k3_widths"]
    # rows the layer dispatches per token: k rows of width l (latent) vs d (full width)
    cfg = replace(configs.TINY_F32, tokens=1, d=w["d"], latent=w["latent"], experts=w["experts"], top_k=w["top_k"])
    assert cfg.rows * cfg.latent == gd["dispatch_values_latent"]["value"]
    assert cfg.rows * cfg.d == gd["dispatch_values_full"]["value"]
    assert w["experts"] // w["top_k"] == gd["sparsity_ratio"]["value"] and w["experts"] % w["top_k"] == 0
    frac = 100.0 * w["top_k"] / w["experts"]
    assert abs(frac - gd["active_fraction_percent"]["value"]) <= gd["active_fraction_percent"]["rounding"]
    assert (w["top_k"] * w["latent"] == 8 * w["d"]) is gd["top16_latent_equals_top8_full"]["value"]


# -------------------------------------------------------------------------------------
# Router (eq. 13)
# -------------------------------------------------------------------------------------

def test_router_scores_closed_form():
    x = np.array([[1.0, 0.0]])
    w_r = np.array([[0.0, 5.0], [math.log(3.0), 1.0], [-math.log(3.0), 2.0]])
    s = oracle.router_scores(x, w_r)
    assert np.allclose(s, [[0.5, 0.75, 0.25]], rtol=0, atol=1e-15)


def test_topk_ties_bias_and_weights_by_hand():
    s = np.array([[0.9, 0.8, 0.7, 0.6]])
    b = np.array([0.0, 0.0, 0.5, 0.0])
    idx, gap = oracle.select_topk(s, b, 2)
    assert idx.tolist() == [[2, 0]]                      # keys 0.9, 0.8, 1.2, 0.6
    assert abs(gap[0] - 0.1) < 1e-15
    p = oracle.route_weights(s, idx)
    assert np.allclose(p, [[0.7 / 1.6, 0.9 / 1.6]], rtol=0, atol=1e-15)  # bias absent from p
    # exact ties go to the lower index, ranks kept
    s2 = np.array([[0.5, 0.7, 0.5, 0.7, 0.1]])
    idx2, gap2 = oracle.select_topk(s2, None, 3)
    assert idx2.tolist() == [[1, 3, 0]] and gap2[0] == 0.0


def test_topk_brute_force_full_sort():
    rng = np.random.Generator(np.random.PCG64(11))
    for E, k in [(8, 3), (32, 4), (40, 40), (896, 16)]:
        s = oracle.sigmoid(rng.standard_normal((20, E)))
        b = rng.standard_normal(E) * 0.1
        s[0, :4] = 0.5                                      # some exact ties
        b[:4] = 0.0
        idx, gap = oracle.select_topk(s, b, k)
        for t in range(20):
            keys = [(s[t, e] + b[e], e) for e in range(E)]
            srt = sorted(keys, key=lambda kv: (-kv[0], kv[1]))
            assert idx[t].tolist() == [e for _, e in srt[:k]]
            if k < E:
                assert gap[t] == srt[k - 1][0] - srt[k][0]
            else:
                assert gap[t] == np.inf


def test_route_weights_invariants():
    rng = np.random.Generator(np.random.PCG64(12))
    E, k = 64, 8
    s = oracle.sigmoid(rng.standard_normal((50, E)))
    b = rng.standard_normal(E)
    idx, _ = oracle.select_topk(s, b, k)
    p = oracle.route_weights(s, idx)
    assert np.all(np.abs(p.sum(axis=1) - 1.0) < 1e-12)
    # a constant shift of the bias changes neither selection nor weights
    idx2, _ = oracle.select_topk(s, b + 3.25, k)
    assert np.array_equal(idx, idx2)
    assert np.array_equal(oracle.route_weights(s, idx2), p)
    # k = E selects every expert
    idx3, _ = oracle.select_topk(s, b, E)
    assert all(sorted(r) == list(range(E)) for r in idx3.tolist())


# -------------------------------------------------------------------------------------
# Dispatch
# -------------------------------------------------------------------------------------

def test_dispatch_brute_force():
    rng = np.random.Generator(np.random.PCG64(13))
    T, E, k = 37, 9, 3
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    counts, offsets, tok_of_row, row_of = oracle.dispatch(idx, E)
    rows = []
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    rows.append((t, j))
    assert [r[0] for r in rows] == tok_of_row.tolist()
    for r, (t, j) in enumerate(rows):
        assert row_of[t, j] == r
    for e in range(E):
        assert counts[e] == sum(1 for t in range(T) for j in range(k) if idx[t, j] == e)
        assert offsets[e] == sum(counts[:e])
    assert offsets[E] == T * k


# -------------------------------------------------------------------------------------
# Experts and RMSNorm
# -------------------------------------------------------------------------------------

def test_glu_scalar_closed_form():
    a, b, c, x = 0.7, -1.3, 2.5, 1.9
    out = oracle.glu_expert(np.array([[x]]), np.array([[a], [b]]), np.array([[c]]), 1)
    want = c * (a * x / (1.0 + math.exp(-a * x))) * (b * x)
    assert abs(out[0, 0] - want) < 1e-14
    swapped = c * (b * x / (1.0 + math.exp(-b * x))) * (a * x)
    assert abs(want - swapped) > 0.1


def test_glu_against_torch_silu():
    rng = np.random.Generator(np.random.PCG64(14))
    v = rng.standard_normal((5, 12))
    gu = rng.standard_normal((2 * 7, 12))
    dn = rng.standard_normal((12, 7))
    out = oracle.glu_expert(v, gu, dn, 7)
    tv, tg, td = (torch.from_numpy(a) for a in (v, gu, dn))
    want = (torch.nn.functional.silu(tv @ tg[:7].T) * (tv @ tg[7:].T)) @ td.T
    assert np.allclose(out, want.numpy(), rtol=1e-13, atol=1e-13)


def test_rmsnorm_closed_forms():
    n = oracle.rmsnorm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.0)
    r = math.sqrt((9 + 16) / 2)
    assert np.allclose(n, [[3 / r, 8 / r]], rtol=0, atol=1e-15)
    c, eps = -0.02, 1e-6
    n = oracle.rmsnorm(np.full((1, 6), c), np.full(6, 1.5), eps)
    assert np.allclose(n, 1.5 * np.sign(c) / math.sqrt(1 + eps / c ** 2), rtol=1e-15)


# -------------------------------------------------------------------------------------
# Whole layer on tiny inputs
# -------------------------------------------------------------------------------------

def _tiny(**kw):
    cfg = replace(configs.TINY_F32, tokens=24, d=32, latent=16, hidden=8, experts=12, top_k=3,
                  n_shared=1, shared_hidden=8)
    return replace(cfg, **kw)


def _host(cfg, seed=None):
    return inputs.host_inputs(inputs.make_inputs(cfg, "cpu", seed))


@pytest.mark.parametrize("bias", ["none", "normal1.5"])
def test_layer_matches_dense_all_experts_under_mask(bias):
    cfg = _tiny(bias=bias)
    inp = _host(cfg)
    res = oracle.layer_forward(inp, cfg)
    x = inp["x"].astype(np.float64)
    z = x @ inp["w_down_proj"].astype(np.float64).T
    gu = inp["routed_gate_up"].astype(np.float64)                      # [E, 2h, l]
    dn = inp["routed_down"].astype(np.float64)                         # [E, l, h]
    h = cfg.hidden
    # every expert on every token
    gate = np.einsum("tc,ehc->teh", z, gu[:, :h])
    up = np.einsum("tc,ehc->teh", z, gu[:, h:])
    act = gate / (1 + np.exp(-gate)) * up
    dense = np.einsum("teh,ech->tec", act, dn)                         # [T, E, l]
    # 0/1 mask from a full sort of biased sigmoid scores; weights use the unbiased scores
    s = 1 / (1 + np.exp(-(x @ inp["w_router"].astype(np.float64).T)))
    b = np.zeros(cfg.experts) if inp["router_bias"] is None else inp["router_bias"].astype(np.float64)
    mask = np.zeros_like(s)
    for t in range(cfg.tokens):
        mask[t, np.argsort(-(s[t] + b), kind="stable")[:cfg.top_k]] = 1.0
    wts = s * mask / (s * mask).sum(axis=1, keepdims=True)
    u = np.einsum("te,tec->tc", wts, dense)
    assert np.allclose(res["u"], u, rtol=1e-12, atol=1e-13)
    assert np.abs(res["u"] - u).max() <= 1e-13 * max(1.0, np.abs(u).max())


def test_layer_identity_experts_give_z():
    cfg = _tiny(identity_experts=True)
    inp = _host(cfg)
    res = oracle.layer_forward(inp, cfg)
    assert np.allclose(res["u"], res["z"], rtol=1e-14, atol=1e-14)


def test_layer_zero_routed_weights_give_shared_only():
    cfg = _tiny()
    inp = _host(cfg)
    inp["routed_gate_up"] = np.zeros_like(inp["routed_gate_up"])
    res = oracle.layer_forward(inp, cfg)
    assert np.all(res["u"] == 0) and np.all(res["n"] == 0)
    x = torch.from_numpy(inp["x"].astype(np.float64))
    gu = torch.from_numpy(inp["shared_gate_up"][0].astype(np.float64))
    dn = torch.from_numpy(inp["shared_down"][0].astype(np.float64))
    hs = cfg.shared_hidden
    want = (torch.nn.functional.silu(x @ gu[:hs].T) * (x @ gu[hs:].T)) @ dn.T
    assert np.allclose(res["y"], want.numpy(), rtol=1e-13, atol=1e-13)


def test_layer_no_shared_identity_up_is_textbook_rmsnorm():
    cfg = _tiny(n_shared=0)
    inp = _host(cfg)
    inp["w_up_proj"] = np.zeros((cfg.d, cfg.latent), dtype=np.float32)
    inp["w_up_proj"][:cfg.latent] = np.eye(cfg.latent, dtype=np.float32)
    res = oracle.layer_forward(inp, cfg)
    u = torch.from_numpy(res["u"])
    g = torch.from_numpy(inp["rms_gain"].astype(np.float64))
    want = torch.nn.functional.rms_norm(u, (cfg.latent,), weight=g, eps=cfg.rms_eps).numpy()
    assert np.allclose(res["y"][:, :cfg.latent], want, rtol=1e-13, atol=1e-14)
    assert np.all(res["y"][:, cfg.latent:] == 0)


def test_layer_top1_weight_is_one():
    cfg = _tiny(top_k=1)
    res = oracle.layer_forward(_host(cfg), cfg)
    assert np.all(res["p"] == 1.0)


def test_layer_token_permutation_invariance():
    cfg = _tiny()
    inp = _host(cfg)
    res = oracle.layer_forward(inp, cfg)
    perm = np.random.Generator(np.random.PCG64(3)).permutation(cfg.tokens)
    inp2 = dict(inp)
    inp2["x"] = inp["x"][perm]
    res2 = oracle.layer_forward(inp2, cfg)
    assert np.array_equal(res2["idx"], res["idx"][perm])
    assert np.allclose(res2["y"], res["y"][perm], rtol=1e-13, atol=1e-13)
    # evaluating a row subset is the same sub-problem
    sub = np.array([3, 17, 5])
    res3 = oracle.layer_forward(inp, cfg, tokens=sub)
    assert np.allclose(res3["y"], res["y"][sub], rtol=1e-13, atol=1e-13)


def test_layer_mxfp4_and_bf16_storage_decoded_exactly():
    cfg = _tiny(act="bf16", router_w="bf16", routed_w="mxfp4", hidden=32, latent=32, shared_hidden=32)
    inp = _host(cfg)
    assert inp["x"].dtype == np.uint16 and inp["routed_gate_up"].dtype == np.uint8
    res = oracle.layer_forward(inp, cfg)
    # same layer with the weights pre-decoded to fp64 arrays
    dec = dict(inp)
    for k in ("x", "w_router", "w_down_proj", "w_up_proj", "shared_gate_up", "shared_down"):
        dec[k] = oracle.widen(inp[k])
    dec["routed_gate_up"] = oracle.mxfp4_decode(inp["routed_gate_up"], inp["routed_gate_up_scale"])
    dec["routed_down"] = oracle.mxfp4_decode(inp["routed_down"], inp["routed_down_scale"])
    dec["routed_gate_up_scale"] = dec["routed_down_scale"] = None
    res2 = oracle.layer_forward(dec, cfg)
    assert np.array_equal(res["y"], res2["y"])
    # bf16 bit patterns widen to the values torch holds
    x_t = inputs.make_inputs(cfg, "cpu")["x"].double().numpy()
    assert np.array_equal(oracle.widen(inp["x"]), x_t)


# ---------------------------------------------------------------- MXFP8 activation mode

def test_e4m3_codec_matches_library_float8():
    """All 256 E4M3 codes decode to the values of torch's float8_e4m3fn; rounding to the E4M3
    grid matches torch's conversion at every midpoint between neighbouring values (ties to the
    even code) and on random values across the range."""
    codes = np.arange(256)
    lib = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = oracle.e4m3_value(codes)
    assert np.array_equal(np.isnan(lib), np.isnan(mine))
    assert np.array_equal(lib[~np.isnan(lib)], mine[~np.isnan(mine)])
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9
    vals = np.unique(np.abs(mine[~np.isnan(mine)]))
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(11)
    x = np.concatenate([mids, -mids, vals, rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 1e-2])
    lib_r = torch.tensor(x, dtype=torch.float64).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.e4m3_round(x), lib_r)
    assert oracle.e4m3_round(np.array([1e6, -1e6])).tolist() == [448.0, -448.0]  # saturates


def test_mxfp8_block_scale_rule():
    """The scale is the smallest power of two s with max|v| <= 448 s: a block whose maximum is
    448 * 2^k keeps it exactly (s = 2^k); one just above moves to s = 2^(k+1).  Encoding is
    idempotent, an all-zero block stays zero, and each element is within half a grid step."""
    v = np.zeros((1, 96))
    v[0, :32] = np.linspace(-1, 1, 32) * 448.0 * 2.0 ** -3
    v[0, 32:64] = np.linspace(-1, 1, 32) * 448.0 * 2.0 ** -3 * (1 + 2 ** -20)
    q = oracle.mxfp8_quantize(v)
    assert q[0, 31] == 448.0 * 2.0 ** -3           # exact at the top of its scale
    assert q[0, 63] == 448.0 * 2.0 ** -3           # rounds back from the next scale up
    assert np.all(q[0, 64:] == 0.0)
    assert np.array_equal(oracle.mxfp8_quantize(q), q)
    rng = np.random.default_rng(12)
    w = rng.standard_normal((8, 256)) * np.logspace(-4, 4, 8)[:, None]
    qw = oracle.mxfp8_quantize(w)
    blk = np.abs(w).reshape(8, 8, 32).max(axis=2)
    s = 2.0 ** np.ceil(np.log2(blk / 448.0))
    step = np.repeat(s * 2.0 ** -3 * 2.0 ** np.floor(np.log2(blk / s)), 32, axis=1)  # a block's coarsest step
    assert np.all(np.abs(qw - w) <= step / 2 + 1e-300)


def test_mxfp8_expert_reduces_to_glu_without_quantisation(monkeypatch):
    """With the activation quantiser replaced by the identity, the MXFP8 expert is the GLU expert
    (same gate/up split and composition) and the MXFP8 layer is the plain layer."""
    rng = np.random.default_rng(13)
    v, gate_up, down = rng.standard_normal((5, 64)), rng.standard_normal((2 * 32, 64)), rng.standard_normal((64, 32))
    monkeypatch.setattr(oracle, "mxfp8_quantize", lambda a: a)
    import oracle.latentmoe_oracle as om
    monkeypatch.setattr(om, "mxfp8_quantize", lambda a: a)
    assert np.allclose(om.glu_expert_mxfp8(v, gate_up, down, 32), oracle.glu_expert(v, gate_up, down, 32), rtol=1e-13)
    cfg = configs.TINY_F32
    host = inputs.host_inputs(inputs.make_inputs(cfg, "cpu"))
    a = oracle.layer_forward(host, cfg, tokens=np.arange(8))["y"]
    b = oracle.layer_forward(host, cfg, tokens=np.arange(8), act_quant="mxfp8")["y"]
    assert np.array_equal(a, b)
