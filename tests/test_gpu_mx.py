"""The block-scaled MXFP4 path: three-term activation records and the kind::mxf4 expert GEMMs.

MXFP4 expert weights (page "What K3 actually is", srikanthmalla.com, the MXFP4 passage) meet the
activations on tcgen05.mma kind::mxf4, which multiplies E2M1 by E2M1 with an E8M0 scale per 32
elements along K on both operands (OCP Microscaling v1.0).  The activations are therefore split
into three MXFP4 terms.  These tests pin:
  * the records, bit for bit, against a float32 restatement of the split (scale = smallest power
    of two with no element above 6, E2M1 round-to-nearest-even, residual carried to the next
    term), and their decoded sum against the input;
  * the GLU activations the gate/up kernel writes as records, decoded by the oracle's MXFP4
    decoder, against the oracle's SiLU(G z) * (U z) for every routed row;
  * a layer whose MXFP4 weights use every E2M1 code and scale ramps over rows and blocks (nibble
    order, weight-row and token-row scale placement in TMEM), against the oracle;
  * the block-scaled path against the dequantizing kernels on the same layer.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from parity import REL_FRO, assert_close, device_inputs, to_np
from sparse_moe_layer_sigmoid_gb300 import configs, inputs

pytestmark = pytest.mark.gpu

TERMS = 3


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    from sparse_moe_layer_sigmoid_gb300 import binding as b
    return b


# ------------------------------------------------------------------------------------------------
# float32 restatement of the three-term split (independent of the CUDA code)

def _e2m1_rne(a):
    """Codes (0..7) and values of a >= 0 rounded to the E2M1 grid, ties to the even code."""
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], dtype=np.float32)
    d = np.abs(a[..., None] - grid)
    best = d.min(-1, keepdims=True)
    cand = np.where(d == best, np.arange(8), 99)
    even = np.where(cand % 2 == 0, cand, 99).min(-1)
    code = np.where(even < 99, even, cand.min(-1))
    return code.astype(np.uint8), grid[code]


def split_reference(v):
    """v float32 [rows, K] -> (nibbles [3, rows, K] uint8, scale bytes [3, rows, K/32] uint8)."""
    rows, K = v.shape
    r = v.reshape(rows, K // 32, 32).astype(np.float32).copy()
    nib = np.zeros((TERMS, rows, K // 32, 32), np.uint8)
    sc = np.zeros((TERMS, rows, K // 32), np.uint8)
    for t in range(TERMS):
        amax = np.abs(r).max(-1)
        bits = amax.view(np.uint32)
        e = ((bits >> 23) & 0xFF).astype(np.int64) - 2 + ((bits & 0x7FFFFF) > 0x400000)
        e = np.clip(e, 1, 253)
        s = (e.astype(np.uint32) << 23).view(np.float32)[..., None]
        inv = ((254 - e).astype(np.uint32) << 23).view(np.float32)[..., None]
        code, val = _e2m1_rne(np.abs(r) * inv)
        neg = (r < 0) & (code != 0)
        nib[t] = code | np.where(neg, 8, 0).astype(np.uint8)
        sc[t] = e
        r = (r - np.where(neg, -val, val).astype(np.float32) * s).astype(np.float32)
    return nib.reshape(TERMS, rows, K), sc


def records_split(rec, K):
    """Records [rows, 3K/2 + 3K/32] -> packed [3, rows, K/2], scales [3, rows, K/32]."""
    packed = np.stack([rec[:, t * K // 2:(t + 1) * K // 2] for t in range(TERMS)])
    off = TERMS * K // 2
    scales = np.stack([rec[:, off + t * K // 32:off + (t + 1) * K // 32] for t in range(TERMS)])
    return packed, scales


def records_value(rec, K):
    """fp64 value of each record row: the sum of its three terms (the oracle's MXFP4 decoder)."""
    packed, scales = records_split(rec, K)
    return sum(oracle.mxfp4_decode(packed[t], scales[t]) for t in range(TERMS))


def test_three_term_records_are_bit_exact_and_close(binding):
    K, rows = 1024, 48
    rng = np.random.default_rng(5)
    v = rng.standard_normal((rows, K)).astype(np.float32)
    v[1] = 0.0                                             # all-zero row: every code 0
    v[2] *= 1e-6                                           # fp16 subnormals
    v[3] = np.clip(v[3] * 2e4, -6e4, 6e4)                  # near the fp16 limit
    grid = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5], dtype=np.float32)
    v[4] = np.resize(grid, K) * np.repeat(2.0 ** np.arange(-4, 4), K // 8)   # E2M1 midpoints: ties
    v[5, ::2] = -v[5, 1::2]                                # sign alternation within each byte
    v[6] = 0.0
    v[6, 7::64] = 3.0                                      # one-hot blocks
    x = torch.from_numpy(v).half()
    want_nib, want_sc = split_reference(x.float().numpy())
    dev = torch.device("cuda")
    for dtype in (torch.float16, torch.bfloat16):
        xd = x.to(dtype).to(dev)
        if dtype == torch.bfloat16:
            want_nib, want_sc = split_reference(xd.float().cpu().numpy())
        rec = binding.mx3_quantize(xd).cpu().numpy()
        packed, scales = records_split(rec, K)
        nib = np.empty((TERMS, rows, K), np.uint8)
        nib[..., 0::2] = packed & 0x0F                     # element 2i: the low nibble
        nib[..., 1::2] = packed >> 4
        assert np.array_equal(scales, want_sc), dtype
        assert np.array_equal(nib, want_nib), dtype
        got = records_value(rec, K)
        ref = xd.float().cpu().double().numpy()
        err = np.abs(got - ref)
        s3 = np.repeat(oracle.e8m0_value(scales[TERMS - 1]), 32, axis=-1)
        assert np.all(err <= s3), "the last term leaves at most one step of its own grid"
        nz = np.linalg.norm(ref, axis=1) > 0
        rel = np.linalg.norm(got[nz] - ref[nz]) / np.linalg.norm(ref[nz])
        assert rel < 5e-3, rel
        assert np.all(got[1] == 0) and np.all(got[6][ref[6] == 0] == 0)


def test_glu_records_match_oracle_activations(binding):
    """Every routed row's GLU activations, as written by the gate/up kernel, against SiLU(G z) * (U z)
    from the oracle's z and decoded weights."""
    cfg = replace(configs.K3W_E128_BF16_PREFILL, name="mx_glu", tokens=200, d=512, latent=512, hidden=1024,
                  experts=12, top_k=3, n_shared=1, shared_hidden=256, routed_w="mxfp4", seed=51)
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, False)
    layer = binding.LatentMoE(cfg)
    r = layer.route(inp["x"], inp)
    layer.forward(inp["x"], inp)
    assert layer.status() == 0
    rows = cfg.tokens * cfg.top_k
    h = cfg.hidden
    rec = layer.debug_buffer("act", torch.uint8, (rows, TERMS * h // 2 + TERMS * h // 32)).cpu().numpy()
    a_gpu = records_value(rec, h)
    host = inputs.host_inputs(inp)
    ref = oracle.layer_forward(host, cfg)
    offsets = r["offsets"].cpu().numpy()
    tok = r["tok_of_row"].cpu().numpy()
    a_ref = np.empty_like(a_gpu)
    for e in range(cfg.experts):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        gu = oracle.mxfp4_decode(host["routed_gate_up"][e], host["routed_gate_up_scale"][e])
        z = ref["z"][tok[lo:hi]]
        a_ref[lo:hi] = oracle.silu(z @ gu[:h].T) * (z @ gu[h:].T)
    # SiLU(g) * u is heavy-tailed (products of two near-normal values): the largest elements carry
    # the largest rounding, so the element bound is taken against the rms of the tail's scale
    r = np.linalg.norm(a_gpu - a_ref) / np.linalg.norm(a_ref)
    m = np.abs(a_gpu - a_ref).max() / np.sqrt(np.mean(a_ref ** 2))
    print(f"GLU activations: rel_fro={r:.3e} max/rms={m:.3e}")
    assert r <= REL_FRO["mxfp4"], r
    assert m <= 0.1, m
    layer.close()


def _structured_mxfp4(e_count, rows, K, salt):
    """E2M1 bytes whose nibbles cycle through all 16 codes in an order that differs between the
    low and high nibble, and scale bytes ramping over rows and blocks (2^-8 .. 2^-4, so that a
    row's values keep the magnitude of N(0, 1/K) weights)."""
    f = np.arange(rows)[:, None]
    c = np.arange(K)[None, :]
    nib = ((f * 7 + c * 3 + salt) % 16).astype(np.uint8)
    nib[(f % 5 == 0).repeat(K, 1) & (c % 11 != (f % 11))] = 0   # every 5th row one-hot per 11
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    blk = np.arange(K // 32)[None, :]
    scales = (119 + (f + 3 * blk + salt) % 5).astype(np.uint8)
    return (np.broadcast_to(packed, (e_count, rows, K // 2)).copy(),
            np.broadcast_to(scales, (e_count, rows, K // 32)).copy())


def test_structured_mxfp4_weights_match_oracle(binding):
    cfg = replace(configs.K3W_E128_BF16_PREFILL, name="mx_struct", tokens=300, d=512, latent=512, hidden=512,
                  experts=8, top_k=2, n_shared=1, shared_hidden=256, routed_w="mxfp4", bias="normal1.5", seed=52)
    host_inp = inputs.make_inputs(cfg, "cpu")
    gu, gus = _structured_mxfp4(cfg.experts, 2 * cfg.hidden, cfg.latent, 1)
    dn, dns = _structured_mxfp4(cfg.experts, cfg.latent, cfg.hidden, 5)
    for e in range(cfg.experts):  # experts differ: rotate rows
        gu[e], gus[e] = np.roll(gu[e], 3 * e, axis=0), np.roll(gus[e], 3 * e, axis=0)
        dn[e], dns[e] = np.roll(dn[e], 5 * e, axis=0), np.roll(dns[e], 5 * e, axis=0)
    host_inp["routed_gate_up"], host_inp["routed_gate_up_scale"] = torch.from_numpy(gu), torch.from_numpy(gus)
    host_inp["routed_down"], host_inp["routed_down_scale"] = torch.from_numpy(dn), torch.from_numpy(dns)
    dev = torch.device("cuda")
    inp = {k: (None if v is None else v.to(dev)) for k, v in host_inp.items()}
    ref = oracle.layer_forward(inputs.host_inputs(host_inp), cfg)
    layer = binding.LatentMoE(cfg)
    idx = torch.from_numpy(ref["idx"].astype(np.int32)).to(dev)
    p = torch.from_numpy(ref["p"].astype(np.float32)).to(dev)
    y = layer.forward_routed(inp["x"], inp, idx, p)
    assert layer.status() == 0
    assert_close(to_np(y), ref["y"], REL_FRO["mxfp4"], "structured MXFP4 weights")
    layer.close()


@pytest.mark.parametrize("tokens", [40, 700], ids=["decode", "prefill"])
def test_block_scaled_path_matches_dequantizing_path(binding, tokens):
    cfg = replace(configs.K3W_E128_BF16_PREFILL, name="mx_vs_deq", tokens=tokens, d=512, latent=512, hidden=512,
                  experts=24, top_k=4, n_shared=1, shared_hidden=256, routed_w="mxfp4", seed=53)
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, False)
    mx = binding.LatentMoE(cfg)
    deq = binding.LatentMoE(cfg, flags=binding.LMOE_FLAG_MXFP4_DEQUANT)
    y_mx = mx.forward(inp["x"], inp)
    y_deq = deq.forward(inp["x"], inp)
    assert mx.status() == 0 and deq.status() == 0
    assert_close(to_np(y_mx), to_np(y_deq).astype(np.float64), REL_FRO["mxfp4"], "block-scaled vs dequantized")
    # run-to-run determinism of the block-scaled path
    assert torch.equal(mx.forward(inp["x"], inp), y_mx)
    mx.close()
    deq.close()


def test_mma_rate_microbenchmark(binding):
    """The FP4 roofline denominator: back-to-back kind::mxf4 CTA-pair MMAs against kind::f16 ones of
    the same M x N on this GPU.  A K = 64 E2M1 MMA does 4x the work of a K = 16 bf16 one; the
    measured rate ratio must lie between the two (1x: no gain, 6x: the datasheet's dense FP4:BF16)."""
    f16 = binding.mma_peak_tflops("f16")
    fp4 = binding.mma_peak_tflops("mxf4")
    print(f"kind::f16 {f16:.0f} TFLOP/s, kind::mxf4 {fp4:.0f} TFLOP/s, ratio {fp4 / f16:.2f}")
    assert 1000 < f16 < 4000
    assert 1.0 < fp4 / f16 <= 6.5
