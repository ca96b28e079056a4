"""MXFP8 activations on tcgen05.mma kind::mxf8f6f4 (LMOE_FLAG_MXFP8_ACT).

K3 is trained with MXFP4 weights and MXFP8 activations (page "What K3 actually is",
srikanthmalla.com, the quantization-aware training passage).  In this mode the expert inputs and
the GLU activations become MXFP8 records and the expert GEMMs multiply E2M1 weights by E4M3
activations.  These tests pin:
  * the records, value for value, against the oracle's MXFP8 encoder (RNE on the E4M3 grid, the
    smallest power-of-two block scale keeping every element within 448);
  * the layer against the oracle run with the same activation quantisation
    (layer_forward(act_quant="mxfp8")) on prefill tiles, decode units and sampled rows of the full
    skewed K3 prefill; the distance to the unquantised oracle is printed beside it.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from parity import REL_FRO, assert_close, device_inputs, oracle_for_rows, to_np
from sparse_moe_layer_sigmoid_gb300 import configs, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    from sparse_moe_layer_sigmoid_gb300 import binding as b
    return b


def _decode_records(rec: np.ndarray, K: int) -> np.ndarray:
    codes = rec[:, :K]
    scales = rec[:, K:K + K // 32]
    return oracle.e4m3_value(codes) * np.repeat(oracle.e8m0_value(scales), 32, axis=1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_mxfp8_records_match_oracle_encoder(binding, dtype):
    g = torch.Generator().manual_seed(3)
    rows, K = 96, 1024
    x = torch.randn((rows, K), generator=g) * torch.logspace(-3, 3, rows).unsqueeze(1)
    x[5] = 0.0                      # an all-zero row: zero codes
    x[7, :32] = 448.0 * 2.0 ** -20  # a block whose maximum sits exactly on a scale boundary
    x[8, 64:96] = -1e-30             # tiny values: the scale clamps
    xd = x.to(dtype).cuda()
    rec = binding.mx8_quantize(xd).cpu().numpy()
    got = _decode_records(rec, K)
    want = oracle.mxfp8_quantize(xd.float().cpu().double().numpy())
    assert np.array_equal(got, want), float(np.nanmax(np.abs(got - want)))
    assert not np.any(rec[:, :K] == 0x80)  # no negative zero codes


# Per-element bound in this mode.  The GPU quantises its fp16 z and fp32 GLU activations, the
# oracle its fp64 ones: where a value sits within their difference (~1e-3 relative) of an E4M3
# rounding boundary the two land one code apart, a step of up to 2^-3 of the value, and a step
# in a large GLU activation moves every output of its row.  The Frobenius bound stays the
# MXFP4 tolerance.
MXFP8_MAX_ERR_RMS = 0.25

MXFP8_SMALL = [
    replace(configs.K3_MXFP4_PREFILL_SKEW, name="mxfp8_prefill_tiles", tokens=700, d=512, latent=512, hidden=1024,
            experts=24, top_k=4, n_shared=1, shared_hidden=256, seed=61),
    replace(configs.K3_MXFP4_DECODE, name="mxfp8_decode_units", tokens=40, d=512, latent=512, hidden=512,
            experts=24, top_k=4, n_shared=1, shared_hidden=256, seed=62),
]


def _mxfp8_check(b, cfg, sample=None, on_device=False):
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, on_device)
    layer = b.LatentMoE(cfg, flags=b.LMOE_FLAG_MXFP8_ACT)
    r = layer.route(inp["x"], inp)
    y = layer.forward(inp["x"], inp)
    assert layer.status() == 0
    rows = inputs.sample_tokens(cfg.tokens, sample or cfg.tokens, cfg.seed)
    idx = r["idx"].cpu().numpy()[rows]
    p = r["p"].cpu().numpy()[rows]
    host = inputs.host_inputs(inp, lazy_experts=True)
    # the GPU's routing (equal to the oracle's; tested elsewhere) for both oracle evaluations
    want = oracle.layer_forward(host, cfg, tokens=rows, routing=(idx, p), act_quant="mxfp8")["y"]
    plain = oracle.layer_forward(host, cfg, tokens=rows, routing=(idx, p))["y"]
    got = to_np(y)[rows]
    rel = float(np.linalg.norm(got - want) / np.linalg.norm(want))
    mx = float(np.abs(got - want).max() / np.sqrt(np.mean(want * want)))
    assert rel <= REL_FRO["mxfp4"], f"{cfg.name}: relative Frobenius error {rel:.3e} vs the oracle's MXFP8 mode"
    assert mx <= MXFP8_MAX_ERR_RMS, f"{cfg.name}: max element error {mx:.3e} x rms"
    rel_plain = float(np.linalg.norm(got - plain) / np.linalg.norm(plain))
    oracle_gap = float(np.linalg.norm(want - plain) / np.linalg.norm(plain))
    print(f"{cfg.name}: rel_fro={rel:.3e} max/rms={mx:.3e}; vs the unquantised oracle {rel_plain:.3e} "
          f"(the oracle's own MXFP8 mode is {oracle_gap:.3e} from it)")
    layer.close()
    return rel


@pytest.mark.parametrize("cfg", MXFP8_SMALL, ids=lambda c: c.name)
def test_mxfp8_layer_matches_oracle_mxfp8_mode(binding, cfg):
    _mxfp8_check(binding, cfg)


def test_mxfp8_k3_prefill_skew_sampled_rows(binding):
    _mxfp8_check(binding, configs.K3_MXFP4_PREFILL_SKEW, sample=24, on_device=True)
