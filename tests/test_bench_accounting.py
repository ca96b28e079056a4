"""bench.py's algorithmic work per stage (the roofline numerators) against figures the pages print.

"Lesson 6 - LatentMoE", section "Deriving the headline number", gives the parameter counts of
one routed expert (33.0M), of the W_down/W_up projections (4.7B over 92 layers) and of the shared
experts (12.2B over 92 layers).  A forward pass does 2 FLOP per parameter it applies, so the
per-token work that bench.py divides by its stage times must match those counts to the pages'
rounding; the MXFP4 byte count of one expert follows from the same parameter count (half a
byte per value plus one scale byte per 32).
"""
import json
import os

import pytest

import bench
from sparse_moe_layer_sigmoid_gb300 import configs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_arithmetic.json")


@pytest.fixture(scope="module")
def pages():
    with open(GOLDEN) as f:
        return json.load(f)


def _per_token(work, keys, T):
    return sum(work[k][1] for k in keys) / T


def test_routed_flops_per_token_match_expert_size(pages):
    cfg = configs.K3W_E128_BF16_PREFILL
    work = bench.stage_work(cfg, cfg.experts)
    assert work["routed_gate_up_glu"][0] == "tensor" and work["routed_down"][0] == "tensor"
    routed = _per_token(work, ("routed_gate_up_glu", "routed_down"), cfg.tokens)
    per_expert = pages["params_per_routed_expert"]
    want = 2 * cfg.top_k * per_expert["value"]
    assert abs(routed - want) <= 2 * cfg.top_k * per_expert["rounding"]
    # the 92-layer activated-routed figure pins k and the expert size together
    act = pages["activated_routed_all_layers"]
    layers = pages["k3_widths"]["moe_layers"]
    assert abs(routed / 2 * layers - act["value"]) <= act["rounding"] + layers * cfg.top_k * per_expert["rounding"]


def test_dense_flops_per_token_match_projection_and_shared_sizes(pages):
    cfg = configs.K3W_E128_BF16_PREFILL
    work = bench.stage_work(cfg, cfg.experts)
    dense = _per_token(work, ("w_down", "shared_gate_up_glu", "final_gemm"), cfg.tokens)
    layers = pages["k3_widths"]["moe_layers"]
    proj, shared = pages["projections_all_layers"], pages["shared_experts_all_layers"]
    want = 2 * (proj["value"] + shared["value"]) / layers
    tol = 2 * (proj["rounding"] + shared["rounding"]) / layers
    assert abs(dense - want) <= tol


def test_mxfp4_expert_bytes_match_expert_size(pages):
    cfg = configs.K3_MXFP4_DECODE
    h, l = cfg.hidden, cfg.latent
    per_expert = pages["params_per_routed_expert"]
    got = bench.expert_weight_bytes(cfg, 2 * h, l) + bench.expert_weight_bytes(cfg, l, h)
    ratio = 0.5 + 1 / 32  # E2M1 value + one E8M0 byte per 32 values
    assert abs(got - ratio * per_expert["value"]) <= ratio * per_expert["rounding"]


def test_decode_stages_are_counted_in_bytes_prefill_in_flops():
    dec = configs.K3_MXFP4_DECODE
    w = bench.stage_work(dec, 399)
    assert w["routed_gate_up_glu"][0] == "hbm" and w["routed_down"][0] == "hbm"
    # 399 touched experts stream their gate/up bytes at least once
    assert w["routed_gate_up_glu"][1] >= 399 * bench.expert_weight_bytes(dec, 2 * dec.hidden, dec.latent)
    pre = configs.K3_MXFP4_PREFILL_SKEW
    assert bench.stage_work(pre, 34)["routed_gate_up_glu"][0] == "tensor"
