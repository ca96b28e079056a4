"""latentmoe_route_noalloc against latentmoe_route, through the C ABI.

The no-allocation entry point serves callers that may not allocate device memory (a plugin
inside a host framework that owns all device memory, a serving loop with a fixed memory plan):
it runs the same router and dispatch with its scratch in a fixed array inside the library.
Two calls in a row with different inputs must each reproduce the handle-based route, so stale
scratch contents from the first call cannot leak into the second.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from parity import compare_routing, oracle_routing
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


def _outputs(T, k, E, dev):
    return {"idx": torch.full((T, k), -7, dtype=torch.int32, device=dev),
            "p": torch.full((T, k), -7.0, dtype=torch.float32, device=dev),
            "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
            "tok_of_row": torch.full((T * k,), -7, dtype=torch.int32, device=dev),
            "row_of": torch.full((T, k), -7, dtype=torch.int32, device=dev)}


def test_route_noalloc_matches_route_on_two_calls_in_a_row(binding):
    dev = torch.device("cuda")
    assert binding.route_noalloc_status() == binding.LMOE_OK  # set-up of this device; the word starts clear
    cases = [replace(configs.K3W_E128_BF16_PREFILL, name="na1", tokens=1000, d=512, latent=256, hidden=256,
                     seed=41),
             replace(configs.ROUTING_DISPATCH_STRESS, name="na2", tokens=777, d=512, latent=256, experts=96,
                     top_k=8, seed=42),
             # fp32 activations: the CUDA-core router GEMM instead of the tensor cores
             replace(configs.TINY_F32, name="na3", seed=43)]
    for cfg in cases:  # each call reuses the scratch the previous one filled
        inp = {k_: (None if v is None else v.to(dev)) for k_, v in inputs.make_inputs(cfg, "cpu").items()}
        layer = binding.LatentMoE(cfg)
        want = layer.route(inp["x"], inp)
        got = _outputs(cfg.tokens, cfg.top_k, cfg.experts, dev)
        assert binding.route_noalloc(cfg, inp["x"], inp, got) == binding.LMOE_OK
        assert binding.route_noalloc_status() == binding.LMOE_OK
        for key in ("idx", "offsets", "tok_of_row", "row_of"):
            assert torch.equal(got[key], want[key]), (cfg.name, key)
        torch.testing.assert_close(got["p"], want["p"], rtol=1e-6, atol=0)
        layer.close()


def test_route_noalloc_bf16_router_width_the_handle_refuses(binding):
    """d = 320 with a bf16 W_r: the no-allocation route needs d % 64 == 0 only (the handle needs
    d % 256 == 0 for its other GEMMs), so it is checked against the oracle instead: rank order
    bit-exact except near ties, dispatch bit-exact.  Two calls in a row with different inputs."""
    dev = torch.device("cuda")
    for seed in (44, 45):
        cfg = replace(configs.K3W_E128_BF16_PREFILL, name="na_d320", tokens=300, d=320, latent=256, hidden=256,
                      experts=36, top_k=6, bias="normal0.05", seed=seed)
        host_inp = inputs.make_inputs(cfg, "cpu")
        inp = {k_: (None if v is None else v.to(dev)) for k_, v in host_inp.items()}
        got = _outputs(cfg.tokens, cfg.top_k, cfg.experts, dev)
        assert binding.route_noalloc(cfg, inp["x"], inp, got) == binding.LMOE_OK
        assert binding.route_noalloc_status() == binding.LMOE_OK
        ref = oracle_routing(inputs.host_inputs(host_inp), cfg)
        idx = got["idx"].cpu().numpy()
        mism, _ = compare_routing(idx, ref)
        assert np.allclose(got["p"].cpu().numpy()[~mism], ref["p"][~mism], rtol=1e-4, atol=1e-7)
        _, offsets, tok_of_row, row_of = oracle.dispatch(idx.astype(np.int64), cfg.experts)
        assert np.array_equal(got["offsets"].cpu().numpy(), offsets)
        assert np.array_equal(got["tok_of_row"].cpu().numpy(), tok_of_row)
        assert np.array_equal(got["row_of"].cpu().numpy(), row_of)


def test_route_noalloc_rejects_sizes_beyond_its_scratch(binding):
    cfg = replace(configs.ROUTING_DISPATCH_STRESS, name="na_big", tokens=5000, d=512, latent=256)
    dev = torch.device("cuda")
    x = torch.zeros((cfg.tokens, cfg.d), dtype=torch.bfloat16, device=dev)
    w = {"w_router": torch.zeros((cfg.experts, cfg.d), dtype=torch.float32, device=dev)}
    out = _outputs(cfg.tokens, cfg.top_k, cfg.experts, dev)
    assert binding.route_noalloc(cfg, x, w, out) == binding.LMOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(out["idx"][0, 0]) == -7  # nothing was launched
