"""latentmoe_route_noalloc against latentmoe_route, through the C ABI.

The no-allocation entry point serves callers that may not allocate device memory (a plugin
inside a host framework that owns all device memory, a serving loop with a fixed memory plan):
it runs the same router and dispatch with its scratch in a fixed array inside the library.
Two calls in a row with different inputs must each reproduce the handle-based route, so stale
scratch contents from the first call cannot leak into the second.
"""
from dataclasses import replace

import pytest
import torch

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
    cases = [replace(configs.K3W_E128_BF16_PREFILL, name="na1", tokens=1000, d=512, latent=256, hidden=256,
                     seed=41),
             replace(configs.ROUTING_DISPATCH_STRESS, name="na2", tokens=777, d=512, latent=256, experts=96,
                     top_k=8, seed=42)]
    for cfg in cases:  # the second call reuses the scratch the first one filled
        inp = {k_: (None if v is None else v.to(dev)) for k_, v in inputs.make_inputs(cfg, "cpu").items()}
        layer = binding.LatentMoE(cfg)
        want = layer.route(inp["x"], inp)
        got = _outputs(cfg.tokens, cfg.top_k, cfg.experts, dev)
        assert binding.route_noalloc(cfg, inp["x"], inp, got) == binding.LMOE_OK
        torch.cuda.synchronize()
        for key in ("idx", "offsets", "tok_of_row", "row_of"):
            assert torch.equal(got[key], want[key]), (cfg.name, key)
        torch.testing.assert_close(got["p"], want["p"], rtol=1e-6, atol=0)
        layer.close()


def test_route_noalloc_rejects_sizes_beyond_its_scratch(binding):
    cfg = replace(configs.ROUTING_DISPATCH_STRESS, name="na_big", tokens=5000, d=512, latent=256)
    dev = torch.device("cuda")
    x = torch.zeros((cfg.tokens, cfg.d), dtype=torch.bfloat16, device=dev)
    w = {"w_router": torch.zeros((cfg.experts, cfg.d), dtype=torch.float32, device=dev)}
    out = _outputs(cfg.tokens, cfg.top_k, cfg.experts, dev)
    assert binding.route_noalloc(cfg, x, w, out) == binding.LMOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(out["idx"][0, 0]) == -7  # nothing was launched
