"""Expert-parallel dispatch and combine emulated on one GPU (latentmoe_ep_emulate): the rows
travel pack -> exchange -> return -> combine and must reach the same u as the single-GPU path,
with the per-rank-pair row counts of the routing."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from parity import device_inputs
from sparse_moe_layer_sigmoid_gb300 import configs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    from sparse_moe_layer_sigmoid_gb300 import binding as b
    return b


def _cells(idx: np.ndarray, T: int, E: int, R: int) -> np.ndarray:
    """Rows sent from rank src (owner of the token) to rank dst (owner of the expert)."""
    src = np.repeat(np.arange(T) // (T // R), idx.shape[1])
    dst = idx.reshape(-1) // (E // R)
    out = np.zeros((R, R), dtype=np.int64)
    np.add.at(out, (src, dst), 1)
    return out


IDENTITY = replace(configs.ROUTING_DISPATCH_STRESS, name="ep_identity", tokens=512, d=512, latent=256, experts=64,
                   top_k=8, seed=51)


@pytest.mark.parametrize("ranks", [1, 4, 8, 64])
def test_latent_rows_round_trip_to_the_layer_output(binding, ranks):
    """Identity experts: u = sum_j p_j z_t, the layer's own output, bit for bit (the same rows
    summed in rank order with the same p)."""
    cfg = IDENTITY
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, False)
    layer = binding.LatentMoE(cfg)
    u_ref = layer.forward(inp["x"], inp).clone()
    u, cells = layer.ep_emulate(inp["x"], inp, ranks, False)
    r = layer.route(inp["x"], inp)
    assert layer.status() == 0
    assert torch.equal(u, u_ref)
    idx = r["idx"].cpu().numpy()
    assert np.array_equal(cells.cpu().numpy(), _cells(idx, cfg.tokens, cfg.experts, ranks))
    layer.close()


def test_full_width_rows_and_mxfp4_latent_rows(binding):
    """Full width: the rows are x itself, so u = x * sum_j p_j = x up to the bf16 rounding of the
    p-weighted sum.  With MXFP4 experts the latent rows are fp16 z; u matches sum_j p_j z_t."""
    cfg = replace(configs.K3_MXFP4_DECODE, name="ep_mx", tokens=96, d=512, latent=512, hidden=512, experts=32,
                  top_k=4, n_shared=1, shared_hidden=256, seed=52)
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, False)
    layer = binding.LatentMoE(cfg)
    R = 4
    u_full, cells_full = layer.ep_emulate(inp["x"], inp, R, True)
    u_lat, cells_lat = layer.ep_emulate(inp["x"], inp, R, False)
    r = layer.route(inp["x"], inp)
    assert layer.status() == 0
    x = inp["x"].float()
    assert (u_full.float() - x).abs().max().item() <= 2.0 ** -7 * x.abs().max().item()
    assert torch.equal(cells_full, cells_lat)
    assert np.array_equal(cells_lat.cpu().numpy(), _cells(r["idx"].cpu().numpy(), cfg.tokens, cfg.experts, R))
    # z of the last call is in the handle's workspace: u = sum_j p_j z (fp32 sum, bf16 out)
    z = layer.debug_buffer("z", torch.float16, (cfg.tokens, cfg.latent)).float()
    p = r["p"].float()
    ref = z * p.sum(dim=1, keepdim=True)
    assert (u_lat.float() - ref).abs().max().item() <= 2.0 ** -7 * ref.abs().max().item() + 1e-6
    with pytest.raises(binding.LatentMoEError):
        layer.ep_emulate(inp["x"], inp, 5, False)  # 32 experts do not split over 5 ranks
    layer.close()
