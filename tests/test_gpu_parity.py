"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded inputs."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from parity import (REL_FRO, assert_close, check_dispatch, compare_routing, device_inputs, oracle_for_rows,
                    oracle_routing, to_np)
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


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


# Reduced-width bf16 layers with K3's structure: several tiles in every GEMM dimension and
# ragged per-expert row counts.
SMALL_BF16 = replace(configs.K3W_E128_BF16_PREFILL, name="small_bf16", tokens=300, d=512, latent=256, hidden=256,
                     experts=16, top_k=4, n_shared=2, shared_hidden=256, seed=21)
SMALL_CASES = [
    configs.TINY_F32,
    SMALL_BF16,
    replace(SMALL_BF16, name="small_bf16_noshared", n_shared=0, seed=22),
    replace(SMALL_BF16, name="small_bf16_skew", bias="normal1.5", tokens=777, seed=23),
    replace(SMALL_BF16, name="small_bf16_k1", top_k=1, tokens=129, seed=24),
    replace(SMALL_BF16, name="small_bf16_wide", tokens=520, d=1024, latent=512, hidden=384, experts=40, top_k=6,
            shared_hidden=384, seed=25),
    replace(configs.ROUTING_DISPATCH_STRESS, name="small_identity", tokens=1000, d=512, latent=256, experts=64,
            top_k=8, seed=26),
    replace(configs.TINY_F32, name="tiny_f32_skew_ragged", tokens=301, bias="normal1.5", seed=27),
    replace(SMALL_BF16, name="small_mxfp4", routed_w="mxfp4", latent=512, hidden=512, seed=28),
    replace(SMALL_BF16, name="small_mxfp4_skew", routed_w="mxfp4", latent=512, hidden=1024, experts=24,
            bias="normal1.5", tokens=900, seed=29),
    # decode-shaped (T*k <= 32*E): the swapped-operand expert GEMMs
    replace(SMALL_BF16, name="small_bf16_decode", tokens=24, seed=36),
    replace(SMALL_BF16, name="small_bf16_decode_skew", tokens=150, top_k=2, bias="normal1.5", seed=37),
    replace(SMALL_BF16, name="small_mxfp4_decode", routed_w="mxfp4", latent=512, hidden=512, experts=24, tokens=40,
            seed=38),
    # >= 256 rows per expert on average: routed GEMMs on CTA pairs (256-row tiles), ragged counts
    replace(SMALL_BF16, name="small_bf16_pair_skew", tokens=700, experts=8, bias="normal1.5", seed=39),
    replace(SMALL_BF16, name="small_bf16_pair_wide", tokens=600, d=1024, latent=512, hidden=384, experts=4,
            top_k=2, n_shared=1, shared_hidden=384, seed=40),
]


def _run_and_check(b, cfg, on_device=False, sample=None, full_routing=False):
    """Route and forward through the C ABI and compare with the oracle on the sampled rows (all rows
    when ``sample`` is None): routing in rank order, p, dispatch, per-stage intermediates and the
    output.  With ``full_routing`` the routing of every token is compared as well."""
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, on_device)
    layer = b.LatentMoE(cfg)
    x = inp["x"]
    r = layer.route(x, inp)
    stats = layer.routing_stats()
    y = layer.forward(x, inp)
    assert layer.status() == 0
    n_launch = layer.last_launch_count()
    assert n_launch >= 7
    T = cfg.tokens
    rows = inputs.sample_tokens(T, sample or T, cfg.seed)
    ref, host = oracle_for_rows(inp, cfg, rows)
    idx_gpu = r["idx"].cpu().numpy()
    p_gpu = r["p"].cpu().numpy()
    mism, near = compare_routing(idx_gpu[rows], ref)
    if rows.size == T:  # the GPU's count of near ties is the oracle's
        assert stats["near_ties"] == near, (stats, near)
    if full_routing and rows.size < T:
        full = oracle_routing(host, cfg)
        mism_all, near_all = compare_routing(idx_gpu, full)
        assert stats["near_ties"] == near_all, (stats, near_all)
        ok_all = ~mism_all
        assert np.allclose(p_gpu[ok_all], full["p"][ok_all], rtol=1e-4, atol=1e-7)
        near = near_all
    counts = check_dispatch(r, idx_gpu, cfg.experts)
    ok = ~mism
    # p: fp32 from logits accurate to the router margin -> relative error well below 1e-4
    assert np.allclose(p_gpu[rows][ok], ref["p"][ok], rtol=1e-4, atol=1e-7)
    # per-stage intermediates of the last forward, against the oracle on the same rows
    logits = to_np(layer.debug_buffer("logits", torch.float32, (T, cfg.experts)))[rows]
    want_l = oracle.router_logits(oracle.widen(host["x"][rows]), oracle.widen(host["w_router"]))
    l_err = float(np.abs(logits - want_l).max())
    assert l_err < 0.25e-3, f"router logit error {l_err:.3e} above a quarter of the refinement margin"
    z_dtype = torch.float16 if cfg.routed_w == "mxfp4" and not cfg.identity_experts else x.dtype
    z = to_np(layer.debug_buffer("z", z_dtype, (T, cfg.latent)))[rows]
    assert_close(z, ref["z"], REL_FRO[cfg.act], cfg.name + " z")
    if not cfg.identity_experts:
        kcat = cfg.n_shared * cfg.shared_hidden + cfg.latent
        n_gpu = to_np(layer.debug_buffer("act_cat", x.dtype, (T, kcat)))[rows][:, kcat - cfg.latent:]
        n_ok = ~mism
        assert_close(n_gpu[n_ok], ref["n"][n_ok], REL_FRO[cfg.routed_w], cfg.name + " RMSNorm(u)")
    key = "u" if cfg.identity_experts else "y"
    want = ref[key].copy()
    if mism.any():  # near-tie tokens: compare against the oracle under the GPU's own choice
        sub = rows[mism]
        s_sel = np.take_along_axis(ref["s"][mism], idx_gpu[sub].astype(np.int64), axis=1)
        ref2 = oracle.layer_forward(host, cfg, tokens=sub, routing=(idx_gpu[sub], s_sel / s_sel.sum(1, keepdims=True)))
        want[mism] = ref2[key]
    got = to_np(y)[rows]
    rel, mx = assert_close(got, want, REL_FRO[cfg.routed_w if not cfg.identity_experts else cfg.act], cfg.name)
    layer.close()
    return {"rel": rel, "max": mx, "near_ties": near, "refined": stats["refined_tokens"], "counts": counts, "y": y,
            "inp": inp, "logit_err": l_err}


@pytest.mark.parametrize("cfg", SMALL_CASES, ids=lambda c: c.name)
def test_small_layers_match_oracle(binding, cfg):
    res = _run_and_check(binding, cfg)
    print(f"{cfg.name}: rel_fro={res['rel']:.3e} max/rms={res['max']:.3e} near_ties={res['near_ties']} "
          f"logit_err={res['logit_err']:.2e}")


def _report(cfg, res, extra=""):
    c = res["counts"]
    print(f"{cfg.name}: rel_fro={res['rel']:.3e} max/rms={res['max']:.3e} near_ties={res['near_ties']} "
          f"refined={res['refined']} experts touched={int((c > 0).sum())} load max/mean={c.max() / c.mean():.2f} "
          f"logit_err={res['logit_err']:.2e}{extra}")


def test_k3w_e128_bf16_prefill_sampled_rows(binding):
    cfg = configs.K3W_E128_BF16_PREFILL
    res = _run_and_check(binding, cfg, on_device=True, sample=256, full_routing=True)
    _report(cfg, res)
    del res
    _free()


def test_k3_mxfp4_decode_all_rows(binding):
    cfg = configs.K3_MXFP4_DECODE
    res = _run_and_check(binding, cfg, on_device=True)
    _report(cfg, res)
    del res
    _free()


def test_k3_mxfp4_prefill_skew_sampled_rows(binding):
    cfg = configs.K3_MXFP4_PREFILL_SKEW
    res = _run_and_check(binding, cfg, on_device=True, sample=256, full_routing=True)
    _report(cfg, res)
    del res
    _free()


def test_k3_mxfp4_prefill_mild_sampled_rows(binding):
    """The 2-10x skew variant: about 840 experts touched with ~150 rows each.  The oracle decodes
    every expert a sampled row selects, so 32 rows (about 400 experts) are compared on the output;
    the routing of all 8192 tokens is compared in full."""
    cfg = configs.K3_MXFP4_PREFILL_MILD
    res = _run_and_check(binding, cfg, on_device=True, sample=32, full_routing=True)
    _report(cfg, res)
    del res
    _free()


def test_routing_dispatch_stress_sampled_rows(binding):
    cfg = configs.ROUTING_DISPATCH_STRESS
    res = _run_and_check(binding, cfg, on_device=True, sample=256, full_routing=True)
    _report(cfg, res)
    assert res["counts"].sum() == cfg.tokens * cfg.top_k
    del res
    _free()


def test_token_permutation_is_bitwise_invariant(binding):
    cfg = replace(SMALL_BF16, name="perm", tokens=333, seed=31)
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, False)
    layer = binding.LatentMoE(cfg)
    y = layer.forward(inp["x"], inp).clone()
    perm = torch.randperm(cfg.tokens, generator=torch.Generator().manual_seed(5)).to(dev)
    y2 = layer.forward(inp["x"][perm].contiguous(), inp)
    assert layer.status() == 0
    assert torch.equal(y2, y[perm])
    y3 = layer.forward(inp["x"], inp)
    assert torch.equal(y3, y)  # run-to-run determinism
    layer.close()


@pytest.mark.parametrize("cfg", [replace(SMALL_BF16, name="fork_prefill", tokens=520, seed=42),
                                 replace(SMALL_BF16, name="fork_decode_mx", routed_w="mxfp4", latent=512,
                                         hidden=512, experts=24, tokens=40, seed=43),
                                 replace(configs.ROUTING_DISPATCH_STRESS, name="fork_identity", tokens=700, d=512,
                                         latent=256, experts=64, top_k=8, seed=44)],
                         ids=lambda c: c.name)
def test_second_stream_matches_one_stream(binding, cfg):
    """W_down and the shared GLU run on the handle's second stream unless stages are timed (then
    every stage runs on the caller's stream in order): the same kernels on the same inputs, so
    the outputs are bitwise equal; a call on a side stream is ordered after earlier work there."""
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, False)
    layer = binding.LatentMoE(cfg)
    y_fork = layer.forward(inp["x"], inp).clone()
    layer.enable_stage_timing()
    y_serial = layer.forward(inp["x"], inp).clone()
    layer.disable_stage_timing()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        x2 = inp["x"] * 1  # produced on the side stream just before the call
        y_side = layer.forward(x2, inp, stream=side)
    side.synchronize()
    assert layer.status() == 0
    assert torch.equal(y_fork, y_serial)
    assert torch.equal(y_side, y_fork)
    layer.close()


@pytest.mark.parametrize("cfg", [replace(SMALL_BF16, name="graph_decode_mx", routed_w="mxfp4", latent=512,
                                         hidden=512, experts=24, tokens=40, seed=45),
                                 replace(SMALL_BF16, name="graph_prefill", tokens=300, seed=46)],
                         ids=lambda c: c.name)
def test_forward_captured_in_a_cuda_graph(binding, cfg):
    """The forward (every launch, the second stream's fork and joins) captures into one CUDA
    graph; replays compute what stream launches compute, bit for bit, for new contents of x."""
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, False)
    layer = binding.LatentMoE(cfg)
    x = inp["x"].clone()
    y = torch.empty((cfg.tokens, layer.out_width), dtype=x.dtype, device=dev)
    layer.forward(x, inp, y)  # one-time setup outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        layer.forward(x, inp, y, stream=torch.cuda.current_stream())
    for seed in (1, 2):
        x.copy_(torch.randn(x.shape, generator=torch.Generator().manual_seed(seed)).to(x.dtype).to(dev))
        g.replay()
        torch.cuda.synchronize()
        y_graph = y.clone()
        y_stream = layer.forward(x, inp)
        assert layer.status() == 0
        assert torch.equal(y_graph, y_stream)
    del g
    layer.close()


@pytest.mark.parametrize("cfg", [SMALL_BF16, replace(SMALL_BF16, name="pair_grouped", tokens=700, experts=8,
                                                      bias="normal1.5", seed=41)], ids=lambda c: c.name)
def test_cta_pair_gemms_match_single_cta(binding, cfg):
    """CTA-pair GEMMs and single-CTA GEMMs accumulate in fp32 (single CTAs split K for dense GEMMs
    of few tiles, which sums in another order); the layer outputs agree up to that and to the
    bf16 rounding of intermediate values."""
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, False)
    pair = binding.LatentMoE(cfg)
    single = binding.LatentMoE(cfg, flags=binding.LMOE_FLAG_SINGLE_CTA_GEMM)
    y_pair = pair.forward(inp["x"], inp)
    y_single = single.forward(inp["x"], inp)
    assert pair.status() == 0 and single.status() == 0
    diff = (y_pair.float() - y_single.float()).abs().max().item()
    same = torch.equal(y_pair, y_single)
    print(f"{cfg.name}: bitwise equal={same} max abs diff={diff:.3e}")
    assert_close(to_np(y_pair), to_np(y_single).astype(np.float64), 1e-3, "pair vs single")
    pair.close()
    single.close()


def test_forward_routed_tile_boundary_counts(binding):
    """Caller routing that gives experts row counts at every tile boundary of the 16-, 128- and
    256-row tile lists (0, 1, 127..129, 255..257, 383..385, 512): pair tiles, their 128-row tail
    tiles and single-CTA tiles all match the oracle on every row."""
    counts = [0, 1, 127, 128, 129, 255, 256, 257, 383, 384, 385, 512, 0, 16, 17, 14]
    E, k = len(counts), 2
    T = sum(counts) // k
    cfg = replace(SMALL_BF16, name="tile_counts", tokens=T, experts=E, top_k=k, n_shared=1, seed=42)
    slots = np.repeat(np.arange(E), counts)
    assert slots.size == T * k and max(counts) <= T
    idx_np = np.stack([slots[:T], slots[T:]], axis=1).astype(np.int32)  # distinct experts per token
    assert np.all(idx_np[:, 0] != idx_np[:, 1])
    rng = np.random.default_rng(7)
    p_np = rng.uniform(0.2, 0.8, size=(T, k))
    p_np /= p_np.sum(axis=1, keepdims=True)
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, False)
    host = inputs.host_inputs(inp)
    ref = oracle.layer_forward(host, cfg, routing=(idx_np, p_np))
    for flags in (0, binding.LMOE_FLAG_SINGLE_CTA_GEMM):
        layer = binding.LatentMoE(cfg, flags=flags)
        y = layer.forward_routed(inp["x"], inp, torch.from_numpy(idx_np).to(dev),
                                 torch.from_numpy(p_np.astype(np.float32)).to(dev))
        assert layer.status() == 0
        assert_close(to_np(y), ref["y"], REL_FRO["bf16"], f"tile counts, flags={flags}")
        layer.close()


def test_forward_host_matches_device_path(binding):
    cfg = replace(SMALL_BF16, name="host", seed=32)
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, False)
    layer = binding.LatentMoE(cfg)
    y = layer.forward(inp["x"], inp)
    x_host = inp["x"].cpu().pin_memory()
    y_host = layer.forward_host(x_host, inp)
    assert torch.equal(y_host, y.cpu())
    assert layer.status() == 0
    layer.close()


def test_edge_sizes_and_errors(binding):
    cfg = replace(SMALL_BF16, name="edges", tokens=64, seed=33)
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, False)
    layer = binding.LatentMoE(cfg)
    # T = 0: nothing launched, OK
    y0 = layer.forward(inp["x"][:0], inp)
    assert y0.shape == (0, cfg.d) and layer.last_launch_count() == 0
    # T = 1 and a ragged T give the same rows as the full batch (rows are independent)
    y_full = layer.forward(inp["x"], inp).clone()
    y1 = layer.forward(inp["x"][:1].contiguous(), inp)
    assert torch.equal(y1, y_full[:1])
    y37 = layer.forward(inp["x"][:37].contiguous(), inp)
    assert torch.equal(y37, y_full[:37])
    # T above max_tokens is rejected on the host
    big = torch.zeros((cfg.tokens + 1, cfg.d), dtype=inp["x"].dtype, device=dev)
    with pytest.raises(binding.LatentMoEError) as ei:
        layer.forward(big, inp)
    assert ei.value.status == binding.LMOE_ERR_INVALID_ARG
    # missing weight pointer is rejected
    bad = dict(inp)
    bad["w_down_proj"] = None
    with pytest.raises(binding.LatentMoEError):
        layer.forward(inp["x"], bad)
    # caller-supplied routing with an out-of-range expert is flagged by the device check
    idx = torch.zeros((cfg.tokens, cfg.top_k), dtype=torch.int32, device=dev)
    idx[:] = torch.arange(cfg.top_k, dtype=torch.int32, device=dev)
    idx[3, 1] = cfg.experts + 5
    p = torch.full((cfg.tokens, cfg.top_k), 1.0 / cfg.top_k, device=dev)
    layer.forward_routed(inp["x"], inp, idx, p)
    assert layer.status() == binding.LMOE_ERR_DEVICE_CHECK
    assert layer.status() == 0  # the status word is cleared once read
    layer.close()
    # unsupported / invalid configurations are refused at create
    with pytest.raises(binding.LatentMoEError) as ei:
        binding.LatentMoE(replace(SMALL_BF16, d=500))
    assert ei.value.status == binding.LMOE_ERR_UNSUPPORTED
    with pytest.raises(binding.LatentMoEError) as ei:
        binding.LatentMoE(replace(SMALL_BF16, top_k=0))
    assert ei.value.status == binding.LMOE_ERR_INVALID_ARG


@pytest.mark.parametrize("cfg", [
    replace(SMALL_BF16, name="ties_bf16", top_k=5, seed=41),
    replace(configs.ROUTING_DISPATCH_STRESS, name="ties_f32_router_zipf", tokens=600, d=512, latent=256,
            experts=64, top_k=7, seed=42),
    replace(configs.TINY_F32, name="ties_f32_skew", tokens=200, top_k=3, bias="normal1.5", seed=43),
], ids=lambda c: c.name)
def test_exact_ties_go_to_the_lower_index(binding, cfg):
    """Experts 2j and 2j+1 get identical router rows and biases, so their keys tie exactly; with
    k odd the k-th selected expert always has its twin as the (k+1)-th, and eq. 13's tie rule
    keeps the lower index (and lists the lower index of every selected pair first).  The expected sets come from the oracle's scores of the distinct
    experts; tokens whose distinct boundary pairs are within 1e-6 of each other are skipped."""
    dev = torch.device("cuda")
    host_inp = inputs.make_inputs(cfg, "cpu")
    w = host_inp["w_router"]
    w[1::2] = w[0::2].clone()
    if host_inp["router_bias"] is not None:
        b = host_inp["router_bias"]
        b[1::2] = b[0::2].clone()
    inp = {k_: (None if v is None else v.to(dev)) for k_, v in host_inp.items()}
    layer = binding.LatentMoE(cfg)
    r = layer.route(inp["x"], inp)
    assert layer.status() == 0
    idx_gpu = r["idx"].cpu().numpy().astype(np.int64)
    p_gpu = r["p"].cpu().numpy()
    layer.close()

    host = inputs.host_inputs(host_inp)
    s_half = oracle.router_scores(oracle.widen(host["x"]), oracle.widen(host["w_router"])[0::2])
    b_half = None if host["router_bias"] is None else oracle.widen(host["router_bias"])[0::2]
    s_full = np.repeat(s_half, 2, axis=1)
    b_full = None if b_half is None else np.repeat(b_half, 2)
    k = cfg.top_k
    want, _ = oracle.select_topk(s_full, b_full, k)
    m = (k - 1) // 2  # rank of the boundary pair among the distinct experts
    _, gap_after = oracle.select_topk(s_half, b_half, m + 1)
    gap_before = oracle.select_topk(s_half, b_half, m)[1] if m > 0 else np.full(cfg.tokens, np.inf)
    clear = (gap_after >= 1e-6) & (gap_before >= 1e-6)
    assert clear.mean() > 0.99
    # the boundary expert is always the even member of its pair
    assert np.all(want[:, k - 1] % 2 == 0)
    # rank order too: each twin pair ties exactly, its lower index first
    bad = np.any(idx_gpu != want, axis=1) & clear
    assert not bad.any(), f"{int(bad.sum())} tokens differ, e.g. {np.nonzero(bad)[0][:5]}"
    p_want = oracle.route_weights(s_full, want)
    assert np.allclose(p_gpu[clear], p_want[clear], rtol=1e-4, atol=1e-7)


@pytest.mark.parametrize("tokens", [40, 600], ids=lambda t: f"T{t}")
def test_clustered_keys_take_the_bisection_fallback(binding, tokens):
    """The 128 largest keys sit four to a group of the short-batch selection's bound (expert
    e = r // 4 + 256 (r % 4) holds rank r: group e % 32 = r // 4, one CTA thread r // 4), so the
    32nd-largest group maximum, the bound, lets 125 keys through: more than its 64-entry sort,
    which hands the token to the bisection selection.  Logits are exact (one non-zero column of x
    and W_r, bf16-representable values): the selection must be the oracle's, ranks 0..31 in
    order.  T=600 runs the two-kernel path."""
    cfg = replace(configs.ROUTING_DISPATCH_STRESS, name="clustered_keys", tokens=tokens, d=512, latent=256,
                  experts=896, top_k=32, bias="none", router_w="bf16", seed=45)
    E, k = cfg.experts, cfg.top_k
    w = torch.zeros((E, cfg.d), dtype=torch.float32)
    w[:, 0] = -2.0
    for rank in range(128):
        w[(rank // 4) + 256 * (rank % 4), 0] = 4.0 - rank / 32.0
    x = torch.zeros((tokens, cfg.d), dtype=torch.float32)
    x[:, 0] = 0.5 + (torch.arange(tokens) % 64).float() / 64.0
    host_inp = {"x": x.to(torch.bfloat16), "w_router": w.to(torch.bfloat16), "router_bias": None,
                "w_down_proj": torch.zeros((cfg.latent, cfg.d), dtype=torch.bfloat16),
                "rms_gain": torch.ones(cfg.latent)}
    dev = torch.device("cuda")
    inp = {k_: (None if v is None else v.to(dev)) for k_, v in host_inp.items()}
    layer = binding.LatentMoE(cfg)
    r = layer.route(inp["x"], inp)
    assert layer.status() == 0
    idx_gpu = r["idx"].cpu().numpy().astype(np.int64)
    p_gpu = r["p"].cpu().numpy()
    layer.close()
    s = oracle.router_scores(oracle.widen(host_inp["x"].float().numpy()),
                             oracle.widen(host_inp["w_router"].float().numpy()))
    want, _ = oracle.select_topk(s, None, k)
    ranked = np.array([(rank // 4) + 256 * (rank % 4) for rank in range(k)])
    assert np.all(want == ranked[None, :])
    assert np.array_equal(idx_gpu, want)
    assert np.allclose(p_gpu, oracle.route_weights(s, want), rtol=1e-5, atol=1e-7)


def test_forward_routed_with_oracle_routing(binding):
    cfg = replace(SMALL_BF16, name="routed", seed=34)
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, False)
    host = inputs.host_inputs(inp)
    ref = oracle.layer_forward(host, cfg)
    layer = binding.LatentMoE(cfg)
    idx = torch.from_numpy(ref["idx"].astype(np.int32)).to(dev)
    p = torch.from_numpy(ref["p"].astype(np.float32)).to(dev)
    y = layer.forward_routed(inp["x"], inp, idx, p)
    assert layer.status() == 0
    assert_close(to_np(y), ref["y"], REL_FRO["bf16"], "forward_routed")
    layer.close()


@pytest.mark.parametrize("case", [
    # (name, config, flags, inject): which kernel family loses one pipeline signal
    ("pair_swap_routed", replace(SMALL_BF16, name="timeout_ps", seed=35), 0, 1),
    ("single_cta_routed", replace(SMALL_BF16, name="timeout_sc", seed=35), "single", 1),
    ("pair_dense_wdown", replace(SMALL_BF16, name="timeout_pd", seed=35), 0, 2),
    ("swap_decode_routed", replace(SMALL_BF16, name="timeout_sw", tokens=24, seed=36), 0, 1),
    ("mx_decode_routed", replace(SMALL_BF16, name="timeout_mxd", routed_w="mxfp4", latent=512, hidden=512,
                                 experts=24, tokens=40, seed=38), 0, 1),
    ("mx_prefill_routed", replace(SMALL_BF16, name="timeout_mxp", routed_w="mxfp4", latent=512, hidden=512,
                                  experts=8, tokens=700, seed=39), 0, 1),
    ("gemv_fp4_decode_routed", replace(SMALL_BF16, name="timeout_gv", routed_w="mxfp4", latent=512, hidden=512,
                                       experts=24, tokens=40, seed=38), "dequant", 1),
], ids=lambda c: c[0])
def test_bounded_wait_runs_out_and_reports_timeout(binding, case):
    """A dropped pipeline-stage signal makes one consumer's bounded wait run out: the kernel waits for
    its own loads and MMAs in flight, unwinds, the status word reports LMOE_ERR_TIMEOUT, and the
    next call is correct again.  Covers the CTA-pair kernels (dense and swapped), the single-CTA
    grouped GEMM, the block-scaled MXFP4 kernel, and the decode kernels (tensor-core swap and the
    MXFP4 GEMV of the dequantizing path)."""
    _, cfg, flags, inject = case
    flags = {"single": binding.LMOE_FLAG_SINGLE_CTA_GEMM, "dequant": binding.LMOE_FLAG_MXFP4_DEQUANT}.get(flags, flags)
    dev = torch.device("cuda")
    inp = device_inputs(cfg, dev, False)
    layer = binding.LatentMoE(cfg, flags=flags)
    y_ref = layer.forward(inp["x"], inp).clone()
    assert layer.status() == 0
    layer.set_wait_limit(50_000_000, inject=inject)  # 50 ms, drop one stage signal in the next forward
    layer.forward(inp["x"], inp)
    assert layer.status() == binding.LMOE_ERR_TIMEOUT
    layer.set_wait_limit(4_000_000_000, inject=0)
    y = layer.forward(inp["x"], inp)
    assert layer.status() == 0
    assert torch.equal(y, y_ref)
    layer.close()
