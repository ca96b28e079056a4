"""Shared parity helpers for the GPU tests: tolerances, error metrics, routing comparison."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from sparse_moe_layer_sigmoid_gb300 import inputs

# Output tolerances: relative Frobenius error by storage precision, and a per-element bound of
# 5e-2 * rms(y).  Routing indices must match except where the oracle's k-th/(k+1)-th key gap is
# below NEAR_TIE.
REL_FRO = {"f32": 1e-4, "bf16": 1e-2, "mxfp4": 2e-2}
MAX_ERR_RMS = 5e-2
NEAR_TIE = 1e-6


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy() if t.dtype != torch.int32 else t.cpu().numpy()


def rel_fro(a, b) -> float:
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def max_err_over_rms(a, b) -> float:
    return float(np.abs(a - b).max() / np.sqrt(np.mean(b * b)))


def assert_close(got, want, tol_rel, what=""):
    r = rel_fro(got, want)
    m = max_err_over_rms(got, want)
    assert r <= tol_rel, f"{what}: relative Frobenius error {r:.3e} > {tol_rel:.1e}"
    assert m <= MAX_ERR_RMS, f"{what}: max element error {m:.3e} x rms > {MAX_ERR_RMS}"
    return r, m


def compare_routing(idx_gpu: np.ndarray, ref: dict):
    """The selected experts in rank order (eq. 13's argtopk with the lower-index tie rule; ranks
    by descending key) must equal the oracle's, except on near-tie tokens, whose k-th/(k+1)-th
    key gap is below NEAR_TIE.  Returns (mismatched token mask, near-tie count); asserts that
    every mismatch is a near tie."""
    mism = np.any(idx_gpu != ref["idx"], axis=1)
    near = ref["gap"] < NEAR_TIE
    bad = mism & ~near
    assert not bad.any(), f"routing differs on {int(bad.sum())} tokens with gap >= {NEAR_TIE}: " \
                          f"{np.nonzero(bad)[0][:10]}"
    return mism, int(near.sum())


def oracle_routing(host: dict, cfg, chunk: int = 2048):
    """The oracle's routing (idx, p, gap) of every token, evaluated in row chunks."""
    T = np.asarray(host["x"]).shape[0]
    w_r = oracle.widen(host["w_router"])
    bias = None if host.get("router_bias") is None else oracle.widen(host["router_bias"])
    idx = np.empty((T, cfg.top_k), dtype=np.int64)
    p = np.empty((T, cfg.top_k))
    gap = np.empty(T)
    for t0 in range(0, T, chunk):
        x = oracle.widen(np.asarray(host["x"][t0:t0 + chunk]))
        s = oracle.router_scores(x, w_r)
        i, g = oracle.select_topk(s, bias, cfg.top_k)
        idx[t0:t0 + chunk], gap[t0:t0 + chunk] = i, g
        p[t0:t0 + chunk] = oracle.route_weights(s, i)
    return {"idx": idx, "p": p, "gap": gap}


def check_dispatch(out: dict, idx_gpu: np.ndarray, E: int):
    """GPU histogram/scan/permutation must equal the oracle's for the same routing, bit for bit."""
    counts, offsets, tok_of_row, row_of = oracle.dispatch(idx_gpu.astype(np.int64), E)
    assert np.array_equal(out["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(out["tok_of_row"].cpu().numpy(), tok_of_row)
    assert np.array_equal(out["row_of"].cpu().numpy(), row_of)
    return counts


def device_inputs(cfg, dev, generate_on_device: bool):
    """Inputs for a workload: drawn on the device for large workloads, else on the CPU."""
    if generate_on_device:
        inp = inputs.make_inputs(cfg, dev)
    else:
        inp = {k: (None if v is None else v.to(dev)) for k, v in inputs.make_inputs(cfg, "cpu").items()}
    return inp


def oracle_for_rows(inp_dev: dict, cfg, rows, routing_gpu=None):
    """Oracle on a row subset; routed weights are copied to the host one expert at a time."""
    host = inputs.host_inputs(inp_dev, lazy_experts=True)
    return oracle.layer_forward(host, cfg, tokens=rows, routing=routing_gpu), host
