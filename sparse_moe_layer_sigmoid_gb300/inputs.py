"""Seeded synthetic inputs for the LatentMoE layer, shared by the oracle tests and the GPU path.

This module draws inputs and stores them in the storage formats the layer consumes
(fp32, bf16, or MXFP4 = E2M1 elements with one E8M0 scale per 32 elements along K).
It holds none of the layer's arithmetic.  The MXFP4 encoder below only *produces*
weight bytes from normal draws, following the OCP Microscaling (MX) v1.0 rule
(shared exponent = floor(log2 amax) - 2, elements rounded to nearest-even on the
E2M1 grid with saturation at +-6); the method itself only ever decodes them.

Draw order for one workload (all from one ``torch.Generator`` seeded with the
workload's seed, on the requested device): x, W_r, b, W_down, g, routed gate_up
(expert by expert), routed down (expert by expert), W_up, shared gate_up, shared down.
Weights are N(0, 1/fan_in), x ~ N(0, 1), g ~ 1 + N(0, 0.1).  Draws are fp32 and are
rounded to nearest-even into the stored type.

Bias recipes (router bias enters expert selection only):
  "normal1.5"  : b_e = 1.5 * z_e, z ~ N(0,1)
  "normal0.05" : b_e = 0.05 * z_e
  "zipf1.1"    : b_{pi(r)} = r^-1.1 / sum_{r'=1..E} r'^-1.1, pi a seeded random permutation
"""
from __future__ import annotations

import math

import numpy as np
import torch

from .configs import LayerConfig

_TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}

# E2M1 magnitudes in code order 0..7 (OCP MX v1.0, FP4 E2M1 table).
_E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
# Midpoints between consecutive magnitudes; a tie rounds toward the even code.
_E2M1_MID = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def encode_mxfp4(w: torch.Tensor):
    """Encode fp32 ``w`` [..., K] (K % 32 == 0) into MXFP4 bytes.

    Returns (packed uint8 [..., K/2], scales uint8 [..., K/32]).  Element 2i is the low
    nibble of byte i and element 2i+1 the high nibble; nibble = sign<<3 | code.
    """
    assert w.shape[-1] % 32 == 0
    lead = w.shape[:-1]
    K = w.shape[-1]
    blocks = w.float().reshape(*lead, K // 32, 32)
    amax = blocks.abs().amax(dim=-1)
    # shared exponent: floor(log2(amax)) - emax(E2M1)=2, biased by 127; all-zero block -> 2^0
    e = torch.where(amax > 0, torch.floor(torch.log2(torch.where(amax > 0, amax, torch.ones_like(amax)))) - 2.0,
                    torch.zeros_like(amax))
    e = e.clamp(-127.0, 127.0)
    scale = torch.exp2(e).unsqueeze(-1)
    v = blocks / scale
    mag = v.abs()
    code = torch.zeros_like(mag, dtype=torch.uint8)
    for i, m in enumerate(_E2M1_MID):
        # code i -> i+1 boundary; ties go to the even code
        up_on_tie = (i + 1) % 2 == 0
        step = (mag >= m) if up_on_tie else (mag > m)
        code += step.to(torch.uint8)
    sign = (v < 0).to(torch.uint8) & (code > 0).to(torch.uint8)
    nib = (sign << 3) | code
    nib = nib.reshape(*lead, K)
    packed = (nib[..., 0::2] | (nib[..., 1::2] << 4)).contiguous()
    scales = (e + 127.0).to(torch.uint8).contiguous()
    return packed, scales


def _normal(shape, std, g, device):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def _store(t: torch.Tensor, kind: str) -> torch.Tensor:
    return t.to(_TORCH_DT[kind]).contiguous()


def make_inputs(cfg: LayerConfig, device="cpu", seed: int | None = None) -> dict:
    """Draw every tensor of one workload on ``device`` (see module docstring for the recipe).

    Keys: x, w_router, router_bias (or None), w_down_proj, rms_gain, routed_gate_up,
    routed_gate_up_scale, routed_down, routed_down_scale, w_up_proj, shared_gate_up,
    shared_down.  Absent parts are None.  Layouts are row-major [out][in]:
      x [T][d]; w_router [E][d]; w_down_proj [l][d]; rms_gain [l] fp32;
      routed_gate_up [E][2h][l] (gate rows 0..h-1, up rows h..2h-1), MXFP4: [E][2h][l/2] bytes
        + routed_gate_up_scale [E][2h][l/32];
      routed_down [E][l][h], MXFP4: [E][l][h/2] + routed_down_scale [E][l][h/32];
      w_up_proj [d][l]; shared_gate_up [N_s][2h_s][d]; shared_down [N_s][d][h_s].
    """
    seed = cfg.seed if seed is None else seed
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    T, d, l, h, E = cfg.tokens, cfg.d, cfg.latent, cfg.hidden, cfg.experts
    out = {k: None for k in ("x", "w_router", "router_bias", "w_down_proj", "rms_gain",
                             "routed_gate_up", "routed_gate_up_scale", "routed_down",
                             "routed_down_scale", "w_up_proj", "shared_gate_up", "shared_down")}
    out["x"] = _store(_normal((T, d), 1.0, g, dev), cfg.act)
    out["w_router"] = _store(_normal((E, d), 1.0 / math.sqrt(d), g, dev), cfg.router_w)
    if cfg.bias.startswith("normal"):
        sigma = float(cfg.bias[len("normal"):])
        out["router_bias"] = (_normal((E,), 1.0, g, dev) * sigma).contiguous()
    elif cfg.bias.startswith("zipf"):
        s = float(cfg.bias[len("zipf"):])
        perm = torch.randperm(E, generator=g, device=dev)
        ranks = torch.arange(1, E + 1, device=dev, dtype=torch.float64)
        pmf = ranks.pow(-s)
        pmf = pmf / pmf.sum()
        b = torch.empty(E, dtype=torch.float64, device=dev)
        b[perm] = pmf
        out["router_bias"] = b.to(torch.float32).contiguous()
    out["w_down_proj"] = _store(_normal((l, d), 1.0 / math.sqrt(d), g, dev), cfg.act)
    out["rms_gain"] = (1.0 + _normal((l,), 0.1, g, dev)).contiguous()
    if not cfg.identity_experts:
        if cfg.routed_w == "mxfp4":
            gu = torch.empty((E, 2 * h, l // 2), dtype=torch.uint8, device=dev)
            gus = torch.empty((E, 2 * h, l // 32), dtype=torch.uint8, device=dev)
            for e in range(E):
                gu[e], gus[e] = encode_mxfp4(_normal((2 * h, l), 1.0 / math.sqrt(l), g, dev))
            dn = torch.empty((E, l, h // 2), dtype=torch.uint8, device=dev)
            dns = torch.empty((E, l, h // 32), dtype=torch.uint8, device=dev)
            for e in range(E):
                dn[e], dns[e] = encode_mxfp4(_normal((l, h), 1.0 / math.sqrt(h), g, dev))
            out["routed_gate_up"], out["routed_gate_up_scale"] = gu, gus
            out["routed_down"], out["routed_down_scale"] = dn, dns
        else:
            dt = _TORCH_DT[cfg.routed_w]
            gu = torch.empty((E, 2 * h, l), dtype=dt, device=dev)
            for e in range(E):
                gu[e] = _normal((2 * h, l), 1.0 / math.sqrt(l), g, dev).to(dt)
            dn = torch.empty((E, l, h), dtype=dt, device=dev)
            for e in range(E):
                dn[e] = _normal((l, h), 1.0 / math.sqrt(h), g, dev).to(dt)
            out["routed_gate_up"], out["routed_down"] = gu, dn
        out["w_up_proj"] = _store(_normal((d, l), 1.0 / math.sqrt(l), g, dev), cfg.act)
        if cfg.n_shared > 0:
            hs = cfg.shared_hidden
            out["shared_gate_up"] = _store(_normal((cfg.n_shared, 2 * hs, d), 1.0 / math.sqrt(d), g, dev), cfg.act)
            out["shared_down"] = _store(_normal((cfg.n_shared, d, hs), 1.0 / math.sqrt(hs), g, dev), cfg.act)
    return out


def to_host(t: torch.Tensor | None):
    """Copy a stored tensor to a numpy array without changing its bytes.

    bf16 becomes uint16 (the raw bit pattern), fp32 stays float32, bytes stay uint8.
    """
    if t is None:
        return None
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


class ExpertSlices:
    """Lazy host view of a device tensor with a leading expert axis: ``obj[e]`` copies expert e.

    Lets the oracle touch only the experts a token sample selects, without copying a
    multi-gigabyte routed-weight pool to the host.
    """

    def __init__(self, t: torch.Tensor | None):
        self.t = t
        self._cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self._cache:
            self._cache[e] = to_host(self.t[e])
        return self._cache[e]

    def __len__(self):
        return self.t.shape[0]


def host_inputs(inp: dict, lazy_experts: bool = False) -> dict:
    """Host (numpy) copy of ``make_inputs`` output for the oracle; routed weights optionally lazy."""
    out = {}
    for k, v in inp.items():
        if v is None:
            out[k] = None
        elif lazy_experts and k.startswith("routed_"):
            out[k] = ExpertSlices(v)
        else:
            out[k] = to_host(v)
    return out


def sample_tokens(T: int, n: int, seed: int) -> np.ndarray:
    """Seeded random subset of ``n`` distinct token rows (sorted), or all rows when T <= n."""
    if T <= n:
        return np.arange(T)
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    return np.sort(rng.choice(T, size=n, replace=False))
