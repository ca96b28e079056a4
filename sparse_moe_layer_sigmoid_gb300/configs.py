"""Workload table for the LatentMoE layer forward pass.

Shapes and precisions of the five synthetic workloads used for parity tests and
benchmarking (plus a milder-skew variant of the MXFP4 prefill workload).  The
widths d=7168, l=3584, h=3072, E=896, k=16, N_s=2 are the Kimi K3 numbers quoted
on "Lesson 6 - LatentMoE" (kimi-k3-course.pages.dev), sections "Deriving the
headline number" and "How routing works".

This module holds only shapes and generator recipes; no arithmetic of the method.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class LayerConfig:
    name: str
    tokens: int          # T
    d: int               # model width
    latent: int          # l, routed-expert width
    hidden: int          # h, routed-expert GLU hidden width (0 with identity experts)
    experts: int         # E, routed experts
    top_k: int           # k
    n_shared: int        # N_s, shared experts
    shared_hidden: int   # shared-expert GLU hidden width
    act: str             # activation / dense-weight storage: "f32" | "bf16"
    router_w: str        # "f32" | "bf16"
    routed_w: str        # "f32" | "bf16" | "mxfp4"
    bias: str            # "none" | "normal1.5" | "normal0.05" | "zipf1.1"
    identity_experts: bool
    seed: int
    rms_eps: float = 1e-6

    @property
    def rows(self) -> int:
        """Number of (token, expert) pairs, T*k."""
        return self.tokens * self.top_k


TINY_F32 = LayerConfig("tiny_f32", 64, 256, 128, 96, 32, 4, 1, 96,
                       "f32", "f32", "f32", "none", False, 0)
K3W_E128_BF16_PREFILL = LayerConfig("k3w_e128_bf16_prefill", 4096, 7168, 3584, 3072, 128, 16, 2, 3072,
                                    "bf16", "bf16", "bf16", "none", False, 1)
K3_MXFP4_DECODE = LayerConfig("k3_mxfp4_decode", 32, 7168, 3584, 3072, 896, 16, 2, 3072,
                              "bf16", "bf16", "mxfp4", "none", False, 2)
K3_MXFP4_PREFILL_SKEW = LayerConfig("k3_mxfp4_prefill_skew", 8192, 7168, 3584, 3072, 896, 16, 2, 3072,
                                    "bf16", "bf16", "mxfp4", "normal1.5", False, 3)
K3_MXFP4_PREFILL_MILD = replace(K3_MXFP4_PREFILL_SKEW, name="k3_mxfp4_prefill_mild", bias="normal0.05")
ROUTING_DISPATCH_STRESS = LayerConfig("routing_dispatch_t65536", 65536, 7168, 3584, 0, 896, 16, 0, 0,
                                      "bf16", "f32", "bf16", "zipf1.1", True, 4)

# Same widths as the bf16 prefill workload with 32 experts and 1024 tokens: about 2.5 GB on the
# device (weights still far larger than L2), small enough for multi-pass profiler captures.
K3W_E32_BF16_PROFILE = replace(K3W_E128_BF16_PREFILL, name="k3w_e32_bf16_t1024", tokens=1024, experts=32)

# MXFP4 cases of the same kind for profiler captures: decode-shaped (8 tokens over 128 experts,
# about one row per touched expert) and prefill-shaped (1024 tokens over 32 experts).
K3_MXFP4_DECODE_PROFILE = replace(K3_MXFP4_DECODE, name="k3_mxfp4_decode_e128_t8", tokens=8, experts=128)
K3_MXFP4_PREFILL_PROFILE = replace(K3_MXFP4_PREFILL_SKEW, name="k3_mxfp4_prefill_e32_t1024", tokens=1024,
                                   experts=32, bias="none")
# The routing stress workload at 8192 tokens (about 0.5 GB on the device) for captures of the
# routing kernels.
ROUTING_DISPATCH_PROFILE = replace(ROUTING_DISPATCH_STRESS, name="routing_dispatch_t8192", tokens=8192)
# The decode layer's routing (T=32, E=896, the same seed and router) with identity experts: the
# short-batch routing kernels on about 0.1 GB of weights, for captures of those kernels.
ROUTING_DECODE_PROFILE = replace(K3_MXFP4_DECODE, name="routing_decode_t32", hidden=0, n_shared=0,
                                 routed_w="bf16", identity_experts=True)

CONFIGS = {c.name: c for c in (TINY_F32, K3W_E128_BF16_PREFILL, K3_MXFP4_DECODE,
                               K3_MXFP4_PREFILL_SKEW, K3_MXFP4_PREFILL_MILD,
                               ROUTING_DISPATCH_STRESS, K3W_E32_BF16_PROFILE,
                               K3_MXFP4_DECODE_PROFILE, K3_MXFP4_PREFILL_PROFILE,
                               ROUTING_DISPATCH_PROFILE, ROUTING_DECODE_PROFILE)}


def scaled(cfg: LayerConfig, **kw) -> LayerConfig:
    """A copy of ``cfg`` with some fields replaced (used for reduced-size parity cases)."""
    return replace(cfg, **kw)
