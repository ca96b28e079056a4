"""ctypes binding of the C-ABI library (argument marshalling only; every step runs in the
library's CUDA kernels).  torch supplies device memory and streams.

Raises if the shared library is missing: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import torch

from .configs import LayerConfig

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "liblatentmoe.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "latentmoe.h")

LMOE_OK, LMOE_ERR_INVALID_ARG, LMOE_ERR_UNSUPPORTED, LMOE_ERR_CUDA, LMOE_ERR_OOM, LMOE_ERR_TIMEOUT, \
    LMOE_ERR_DEVICE_CHECK = range(7)
DTYPES = {"f32": 0, "bf16": 1, "mxfp4": 2}
LMOE_FLAG_IDENTITY_EXPERTS = 0x1
LMOE_FLAG_SINGLE_CTA_GEMM = 0x2
LMOE_FLAG_MXFP4_DEQUANT = 0x4
LMOE_FLAG_MXFP8_ACT = 0x8
LMOE_NUM_STAGES = 10


class LmoeConfig(C.Structure):
    _fields_ = [("d", C.c_int32), ("latent", C.c_int32), ("hidden", C.c_int32), ("num_experts", C.c_int32),
                ("top_k", C.c_int32), ("num_shared", C.c_int32), ("shared_hidden", C.c_int32),
                ("max_tokens", C.c_int32), ("act", C.c_int32), ("router_w", C.c_int32), ("routed_w", C.c_int32),
                ("rms_eps", C.c_float), ("flags", C.c_uint32)]


class LmoeWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "w_router", "router_bias", "w_down_proj", "rms_gain", "routed_gate_up", "routed_gate_up_scale",
        "routed_down", "routed_down_scale", "w_up_proj", "shared_gate_up", "shared_down")]


class LatentMoEError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib().latentmoe_status_string(status).decode()} (status {status})")


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} (run sparse_moe_layer_sigmoid_gb300.build)")
        lib = C.CDLL(LIB_PATH)
        vp, i32, st = C.c_void_p, C.c_int32, C.c_int
        lib.latentmoe_create.argtypes = [C.POINTER(LmoeConfig), C.POINTER(vp)]
        lib.latentmoe_destroy.argtypes = [vp]
        lib.latentmoe_route.argtypes = [vp, vp, i32, C.POINTER(LmoeWeights), vp, vp, vp, vp, vp, vp]
        lib.latentmoe_forward.argtypes = [vp, vp, i32, C.POINTER(LmoeWeights), vp, vp]
        lib.latentmoe_forward_routed.argtypes = [vp, vp, i32, C.POINTER(LmoeWeights), vp, vp, vp, vp]
        lib.latentmoe_forward_host.argtypes = [vp, vp, i32, C.POINTER(LmoeWeights), vp, vp]
        lib.latentmoe_ep_emulate.argtypes = [vp, vp, i32, C.POINTER(LmoeWeights), i32, i32, vp, vp, C.c_size_t, vp,
                                             vp, C.POINTER(vp), vp]
        lib.latentmoe_status.argtypes = [vp, vp]
        lib.latentmoe_last_launch_count.argtypes = [vp]
        lib.latentmoe_last_launch_count.restype = i32
        lib.latentmoe_workspace_bytes.argtypes = [vp]
        lib.latentmoe_workspace_bytes.restype = C.c_size_t
        lib.latentmoe_set_wait_limit.argtypes = [vp, C.c_uint64, i32]
        lib.latentmoe_set_stage_events.argtypes = [vp, C.POINTER(vp), i32]
        lib.latentmoe_set_stage_events.restype = st
        lib.latentmoe_stage_name.argtypes = [i32]
        lib.latentmoe_stage_name.restype = C.c_char_p
        lib.latentmoe_route_noalloc.argtypes = [C.POINTER(LmoeConfig), vp, i32, C.POINTER(LmoeWeights), vp, vp,
                                                vp, vp, vp, vp]
        lib.latentmoe_route_noalloc.restype = st
        lib.latentmoe_mx3_quantize.argtypes = [vp, i32, C.c_int64, i32, vp, vp]
        lib.latentmoe_mx3_quantize.restype = st
        lib.latentmoe_mx8_quantize.argtypes = [vp, i32, C.c_int64, i32, vp, vp]
        lib.latentmoe_mx8_quantize.restype = st
        lib.latentmoe_mma_peak.argtypes = [i32, C.POINTER(C.c_double), vp]
        lib.latentmoe_mma_peak.restype = st
        lib.latentmoe_route_noalloc_status.argtypes = [vp]
        lib.latentmoe_route_noalloc_status.restype = st
        lib.latentmoe_debug_buffer.argtypes = [vp, C.c_char_p, C.POINTER(vp), C.POINTER(C.c_size_t)]
        lib.latentmoe_debug_buffer.restype = st
        lib.latentmoe_status_string.argtypes = [st]
        lib.latentmoe_status_string.restype = C.c_char_p
        for name in ("latentmoe_create", "latentmoe_destroy", "latentmoe_route", "latentmoe_forward",
                     "latentmoe_forward_routed", "latentmoe_forward_host", "latentmoe_status",
                     "latentmoe_set_wait_limit"):
            getattr(lib, name).restype = st
        _LIB = lib
    return _LIB


def header_functions():
    """Names of the functions declared in include/latentmoe.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(latentmoe_\w+)\s*\(", text)))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(status, what):
    if status != LMOE_OK:
        raise LatentMoEError(status, what)


class _DeviceArray:
    """Minimal __cuda_array_interface__ holder for a raw device pointer (no ownership)."""

    def __init__(self, ptr: int, nbytes: int):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1", "data": (ptr, False), "version": 3}


def _wrap_device_pointer(ptr: int, nbytes: int, dtype, shape):
    """Copy `nbytes` at a raw device pointer into a new torch tensor viewed as dtype/shape."""
    torch.cuda.synchronize()
    raw = torch.as_tensor(_DeviceArray(ptr, nbytes), device="cuda")
    return raw.clone().view(dtype).reshape(shape)


def make_config(cfg: LayerConfig, max_tokens: int | None = None, flags: int = 0) -> LmoeConfig:
    return LmoeConfig(cfg.d, cfg.latent, cfg.hidden, cfg.experts, cfg.top_k, cfg.n_shared, cfg.shared_hidden,
                      max_tokens or cfg.tokens, DTYPES[cfg.act], DTYPES[cfg.router_w], DTYPES[cfg.routed_w],
                      cfg.rms_eps, flags | (LMOE_FLAG_IDENTITY_EXPERTS if cfg.identity_experts else 0))


def make_weights(inp: dict) -> LmoeWeights:
    return LmoeWeights(*[_ptr(inp.get(n)) for n, _ in LmoeWeights._fields_])


def route_noalloc(cfg: LayerConfig, x, weights: dict, out: dict, stream=None):
    """Router and dispatch through latentmoe_route_noalloc (no handle, no device allocation).

    ``out`` holds the caller's output tensors idx, p, offsets, tok_of_row, row_of."""
    c = make_config(cfg, max(1, x.shape[0]))
    w = make_weights(weights)
    return _lib().latentmoe_route_noalloc(C.byref(c), _ptr(x), x.shape[0], C.byref(w), _ptr(out["idx"]),
                                          _ptr(out["p"]), _ptr(out["offsets"]), _ptr(out["tok_of_row"]),
                                          _ptr(out["row_of"]), _stream(stream))


def mx3_quantize(x: torch.Tensor, stream=None) -> torch.Tensor:
    """Three-term MXFP4 records of the rows of x (bf16 or fp16 [rows][K]) as uint8 [rows][3K/2 + 3K/32]."""
    rows, K = x.shape
    out = torch.empty((rows, 3 * K // 2 + 3 * K // 32), dtype=torch.uint8, device=x.device)
    dt = {torch.bfloat16: 1, torch.float16: 3}[x.dtype]
    _check(_lib().latentmoe_mx3_quantize(_ptr(x), dt, rows, K, _ptr(out), _stream(stream)), "mx3_quantize")
    return out


def mx8_quantize(x: torch.Tensor, stream=None) -> torch.Tensor:
    """MXFP8 records of the rows of x (bf16 or fp16 [rows][K]) as uint8 [rows][K + K/32]."""
    rows, K = x.shape
    out = torch.empty((rows, K + K // 32), dtype=torch.uint8, device=x.device)
    dt = {torch.bfloat16: 1, torch.float16: 3}[x.dtype]
    _check(_lib().latentmoe_mx8_quantize(_ptr(x), dt, rows, K, _ptr(out), _stream(stream)), "mx8_quantize")
    return out


def mma_peak_tflops(kind: str, stream=None) -> float:
    """Measured tensor-core rate (TFLOP/s) of back-to-back CTA-pair MMAs: kind "f16" or "mxf4"."""
    out = C.c_double()
    _check(_lib().latentmoe_mma_peak({"f16": 0, "mxf4": 1}[kind], C.byref(out), _stream(stream)), "mma_peak")
    return out.value


def route_noalloc_status(stream=None) -> int:
    """Sticky status of the no-allocation route's kernels on the current device (read and cleared)."""
    return _lib().latentmoe_route_noalloc_status(_stream(stream))


class LatentMoE:
    """One layer instance: a handle with a workspace sized for ``max_tokens`` tokens."""

    def __init__(self, cfg: LayerConfig, max_tokens: int | None = None, flags: int = 0):
        self.cfg = cfg
        self.max_tokens = max_tokens or cfg.tokens
        self._c = make_config(cfg, self.max_tokens, flags)
        h = C.c_void_p()
        _check(_lib().latentmoe_create(C.byref(self._c), C.byref(h)), "latentmoe_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            _lib().latentmoe_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def out_width(self):
        return self.cfg.latent if self.cfg.identity_experts else self.cfg.d

    def _out(self, x, y):
        if y is None:
            y = torch.empty((x.shape[0], self.out_width), dtype=x.dtype, device=x.device)
        return y

    def forward(self, x, weights: dict, y=None, stream=None):
        y = self._out(x, y)
        w = make_weights(weights)
        _check(_lib().latentmoe_forward(self._h, _ptr(x), x.shape[0], C.byref(w), _ptr(y), _stream(stream)),
               "latentmoe_forward")
        return y

    def forward_routed(self, x, weights: dict, topk_idx, topk_p, y=None, stream=None):
        y = self._out(x, y)
        w = make_weights(weights)
        _check(_lib().latentmoe_forward_routed(self._h, _ptr(x), x.shape[0], C.byref(w), _ptr(topk_idx),
                                               _ptr(topk_p), _ptr(y), _stream(stream)), "latentmoe_forward_routed")
        return y

    def ep_emulate(self, x, weights: dict, ranks: int, full_width: bool, send=None, recv=None, stream=None,
                   events=None):
        """Expert-parallel dispatch + combine emulated on one GPU (latentmoe_ep_emulate): returns
        (u, cells) with u [T][width] and cells [ranks][ranks] int32 rows sent src -> dst."""
        T = x.shape[0]
        width = self.cfg.d if full_width else self.cfg.latent
        row_dtype = x.dtype if full_width else (torch.float16 if self.cfg.routed_w == "mxfp4" else x.dtype)
        rows = T * self.cfg.top_k
        if send is None:
            send = torch.empty((rows, width), dtype=row_dtype, device=x.device)
        if recv is None:
            recv = torch.empty((rows, width), dtype=row_dtype, device=x.device)
        nbytes = min(send.numel() * send.element_size(), recv.numel() * recv.element_size())
        u = torch.empty((T, width), dtype=x.dtype, device=x.device)
        cells = torch.zeros((ranks, ranks), dtype=torch.int32, device=x.device)
        w = make_weights(weights)
        ev = None
        if events is not None:
            ev = (C.c_void_p * 6)(*[e.cuda_event for e in events])
        _check(_lib().latentmoe_ep_emulate(self._h, _ptr(x), T, C.byref(w), int(ranks), int(bool(full_width)),
                                           _ptr(send), _ptr(recv), nbytes, _ptr(u), _ptr(cells), ev,
                                           _stream(stream)), "latentmoe_ep_emulate")
        return u, cells

    def forward_host(self, x_host, weights: dict, y_host=None, stream=None):
        if y_host is None:
            y_host = torch.empty((x_host.shape[0], self.out_width), dtype=x_host.dtype, pin_memory=True)
        w = make_weights(weights)
        _check(_lib().latentmoe_forward_host(self._h, _ptr(x_host), x_host.shape[0], C.byref(w), _ptr(y_host),
                                             _stream(stream)), "latentmoe_forward_host")
        return y_host

    def route(self, x, weights: dict, stream=None):
        T, k, E = x.shape[0], self.cfg.top_k, self.cfg.experts
        dev = x.device
        out = {"idx": torch.empty((T, k), dtype=torch.int32, device=dev),
               "p": torch.empty((T, k), dtype=torch.float32, device=dev),
               "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
               "tok_of_row": torch.empty(T * k, dtype=torch.int32, device=dev),
               "row_of": torch.empty((T, k), dtype=torch.int32, device=dev)}
        w = make_weights(weights)
        _check(_lib().latentmoe_route(self._h, _ptr(x), T, C.byref(w), _ptr(out["idx"]), _ptr(out["p"]),
                                      _ptr(out["offsets"]), _ptr(out["tok_of_row"]), _ptr(out["row_of"]),
                                      _stream(stream)), "latentmoe_route")
        return out

    def debug_buffer(self, name: str, dtype, shape):
        """View of a workspace intermediate of the last call (test hook; see latentmoe.h)."""
        ptr, nbytes = C.c_void_p(), C.c_size_t()
        _check(_lib().latentmoe_debug_buffer(self._h, name.encode(), C.byref(ptr), C.byref(nbytes)),
               f"debug_buffer({name})")
        n = 1
        for s_ in shape:
            n *= s_
        esize = torch.empty((), dtype=dtype).element_size()
        assert n * esize <= nbytes.value, (name, n * esize, nbytes.value)
        return _wrap_device_pointer(ptr.value, n * esize, dtype, shape)

    def routing_stats(self) -> dict:
        """Tokens of the last routing settled on exact keys, and the near ties among them."""
        v = self.debug_buffer("refine_count", torch.int32, (2,)).cpu()
        return {"refined_tokens": int(v[0]), "near_ties": int(v[1])}

    def status(self, stream=None) -> int:
        return _lib().latentmoe_status(self._h, _stream(stream))

    def last_launch_count(self) -> int:
        return _lib().latentmoe_last_launch_count(self._h)

    def workspace_bytes(self) -> int:
        return _lib().latentmoe_workspace_bytes(self._h)

    def enable_stage_timing(self):
        """Record a CUDA event between the stages of later calls (see stage_times_ms)."""
        self._events = [torch.cuda.Event(enable_timing=True) for _ in range(LMOE_NUM_STAGES + 1)]
        for e in self._events:  # torch creates the CUDA event on its first record
            e.record()
        torch.cuda.synchronize()
        arr = (C.c_void_p * len(self._events))(*[e.cuda_event for e in self._events])
        _check(_lib().latentmoe_set_stage_events(self._h, arr, len(self._events)), "set_stage_events")

    def disable_stage_timing(self):
        """Stop recording stage events (calls overlap W_down and the shared GLU again)."""
        _check(_lib().latentmoe_set_stage_events(self._h, None, 0), "set_stage_events")

    def stage_times_ms(self) -> dict:
        """Device time of each stage of the last call (synchronises on its last event)."""
        self._events[-1].synchronize()
        return {_lib().latentmoe_stage_name(i).decode(): self._events[i].elapsed_time(self._events[i + 1])
                for i in range(LMOE_NUM_STAGES)}

    def set_wait_limit(self, timeout_ns: int, inject: int = 0):
        """Bound in-kernel waits; inject 1 (first routed GEMM) or 2 (W_down) drops one pipeline signal."""
        _check(_lib().latentmoe_set_wait_limit(self._h, int(timeout_ns), int(inject)), "set_wait_limit")
