"""The C-ABI library builds, loads, exports every declared entry point, and validates arguments
on the host (no GPU needed: these calls return before touching CUDA)."""
import ctypes as C
from dataclasses import replace

import pytest

from sparse_moe_layer_sigmoid_gb300 import configs


@pytest.fixture(scope="module")
def b():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_moe_layer_sigmoid_gb300 import binding
    return binding


def test_library_exports_every_declared_function(b):
    lib = b._lib()
    names = b.header_functions()
    for required in ("latentmoe_create", "latentmoe_route", "latentmoe_forward", "latentmoe_destroy"):
        assert required in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(b):
    lib = b._lib()
    for s in range(7):
        assert lib.latentmoe_status_string(s)
    assert lib.latentmoe_status_string(b.LMOE_OK) == b"ok"


def test_null_handle_and_bad_config_rejected_on_host(b):
    lib = b._lib()
    w = b.LmoeWeights()
    assert lib.latentmoe_forward(None, None, 0, C.byref(w), None, None) == b.LMOE_ERR_INVALID_ARG
    assert lib.latentmoe_route(None, None, 0, C.byref(w), None, None, None, None, None, None) == b.LMOE_ERR_INVALID_ARG
    assert lib.latentmoe_status(None, None) == b.LMOE_ERR_INVALID_ARG
    assert lib.latentmoe_destroy(None) == b.LMOE_OK
    assert lib.latentmoe_last_launch_count(None) == 0
    h = C.c_void_p()
    for bad in (replace(configs.TINY_F32, top_k=0), replace(configs.TINY_F32, experts=2000),
                replace(configs.TINY_F32, top_k=40, experts=64), replace(configs.TINY_F32, tokens=0)):
        c = b.make_config(bad, max(bad.tokens, 0) or None)
        if bad.tokens == 0:
            c.max_tokens = 0
        assert lib.latentmoe_create(C.byref(c), C.byref(h)) == b.LMOE_ERR_INVALID_ARG
        assert not h.value
    # shapes the tensor-core tiles cannot cover are refused as unsupported
    c = b.make_config(replace(configs.K3W_E128_BF16_PREFILL, d=7000))
    assert lib.latentmoe_create(C.byref(c), C.byref(h)) == b.LMOE_ERR_UNSUPPORTED
    assert lib.latentmoe_create(None, C.byref(h)) == b.LMOE_ERR_INVALID_ARG


def test_config_table_matches_workloads():
    c1 = configs.K3W_E128_BF16_PREFILL
    assert (c1.tokens, c1.d, c1.latent, c1.hidden, c1.experts, c1.top_k, c1.n_shared) == (4096, 7168, 3584, 3072,
                                                                                           128, 16, 2)
    c4 = configs.ROUTING_DISPATCH_STRESS
    assert c4.identity_experts and c4.rows == 65536 * 16
