"""Host-side checks of the C ABI that need no GPU: the library loads, exports every function
include/moe.h declares, and rejects invalid arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import sparse_moe_02_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\*]+\s+\**(moe_\w+)\s*\(", src, re.M)))


def test_library_exports_every_declared_function():
    declared = _declared_functions()
    assert "moe_create" in declared and "moe_forward" in declared
    L = moe.lib()
    for fn in declared:
        assert hasattr(L, fn), f"{fn} declared in include/moe.h but not exported"
    assert set(declared) == set(moe.EXPORTS)


def _cfg(**kw):
    base = dict(d=512, n_experts=256, top_k=8, ffn_dim=128, shared_ffn_dim=128, max_tokens=64,
                schedule=0, chunk_tokens=0)
    base.update(kw)
    return moe.moe_config(**base)


def _weights(addr=0x10000, **kw):
    names = ["w_router", "router_bias", "w_gate", "w_up", "w_down", "ws_gate", "ws_up",
             "ws_down"]
    vals = {n: addr + 0x100000 * i for i, n in enumerate(names)}
    vals["router_bias"] = None
    vals.update(kw)
    return moe.moe_weights(**vals)


@pytest.mark.parametrize("kw,status", [
    (dict(n_experts=128), moe.MOE_ERR_UNSUPPORTED),
    (dict(top_k=4), moe.MOE_ERR_UNSUPPORTED),
    (dict(d=500), moe.MOE_ERR_UNSUPPORTED),
    (dict(d=16384), moe.MOE_ERR_UNSUPPORTED),
    (dict(ffn_dim=96), moe.MOE_ERR_UNSUPPORTED),
    (dict(shared_ffn_dim=4096), moe.MOE_ERR_UNSUPPORTED),
    (dict(max_tokens=0), moe.MOE_ERR_INVALID_ARG),
    (dict(max_tokens=(1 << 20) + 1), moe.MOE_ERR_UNSUPPORTED),
    (dict(d=0), moe.MOE_ERR_INVALID_ARG),
    (dict(schedule=7), moe.MOE_ERR_INVALID_ARG),
    (dict(chunk_tokens=-1), moe.MOE_ERR_INVALID_ARG),
])
def test_create_rejects_bad_config(kw, status):
    st, h = moe.moe_create(_cfg(**kw), _weights())
    assert st == status and not h.value


def test_create_rejects_bad_weight_pointers():
    st, h = moe.moe_create(_cfg(), _weights(w_gate=None))
    assert st == moe.MOE_ERR_INVALID_ARG and not h.value
    st, h = moe.moe_create(_cfg(), _weights(w_down=0x10008))
    assert st == moe.MOE_ERR_ALIGNMENT and not h.value
    st, h = moe.moe_create(_cfg(), _weights(router_bias=0x10002))
    assert st == moe.MOE_ERR_ALIGNMENT and not h.value
    L = moe.lib()
    assert L.moe_create(None, None, None) == moe.MOE_ERR_INVALID_ARG


def test_calls_on_null_handle_are_rejected():
    assert moe.moe_forward(None, None, 1, None, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_forward_host(None, None, 1, None, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_route(None, None, 1, None, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_get_device_error(None, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_test_expire_waits(None, 1) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_destroy(None) == moe.MOE_OK


def test_status_strings():
    for st in range(8):
        assert moe.moe_status_string(st) and moe.moe_status_string(st) != "unknown status"
    assert moe.moe_status_string(99) == "unknown status"


def test_create_without_gpu_reports_cuda_error():
    # on a host without a GPU the first CUDA call fails; the handle is not created
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = moe.moe_create(_cfg(), _weights())
    assert st == moe.MOE_ERR_CUDA and not h.value
