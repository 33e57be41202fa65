"""Host-side checks of the C ABI that need no GPU: the library loads, exports every function
include/moe.h and include/gdn.h declare, and rejects invalid arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import sparse_moe_02_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not hdr.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", hdr)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[\w\*]+\s+\**((?:moe|gdn)_\w+)\s*\(", src,
                                re.M))
    return sorted(names)


def test_library_exports_every_declared_function():
    declared = _declared_functions()
    assert "moe_create" in declared and "moe_forward" in declared and "gdn_scan" in declared
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
    A = 0x100000  # aligned stand-in device addresses: every case fails before any CUDA call
    assert moe.moe_check_routing(A, A, A, 4, None, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_check_routing(A, None, A, 4, A, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_check_routing(None, A, A, 4, A, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_check_routing(A, A, A, -1, A, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_check_routing(A, A, A, (1 << 20) + 1, A, None) == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_check_routing(A + 2, A, A, 4, A, None) == moe.MOE_ERR_ALIGNMENT
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


def test_scan_rejects_bad_arguments_before_touching_cuda():
    # 16-byte aligned stand-in addresses, never dereferenced: every case below fails in the
    # argument checks, before any CUDA call
    A = 0x100000
    ok = dict(q=A, k=A + 0x10000, v=A + 0x20000, alpha=A + 0x30000, beta=A + 0x40000,
              state_in=A + 0x50000, state_out=A + 0x60000, o=A + 0x70000, T=64, H=2, dk=128,
              dv=64, stream=None)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return moe.gdn_scan(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["state_in"],
                            a["state_out"], a["o"], a["T"], a["H"], a["dk"], a["dv"], a["stream"])

    assert call(T=-1) == moe.MOE_ERR_INVALID_ARG
    assert call(H=0) == moe.MOE_ERR_INVALID_ARG
    assert call(state_out=None) == moe.MOE_ERR_INVALID_ARG
    for name in ("q", "k", "v", "alpha", "beta", "o"):
        assert call(**{name: None}) == moe.MOE_ERR_INVALID_ARG, name
    assert call(dk=64) == moe.MOE_ERR_UNSUPPORTED
    assert call(dv=48) == moe.MOE_ERR_UNSUPPORTED
    assert call(dv=0) == moe.MOE_ERR_UNSUPPORTED
    assert call(dv=8192) == moe.MOE_ERR_UNSUPPORTED
    assert call(H=65536) == moe.MOE_ERR_UNSUPPORTED
    for name in ("q", "k", "v", "o"):
        assert call(**{name: ok[name] + 8}) == moe.MOE_ERR_ALIGNMENT, name
    for name in ("alpha", "beta", "state_in", "state_out"):
        assert call(**{name: ok[name] + 2}) == moe.MOE_ERR_ALIGNMENT, name
