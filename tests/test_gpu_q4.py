"""GPU parity of batch-1 decode with 4-bit group-affine experts (moe_create_q4) against the
CPU oracle's 4-bit layer: routing bit-exact, outputs within the layer tolerance."""
import numpy as np
import pytest

import sparse_moe_02_gb300 as moe
import synth
from _cases import (assert_close, bf16_bits, build_case, oracle_outputs_q4, oracle_route,
                    q4_to_device, to_device)

pytestmark = pytest.mark.gpu


def _run_q4(c, schedule=moe.MOE_SCHEDULE_AUTO):
    import torch
    W = q4_to_device(c)
    x = torch.from_numpy(c.x.view(np.int16)).cuda().view(torch.bfloat16)
    L = moe.MoeLayer(W, max(c.T, 1), schedule=schedule)
    y = L.forward(x)
    r = L.route(x)
    torch.cuda.synchronize()
    assert L.device_error() == moe.MOE_OK
    out = {k: v.cpu().numpy() for k, v in r.items()}
    out["y"] = bf16_bits(y)
    L.close()
    return out


@pytest.mark.parametrize("d,f,fs,seed", [(512, 128, 256, 1), (2048, 512, 512, 0),
                                         (4096, 2048, 2048, 2), (640, 384, 128, 3)])
def test_q4_decode_matches_oracle(d, f, fs, seed):
    c = build_case("q4-decode", d=d, f=f, fs=fs, T=1, seed=seed, full_host=False)
    for sched in (moe.MOE_SCHEDULE_AUTO, moe.MOE_SCHEDULE_GEMV):
        got = _run_q4(c, sched)
        ref = oracle_route(c)
        assert np.array_equal(got["topk_idx"], ref["topk_idx"])
        assert np.max(np.abs(got["topk_w"] - ref["topk_w"])) <= 1e-5
        assert_close(got["y"], oracle_outputs_q4(c), f"q4 decode d={d} f={f} fs={fs}")


def test_q4_decode_layers_of_the_benchmark():
    for layer in (0, 7):
        c = build_case("q4-bench", d=2048, f=512, fs=512, T=1, seed=1000, layer=layer,
                       full_host=False)
        got = _run_q4(c)
        assert_close(got["y"], oracle_outputs_q4(c), f"q4 decode layer {layer}")


def test_q4_handle_limits():
    import torch
    c = build_case("q4-limits", d=512, f=128, fs=128, T=5, seed=9, full_host=False)
    W = q4_to_device(c)
    x = torch.from_numpy(c.x.view(np.int16)).cuda().view(torch.bfloat16)
    L = moe.MoeLayer(W, 8)
    y = torch.empty_like(x)
    # more than one token: the tensor-core path reads bf16 experts
    assert moe.moe_forward(L.handle, x.data_ptr(), 5, y.data_ptr(), None) == \
        moe.MOE_ERR_UNSUPPORTED
    # routing works for any T (the router stays bf16)
    r = L.route(x)
    torch.cuda.synchronize()
    assert np.array_equal(r["topk_idx"].cpu().numpy(), oracle_route(c)["topk_idx"])
    assert L.device_error() == moe.MOE_OK
    L.close()
    cfg = moe.moe_config(512, 256, 8, 128, 128, 8, moe.MOE_SCHEDULE_GEMM, 0)
    w = moe.moe_weights_q4(W["w_router"].data_ptr(), None,
                           *(moe.moe_q4_matrix(*(t.data_ptr() for t in W[n]))
                             for n in synth.Q4_NAMES))
    st, h = moe.moe_create_q4(cfg, w)
    assert st == moe.MOE_ERR_UNSUPPORTED and not h.value


def test_q4_device_fill_equals_host():
    import torch
    dims = synth.Dims(d=512, f=128, fs=256)
    for nm in ("w_down", "ws_gate"):
        cs, gs = synth.q4_shapes(nm, dims)
        codes = torch.empty(cs, dtype=torch.uint8, device="cuda")
        sc = torch.empty(gs, dtype=torch.int16, device="cuda")
        b = torch.empty(gs, dtype=torch.int16, device="cuda")
        synth.q4_device(4, 2, nm, dims, codes.data_ptr(), sc.data_ptr(), b.data_ptr(),
                        torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        hc, hs, hb = synth.q4_host(4, 2, nm, dims)
        assert np.array_equal(codes.cpu().numpy(), hc)
        assert np.array_equal(sc.cpu().numpy().view(np.uint16), hs)
        assert np.array_equal(b.cpu().numpy().view(np.uint16), hb)
