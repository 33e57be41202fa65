"""moe_route_one_noalloc: routing of one token for callers that cannot allocate device memory.

Such callers (device memory reserved up front by another allocator, or code that may not call
cudaMalloc because it can synchronise the device) cannot create a handle, so this entry point
keeps its scratch in a static device array instead of a workspace.  The test calls it through
the C ABI twice in a row, on two different tokens, and checks each result against the CPU
oracle's routing of that token (x drawn under the 1e-3 logit-gap rule) and against the
handle-based moe_route of the same token: expert ids bit-exact, weights within the 1e-5 the
routing parity tests use.  d = 4096 sums more chunks per lane than the handle's router does
in one piece, so its logits are ordered differently; the gap rule keeps the selection equal.
It runs last (file name) and passes alone or after the others.
"""
import numpy as np
import pytest

import sparse_moe_02_gb300 as moe
from _cases import build_case, oracle_route, to_device

pytestmark = pytest.mark.gpu


def test_noalloc_route_matches_oracle_and_handle_route_on_two_calls():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    for d, skew in ((2048, False), (512, True), (4096, False)):
        c = build_case("noalloc", d=d, f=128, fs=128, T=2, seed=21 + d, skew=skew,
                       full_host=False)
        ref_o = oracle_route(c)
        W, x = to_device(c)
        layer = moe.MoeLayer(W, 1, schedule=moe.MOE_SCHEDULE_GEMV)
        bias = W.get("router_bias")
        stream = torch.cuda.current_stream().cuda_stream
        for t in range(2):  # two calls in a row, different tokens
            ref_h = layer.route(x[t:t + 1])
            idx = torch.full((8,), -1, dtype=torch.int32, device="cuda")
            w = torch.zeros(8, dtype=torch.float32, device="cuda")
            st = moe.moe_route_one_noalloc(x[t].data_ptr(), d, W["w_router"].data_ptr(),
                                           None if bias is None else bias.data_ptr(),
                                           idx.data_ptr(), w.data_ptr(), stream)
            assert st == moe.MOE_OK, moe.moe_status_string(st)
            torch.cuda.synchronize()
            got_i, got_w = idx.cpu().numpy(), w.cpu().numpy()
            assert np.array_equal(got_i, ref_o["topk_idx"][t]), f"d={d} t={t}: ids vs oracle"
            assert np.max(np.abs(got_w - ref_o["topk_w"][t])) <= 1e-5
            assert np.array_equal(got_i, ref_h["topk_idx"][0].cpu().numpy())
            assert np.max(np.abs(got_w - ref_h["topk_w"][0].cpu().numpy())) <= 1e-5
        layer.close()
        del W, x
    # sizes beyond the supported range and misaligned pointers are rejected before any launch
    x0 = torch.zeros(8320, dtype=torch.bfloat16, device="cuda")
    out_i = torch.zeros(8, dtype=torch.int32, device="cuda")
    out_w = torch.zeros(8, dtype=torch.float32, device="cuda")
    assert moe.moe_route_one_noalloc(x0.data_ptr(), 8320, x0.data_ptr(), None, out_i.data_ptr(),
                                     out_w.data_ptr(), None) == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_route_one_noalloc(x0.data_ptr() + 2, 512, x0.data_ptr(), None,
                                     out_i.data_ptr(), out_w.data_ptr(), None) == \
        moe.MOE_ERR_ALIGNMENT
    assert moe.moe_route_one_noalloc(None, 512, x0.data_ptr(), None, out_i.data_ptr(),
                                     out_w.data_ptr(), None) == moe.MOE_ERR_INVALID_ARG
