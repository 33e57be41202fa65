"""GPU parity of the layer with 4-bit group-affine experts (moe_create_q4) against the CPU
oracle's 4-bit layer, on both paths (batch-1 matrix-vector decode and the dequantizing
tensor-core grouped GEMM): routing bit-exact, outputs within the layer tolerance."""
import numpy as np
import pytest

import sparse_moe_02_gb300 as moe
import synth
import oracle
from _cases import (assert_close, bf16_bits, build_case, oracle_outputs_q4, oracle_route,
                    q4_to_device, sample_tokens)

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
                                         (4096, 2048, 2048, 2), (640, 384, 128, 3),
                                         # the streamed launch (d, f, fs multiples of 512,
                                         # d <= 2048): fs > f, f > fs, the largest f it
                                         # takes at d = 2048, four outputs per block
                                         (1024, 512, 1024, 4), (1536, 1024, 512, 5),
                                         (2048, 1536, 512, 6), (512, 512, 512, 7)])
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


# ---------------------------------------------------------------- tensor-core path (T > 1)
# The grouped GEMM dequantizes each 64-input step of a weight tile to bf16 in tensor memory:
# routing bit-exact, outputs within the layer tolerance of the oracle's fp32 dequantization.

@pytest.mark.parametrize("d,f,fs,T,seed,skew", [
    (512, 128, 128, 64, 0, False),     # the tiny layer's shape, every token
    (512, 128, 256, 300, 1, False),    # ragged T, shared inner dim != routed
    (640, 384, 128, 77, 3, False),     # d = 5 x 128: the last down unit has one 128-row tile
    (1024, 256, 256, 500, 4, True),    # skewed routing: empty and crowded experts
])
def test_q4_prefill_matches_oracle(d, f, fs, T, seed, skew):
    c = build_case("q4-prefill", d=d, f=f, fs=fs, T=T, seed=seed, skew=skew, full_host=False)
    got = _run_q4(c)
    ref = oracle_route(c)
    assert np.array_equal(got["topk_idx"], ref["topk_idx"])
    assert np.array_equal(got["perm"], ref["perm"])
    assert np.array_equal(got["offsets"], ref["offsets"])
    assert np.max(np.abs(got["topk_w"] - ref["topk_w"])) <= 1e-5
    assert_close(got["y"], oracle_outputs_q4(c), f"q4 prefill d={d} f={f} fs={fs} T={T}")


@pytest.mark.parametrize("skew", [False, True], ids=["balanced", "skewed"])
def test_q4_prefill_4096(skew):
    """The benchmark's prefill shape (T=4096, d=2048, f=fs=512) in the launch configuration
    the benchmark times: the routing of every token bit-exact, outputs on every token."""
    c = build_case("q4-prefill-4096", d=2048, f=512, fs=512, T=4096, seed=0, skew=skew,
                   full_host=False)
    got = _run_q4(c)
    ref = oracle.route(c.x, c.w_r, c.dims.k, c.bias)
    assert np.array_equal(got["topk_idx"], ref["topk_idx"])
    assert np.max(np.abs(got["topk_w"] - ref["topk_w"])) <= 1e-5
    assert np.array_equal(got["offsets"], ref["offsets"])
    assert np.array_equal(got["perm"], ref["perm"])
    assert_close(got["y"], oracle_outputs_q4(c), f"q4 prefill 4096 skew={skew} (all tokens)")


@pytest.mark.parametrize("d,f", [(8192, 512), (4096, 2048)])
def test_q4_prefill_largest_shapes(d, f):
    """The dequantizing grouped GEMM at the largest shapes the interface accepts; outputs on a
    few sampled tokens."""
    c = build_case("q4-prefill-large", d=d, f=f, fs=f, T=300, seed=13, full_host=False)
    got = _run_q4(c)
    toks = [0, 1, 150, 298, 299]
    idx, _ = oracle.select(oracle.router_logits_f32(c.x[toks], c.w_r, c.bias), c.dims.k)
    assert np.array_equal(got["topk_idx"][toks], idx)
    assert_close(got["y"][toks], oracle_outputs_q4(c, toks), f"q4 prefill d={d} f={f}")


def test_q4_chunked_and_single_token_tensor_core():
    """Chunking leaves the bytes unchanged; T = 1 under the GEMM schedule goes through the
    dequantizing grouped GEMM and matches the oracle."""
    import torch
    T = 700
    c = build_case("q4-chunked", d=512, f=128, fs=256, T=T, seed=5, full_host=False)
    W = q4_to_device(c)
    x = torch.from_numpy(c.x.view(np.int16)).cuda().view(torch.bfloat16)
    L0 = moe.MoeLayer(W, T)
    L1 = moe.MoeLayer(W, T, chunk_tokens=256)
    y0, y1 = bf16_bits(L0.forward(x)), bf16_bits(L1.forward(x))
    # the host entry point over chunks (page-locked buffers: y written in place)
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    L1.forward_host(xh, yh)
    torch.cuda.synchronize()
    assert L0.device_error() == moe.MOE_OK and L1.device_error() == moe.MOE_OK
    assert np.array_equal(y0, y1)
    assert np.array_equal(bf16_bits(yh), y1)
    toks = sample_tokens(T, n_edge=16, stride=29)
    assert_close(y1[toks], oracle_outputs_q4(c, toks), "q4 chunked")
    L0.close()
    L1.close()
    c1 = build_case("q4-one", d=512, f=128, fs=256, T=1, seed=6, full_host=False)
    got = _run_q4(c1, moe.MOE_SCHEDULE_GEMM)
    assert_close(got["y"], oracle_outputs_q4(c1), "q4 T=1 tensor-core")


def test_q4_handle_limits():
    import torch
    c = build_case("q4-limits", d=512, f=128, fs=128, T=5, seed=9, full_host=False)
    W = q4_to_device(c)
    x = torch.from_numpy(c.x.view(np.int16)).cuda().view(torch.bfloat16)
    # the small-batch matrix-vector path reads bf16: GEMV with T > 1 is refused
    L = moe.MoeLayer(W, 8, schedule=moe.MOE_SCHEDULE_GEMV)
    y = torch.empty_like(x)
    assert moe.moe_forward(L.handle, x.data_ptr(), 5, y.data_ptr(), None) == \
        moe.MOE_ERR_UNSUPPORTED
    L.close()
    # AUTO: T = 5 on the tensor-core path; routing as the oracle's
    L = moe.MoeLayer(W, 8)
    y = L.forward(x)
    r = L.route(x)
    torch.cuda.synchronize()
    assert np.array_equal(r["topk_idx"].cpu().numpy(), oracle_route(c)["topk_idx"])
    assert L.device_error() == moe.MOE_OK
    assert_close(bf16_bits(y), oracle_outputs_q4(c), "q4 T=5")
    L.close()


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
