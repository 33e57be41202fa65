"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Bar: expert indices, offsets and the token permutation bit-exact; layer outputs within
max|gpu - ref| <= 2e-2 * max|ref| + 1e-3 (bf16 output, fp32 accumulation); routing weights
within 1e-5.  Inputs are seeded (synth/), x drawn under the 1e-3 logit-gap rule.
"""
import numpy as np
import pytest

import oracle
import sparse_moe_02_gb300 as moe
from _cases import (assert_close, bf16_bits, build_case, oracle_outputs, oracle_route,
                    sample_tokens, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    yield
    torch.cuda.synchronize()


def _layer(c, schedule, max_tokens=None, W=None):
    if W is None:
        W, _ = to_device(c)
    return moe.MoeLayer(W, max_tokens or max(c.T, 1), schedule=schedule), W


def _run(c, schedule, max_tokens=None):
    import torch
    W, x = to_device(c)
    L, _ = _layer(c, schedule, max_tokens, W)
    y = L.forward(x)
    r = L.route(x)
    torch.cuda.synchronize()
    assert L.device_error() == moe.MOE_OK
    out = {k: v.cpu().numpy() for k, v in r.items()}
    out["y"] = bf16_bits(y)
    L.close()
    return out


def _check_routing(c, got, tokens=None):
    ref = oracle_route(c) if tokens is None else None
    if ref is not None:
        assert np.array_equal(got["topk_idx"], ref["topk_idx"]), "topk_idx differs"
        assert np.max(np.abs(got["topk_w"] - ref["topk_w"])) <= 1e-5
        assert np.array_equal(got["offsets"], ref["offsets"]), "offsets differ"
        assert np.array_equal(got["perm"], ref["perm"]), "perm differs"
        return
    # sampled tokens: selection and weights per token; the structure by its invariants
    idx, w = oracle.select(oracle.router_logits_f32(c.x[tokens], c.w_r, c.bias), c.dims.k)
    assert np.array_equal(got["topk_idx"][tokens], idx)
    assert np.max(np.abs(got["topk_w"][tokens] - w)) <= 1e-5
    check_structure(got, c.T, c.dims.E, c.dims.k)


def check_structure(got, T, E, k):
    """perm/offsets are the stable counting sort of the GPU's own topk_idx."""
    flat = got["topk_idx"].reshape(-1).astype(np.int64)
    counts = np.bincount(flat, minlength=E)
    assert np.array_equal(got["offsets"], np.concatenate([[0], np.cumsum(counts)]))
    assert np.array_equal(got["perm"], np.argsort(flat, kind="stable"))


# ---------------------------------------------------------------- tiny layer, every token

@pytest.mark.parametrize("schedule", [moe.MOE_SCHEDULE_GEMM, moe.MOE_SCHEDULE_AUTO])
def test_tiny_layer_all_tokens(schedule):
    c = build_case("tiny", d=512, f=128, fs=128, T=64)
    got = _run(c, schedule)
    _check_routing(c, got)
    assert_close(got["y"], oracle_outputs(c), "tiny T=64")


@pytest.mark.parametrize("schedule", [moe.MOE_SCHEDULE_GEMM, moe.MOE_SCHEDULE_GEMV,
                                      moe.MOE_SCHEDULE_AUTO])
def test_single_token_both_paths(schedule):
    c = build_case("tiny-t1", d=512, f=128, fs=128, T=1, seed=3)
    got = _run(c, schedule)
    _check_routing(c, got)
    assert_close(got["y"], oracle_outputs(c), f"T=1 schedule {schedule}")


@pytest.mark.parametrize("T", [2, 77, 129, 300, 1000])
def test_ragged_token_counts(T):
    c = build_case(f"ragged-{T}", d=512, f=128, fs=256, T=T, seed=T)
    got = _run(c, moe.MOE_SCHEDULE_AUTO)
    _check_routing(c, got)
    assert_close(got["y"], oracle_outputs(c), f"T={T}")


def test_all_tokens_pick_the_same_experts():
    # zero router, bias on 8 experts: every token selects them; 248 groups stay empty and the
    # 8 busy groups (T rows each) span several 256-row chunks
    import synth
    dims = synth.Dims(d=512, f=128, fs=128)
    bias = np.zeros(256, dtype=np.float32)
    hot = [3, 40, 41, 99, 128, 200, 201, 255]
    bias[hot] = np.linspace(1.0, 2.0, 8, dtype=np.float32)
    c = build_case("same-experts", d=512, f=128, fs=128, T=600, seed=5,
                   w_r=np.zeros((256, 512), dtype=np.uint16), bias=bias)
    got = _run(c, moe.MOE_SCHEDULE_AUTO)
    _check_routing(c, got)
    assert np.all(got["topk_idx"] == np.array(hot, dtype=np.int32))
    assert_close(got["y"], oracle_outputs(c), "same experts")


# ---------------------------------------------------------------- the benchmark shapes

@pytest.mark.parametrize("schedule", [moe.MOE_SCHEDULE_GEMV, moe.MOE_SCHEDULE_GEMM])
@pytest.mark.parametrize("layer", [0, 17, 39])
def test_decode_layer(layer, schedule):
    # batch-1 decode, d=2048, f=fs=512; weights generated on the device, oracle side only the
    # selected experts on the host
    c = build_case("decode", d=2048, f=512, fs=512, T=1, seed=0, layer=layer, full_host=False)
    got = _run(c, schedule)
    _check_routing(c, got)
    assert_close(got["y"], oracle_outputs(c), f"decode layer {layer}")


# Batch-1 decode at other sizes: the largest expert inner dimension (d=4096, f=2048) and a
# wide hidden size (d=8192, f=512).
@pytest.mark.parametrize("d,f", [(4096, 2048), (8192, 512)])
def test_decode_other_shapes(d, f):
    c = build_case("decode-shapes", d=d, f=f, fs=f, T=1, seed=5, full_host=False)
    got = _run(c, moe.MOE_SCHEDULE_GEMV)
    _check_routing(c, got)
    assert_close(got["y"], oracle_outputs(c), f"decode d={d} f={f}")


# The tensor-core path at the largest shapes the interface accepts (d = 8192 with f = 512;
# d = 4096 with f = fs = 2048): 128-step K loops, 16 gate/up weight tiles per group; outputs
# on a few sampled tokens (the oracle needs only their experts' weights).
@pytest.mark.parametrize("d,f", [(8192, 512), (4096, 2048)])
def test_prefill_largest_shapes(d, f):
    c = build_case("prefill-large", d=d, f=f, fs=f, T=300, seed=12, full_host=False)
    got = _run(c, moe.MOE_SCHEDULE_GEMM)
    toks = [0, 1, 150, 298, 299]
    _check_routing(c, got, toks)
    assert_close(got["y"][toks], oracle_outputs(c, toks), f"prefill d={d} f={f}")


# Batch-1 decode where the shared expert's inner dim differs from the routed one and d is not
# a power of two (rows end in a partial 4 KB chunk, blocks get uneven shares).
@pytest.mark.parametrize("d,f,fs", [(640, 128, 384), (2176, 384, 128)])
def test_decode_ragged_shapes(d, f, fs):
    c = build_case("decode-ragged", d=d, f=f, fs=fs, T=1, seed=d, full_host=False)
    got = _run(c, moe.MOE_SCHEDULE_GEMV)
    _check_routing(c, got)
    assert_close(got["y"], oracle_outputs(c), f"decode d={d} f={f} fs={fs}")


def test_decode_repeated_and_interleaved_launches():
    # the layer launch keeps its grid-barrier counters in the handle and resets them on exit:
    # back-to-back launches on one handle, and two handles' launches interleaved on one
    # stream, all give the same bytes
    import torch
    cs = [build_case("decode-rep", d=2048, f=512, fs=512, T=1, seed=0, layer=l, full_host=False)
          for l in (3, 4)]
    Ls, xs = [], []
    for c in cs:
        W, x = to_device(c)
        Ls.append(moe.MoeLayer(W, 1, schedule=moe.MOE_SCHEDULE_GEMV))
        xs.append(x)
    first = [bf16_bits(L.forward(x)) for L, x in zip(Ls, xs)]
    for _ in range(5):
        for i, (L, x) in enumerate(zip(Ls, xs)):
            assert np.array_equal(bf16_bits(L.forward(x)), first[i])
    torch.cuda.synchronize()
    for L, c, y in zip(Ls, cs, first):
        assert L.device_error() == moe.MOE_OK
        assert_close(y, oracle_outputs(c), "decode repeated")
        L.close()


@pytest.mark.parametrize("skew", [False, True], ids=["balanced", "skewed"])
def test_prefill_4096(skew):
    c = build_case("prefill", d=2048, f=512, fs=512, T=4096, seed=0, skew=skew)
    got = _run(c, moe.MOE_SCHEDULE_AUTO)
    _check_routing(c, got)
    counts = np.diff(got["offsets"])
    if skew:
        assert counts.max() > 1000 and (counts == 0).sum() > 0
    else:
        assert counts.min() > 64 and counts.max() < 256
    assert_close(got["y"], oracle_outputs(c), f"prefill skew={skew} (all 4096 tokens)")


# The prefill length sweep of the benchmark (T = 256 .. 128K at d = 2048, f = fs = 512,
# balanced routing), in the launch configuration the benchmark times: expert ids, offsets and
# the token permutation bit-exact against the oracle's routing of every token; outputs against
# the oracle on every token up to T = 4096 and above on the first and last 64 tokens plus every
# 17th (the oracle takes about 1.5 ms per token on 16 cores).
@pytest.mark.parametrize("T", [256, 512, 1024, 2048, 8192, 16384, 32768, 65536, 131072])
def test_prefill_sweep_sizes(T):
    c = build_case("sweep", d=2048, f=512, fs=512, T=T, seed=11, full_host=False)
    got = _run(c, moe.MOE_SCHEDULE_AUTO)
    _check_routing(c, got)
    toks = np.arange(T) if T <= 4096 else sample_tokens(T)
    assert_close(got["y"][toks], oracle_outputs(c, toks), f"sweep T={T}")


# The plan and scatter run as one launch up to 128 token blocks (T <= 16384) and as two
# launches above; both sides of that switch, routing checked on sampled tokens plus the
# counting-sort invariants over every token.
@pytest.mark.parametrize("T", [16384, 16385, 32768])
def test_prefill_plan_paths(T):
    c = build_case("plan-paths", d=512, f=128, fs=128, T=T, seed=21, full_host=False)
    got = _run(c, moe.MOE_SCHEDULE_AUTO)
    toks = sample_tokens(T, n_edge=16, stride=251)
    _check_routing(c, got, toks)
    assert_close(got["y"][toks], oracle_outputs(c, toks), f"plan paths T={T}")


# In-layer token chunking: the layer over chunks of at most chunk_tokens tokens (the expert
# buffers sized for one chunk) gives exactly the bytes of the unchunked layer, through the
# device and the host entry points; outputs checked against the oracle on sampled tokens.
@pytest.mark.parametrize("chunk", [1000, 2048])
def test_chunked_forward_is_byte_identical(chunk):
    import torch
    T = 4500
    c = build_case("chunked", d=512, f=128, fs=256, T=T, seed=31)
    W, x = to_device(c)
    L0 = moe.MoeLayer(W, T)
    L1 = moe.MoeLayer(W, T, chunk_tokens=chunk)
    y0 = bf16_bits(L0.forward(x))
    y1 = bf16_bits(L1.forward(x))
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    L1.forward_host(xh, yh)
    torch.cuda.synchronize()
    assert L0.device_error() == moe.MOE_OK and L1.device_error() == moe.MOE_OK
    assert np.array_equal(y0, y1)
    assert np.array_equal(bf16_bits(yh), y1)
    toks = sample_tokens(T, n_edge=16, stride=61)
    assert_close(y1[toks], oracle_outputs(c, toks), f"chunked T={T} chunk={chunk}")
    L0.close()
    L1.close()


@pytest.mark.parametrize("chunk", [3000, 4096])
def test_chunked_forward_at_the_benchmark_shape(chunk):
    # d = 2048, f = fs = 512, 8192 tokens in chunks of 3000 (a ragged last chunk) or 4096:
    # every token is computed independently, so the output is the unchunked output, byte for
    # byte
    T = 8192
    c = build_case("chunked-bench", d=2048, f=512, fs=512, T=T, seed=37, full_host=False)
    W, x = to_device(c)
    L0 = moe.MoeLayer(W, T)
    L1 = moe.MoeLayer(W, T, chunk_tokens=chunk)
    y0 = bf16_bits(L0.forward(x))
    y1 = bf16_bits(L1.forward(x))
    assert L0.device_error() == moe.MOE_OK and L1.device_error() == moe.MOE_OK
    assert np.array_equal(y0, y1)
    toks = sample_tokens(T, n_edge=8, stride=257)
    assert_close(y1[toks], oracle_outputs(c, toks), f"chunked T={T} chunk={chunk}")
    L0.close()
    L1.close()


# ---------------------------------------------------------------- API behaviour on the GPU

def test_deterministic_and_host_entry_point():
    import torch
    c = build_case("det", d=512, f=128, fs=128, T=333, seed=9)
    W, x = to_device(c)
    L = moe.MoeLayer(W, 400)
    y1 = bf16_bits(L.forward(x))
    y2 = bf16_bits(L.forward(x))
    assert np.array_equal(y1, y2)
    xh = x.cpu().pin_memory()
    # pinned y: written in place by the layer's last kernel
    yh = torch.empty_like(xh).pin_memory()
    L.forward_host(xh, yh)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(yh), y1)
    # pageable x and y, and pinned y that is not 16-byte aligned: copied by the copy engine
    yp = torch.empty_like(xh)
    L.forward_host(x.cpu(), yp)
    buf = torch.zeros(xh.numel() * 2 + 16, dtype=torch.uint8).pin_memory()
    yo = buf[2:2 + xh.numel() * 2].view(torch.bfloat16).view(xh.shape)
    L.forward_host(xh, yo)
    # batch-1 decode through the host entry point (the decode kernel writes y in place)
    y1h = torch.empty_like(xh[:1]).pin_memory()
    L.forward_host(xh[:1], y1h)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(yp), y1)
    assert np.array_equal(bf16_bits(yo), y1)
    assert np.array_equal(bf16_bits(y1h), bf16_bits(L.forward(x[:1])))
    assert L.device_error() == moe.MOE_OK
    # T = 0 is a no-op; T beyond max_tokens is rejected before any launch
    assert moe.moe_forward(L.handle, x.data_ptr(), 0, x.data_ptr(), None) == moe.MOE_OK
    assert moe.moe_forward(L.handle, x.data_ptr(), 401, x.data_ptr(), None) == \
        moe.MOE_ERR_UNSUPPORTED
    y = torch.empty_like(x)
    assert moe.moe_forward(L.handle, x.data_ptr() + 2, 10, y.data_ptr(), None) == \
        moe.MOE_ERR_ALIGNMENT
    assert moe.moe_forward(L.handle, x.data_ptr(), 10, x.data_ptr(), None) == \
        moe.MOE_ERR_INVALID_ARG  # y aliases x
    L.close()


def test_gemv_schedule_rejects_shapes_it_does_not_fit():
    import torch
    c = build_case("gemv-t9", d=512, f=128, fs=128, T=9, seed=4)
    W, x = to_device(c)
    L = moe.MoeLayer(W, 16, schedule=moe.MOE_SCHEDULE_GEMV)
    y = torch.empty_like(x)
    assert moe.moe_forward(L.handle, x.data_ptr(), 9, y.data_ptr(), None) == \
        moe.MOE_ERR_UNSUPPORTED
    L.close()
    # 3 tokens x max(f, fs) = 2048 is past the per-block h copy: GEMV rejects, AUTO falls back
    c = build_case("gemv-wide", d=512, f=2048, fs=128, T=3, seed=4, full_host=False)
    W, x = to_device(c)
    L = moe.MoeLayer(W, 3, schedule=moe.MOE_SCHEDULE_GEMV)
    y = torch.empty_like(x)
    assert moe.moe_forward(L.handle, x.data_ptr(), 3, y.data_ptr(), None) == \
        moe.MOE_ERR_UNSUPPORTED
    L.close()
    got = _run(c, moe.MOE_SCHEDULE_AUTO)
    _check_routing(c, got)
    assert_close(got["y"], oracle_outputs(c), "wide T=3 through the tensor-core path")


# Small batches (2..8 tokens, the speculative-verify shape): the matrix-vector path over the
# union of the tokens' experts, routing bit-exact and outputs within tolerance, against the
# oracle; the same tokens through the tensor-core path agree too.  Every T: the small-batch
# kernels are compiled once per token count.
@pytest.mark.parametrize("T", [2, 3, 4, 5, 6, 7, 8])
def test_small_batch_decode(T):
    c = build_case("small-batch", d=512, f=128, fs=256, T=T, seed=40 + T)
    for sched in (moe.MOE_SCHEDULE_GEMV, moe.MOE_SCHEDULE_AUTO, moe.MOE_SCHEDULE_GEMM):
        got = _run(c, sched)
        _check_routing(c, got)
        assert_close(got["y"], oracle_outputs(c), f"small batch T={T} schedule {sched}")


@pytest.mark.parametrize("T", [2, 4, 5])
def test_small_batch_decode_shape(T):
    # the benchmark's decode dimensions, d=2048, f=fs=512, through the matrix-vector path and
    # the default schedule (the tensor-core path routed and planned by the small router)
    c = build_case("small-batch-decode", d=2048, f=512, fs=512, T=T, seed=7, layer=T,
                   full_host=False)
    for sched in (moe.MOE_SCHEDULE_GEMV, moe.MOE_SCHEDULE_AUTO):
        got = _run(c, sched)
        _check_routing(c, got)
        assert_close(got["y"], oracle_outputs(c), f"small batch decode T={T} schedule {sched}")


def test_two_tokens_run_once_per_token():
    """AUTO runs two bf16 tokens as one single-token pass each: the outputs are those of two
    single-token calls byte for byte, and moe_route's selection and weights for the pair
    equal the single-token routes bit for bit."""
    import torch
    c = build_case("two-tokens", d=2048, f=512, fs=512, T=2, seed=8, full_host=False)
    W, x = to_device(c)
    L = moe.MoeLayer(W, 2)
    y2 = bf16_bits(L.forward(x))
    y0, y1 = bf16_bits(L.forward(x[:1])), bf16_bits(L.forward(x[1:2]))
    r2, r0, r1 = L.route(x), L.route(x[:1]), L.route(x[1:2])
    torch.cuda.synchronize()
    assert L.device_error() == moe.MOE_OK
    assert np.array_equal(y2, np.concatenate([y0, y1]))
    for k in ("topk_idx", "topk_w"):
        both = r2[k].cpu().numpy()
        assert np.array_equal(both, np.concatenate([r0[k].cpu().numpy(), r1[k].cpu().numpy()]))
    _check_routing(c, {k: v.cpu().numpy() for k, v in r2.items()})
    assert_close(y2, oracle_outputs(c), "two tokens")
    L.close()


def test_read_probe_hook():
    import torch
    buf = torch.ones(1 << 20, dtype=torch.bfloat16, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert moe.moe_read_probe(buf.data_ptr(), 2 << 20, sink.data_ptr(), s) == moe.MOE_OK
    assert moe.moe_read_probe(buf.data_ptr() + 8, 1024, sink.data_ptr(), s) == \
        moe.MOE_ERR_INVALID_ARG
    assert moe.moe_read_probe(buf.data_ptr(), 1000, sink.data_ptr(), s) == moe.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
