"""Failure detection without a GPU fault: a kernel wait that runs out of time.

The streamed batch-1 decode launch meets at a grid-wide barrier (a counter every block
increments, polled with a time limit).  moe_test_expire_waits makes the next call's barrier
wait for one block more than the launch has, with a 1 ms limit: every block gives up, records
MOE_ERR_TIMEOUT in the handle's device error word and leaves after its own copies have landed
(no copy and no tensor-core operation is in flight when a block exits).  The test checks that
moe_get_device_error reports the timeout once, and that the next forward on the same handle is
back within the parity tolerance of the oracle with a clean error word.
"""
import numpy as np
import pytest

import sparse_moe_02_gb300 as moe
from _cases import assert_close, bf16_bits, build_case, oracle_outputs, to_device

pytestmark = pytest.mark.gpu


def test_grid_barrier_timeout_is_reported_and_the_handle_recovers():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    c = build_case("expire", d=512, f=128, fs=128, T=1, seed=5)
    W, x = to_device(c)
    layer = moe.MoeLayer(W, 1, schedule=moe.MOE_SCHEDULE_GEMV)
    ref = oracle_outputs(c)
    y = layer.forward(x)
    assert layer.device_error() == moe.MOE_OK
    assert_close(bf16_bits(y), ref, "before the expired wait")

    assert moe.moe_test_expire_waits(layer.handle, 1) == moe.MOE_OK
    layer.forward(x)
    assert layer.device_error() == moe.MOE_ERR_TIMEOUT
    assert layer.device_error() == moe.MOE_OK  # read and cleared

    y2 = layer.forward(x)
    assert layer.device_error() == moe.MOE_OK
    assert_close(bf16_bits(y2), ref, "after the expired wait")
    assert np.array_equal(bf16_bits(y2), bf16_bits(y))  # deterministic again
    layer.close()
