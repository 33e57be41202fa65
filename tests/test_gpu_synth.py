"""The device fill of the seeded generator gives the same bits as the host generator."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def test_device_fill_equals_host():
    import torch
    for seed, stream, offset, n, sigma in [(0, synth.stream_id(synth.W_GATE, 3), 12345, 100003, 0.02),
                                           (7, synth.stream_id(synth.X, 0, 2), 0, 4096, 1.0),
                                           (1, 99, (1 << 33) + 5, 777, 0.05)]:
        t = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        synth.normal_bf16_device(seed, stream, offset, n, sigma, t.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        dev = t.cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(dev, synth.normal_bf16(seed, stream, offset, n, sigma))
