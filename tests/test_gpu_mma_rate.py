"""The tensor-core rate hook (sage_measure_mma_rate): every mode runs to completion on every SM with
a clean status, and its rate lies between a sanity floor and the nominal peak of its kind -- the
ceiling the attention roofline is read against."""
import pytest
import torch

import video_diffusion_transformer_sage_gb300 as sage
from video_diffusion_transformer_sage_gb300 import _lib

pytestmark = pytest.mark.gpu

# Nominal dense FLOP per clock per SM: 8192 for 16-bit operands, 16384 for E4M3; modes 2 and 6
# are the attention's per-tile mixes (D = 128, D = 64), half of their FLOPs of each kind.
MIX = 1.0 / (0.5 / 8192 + 0.5 / 16384)
NOMINAL_PER_CLK = {0: 8192, 1: 16384, 2: MIX, 3: 16384, 4: 8192, 5: 16384, 6: MIX}


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4, 5, 6])
def test_mma_rate_modes(mode):
    props = torch.cuda.get_device_properties(0)
    sms = props.multi_processor_count
    status = sage.status_block()
    iters = 2000
    sage.sage_measure_mma_rate(mode, iters, sms, status)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    sage.sage_measure_mma_rate(mode, iters, sms, status)
    b.record()
    torch.cuda.synchronize()
    assert sage.sage_check_device_status(status) == (0, 0)
    ms = a.elapsed_time(b)
    tflops = _lib.MMA_RATE_FLOPS[mode] * iters * sms / (ms * 1e-3) / 1e12
    peak = NOMINAL_PER_CLK[mode] * sms * 2.2e9 / 1e12      # above the 2070 MHz maximum clock
    assert 0.2 * peak < tflops < peak, (mode, tflops, peak)


def test_mma_rate_rejects_bad_arguments():
    status = sage.status_block()
    L = _lib.lib()
    assert L.sage_measure_mma_rate(7, 10, 1, status.data_ptr(), None) == 1
    assert L.sage_measure_mma_rate(0, 0, 1, status.data_ptr(), None) == 1
    assert L.sage_measure_mma_rate(0, 10, 0, status.data_ptr(), None) == 1
    assert L.sage_measure_mma_rate(0, 10, 1, None, None) == 1
