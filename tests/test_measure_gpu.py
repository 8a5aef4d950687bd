"""The FFMA-rate measurement aid (coalesce_measure_ffma) that the bench's FP32
roofline is taken against: it runs, reports the FLOP it performs for the
device's SM count, and measures a rate within the FP32 lanes' nominal bound."""
import ctypes

import pytest
import torch

import gemm_bias_activation_gb300 as g

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g.build()
    g.load_library()
    torch.cuda.set_device(0)


def test_measure_ffma_counts_and_rate():
    lib = g.load_library()
    s = torch.cuda.current_stream()
    sink = torch.zeros(1, dtype=torch.float32, device="cuda")
    flop = ctypes.c_double(0.0)
    iters = 1 << 16
    assert lib.coalesce_measure_ffma(iters, ctypes.c_void_p(sink.data_ptr()), ctypes.byref(flop),
                                     ctypes.c_void_p(s.cuda_stream)) == 0   # warm-up
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    assert lib.coalesce_measure_ffma(iters, ctypes.c_void_p(sink.data_ptr()), ctypes.byref(flop),
                                     ctypes.c_void_p(s.cuda_stream)) == 0
    e1.record(s)
    assert g.coalesce_device_status(s.cuda_stream) == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # 4 blocks of 256 threads per SM, 16 chains of `iters` FMAs each, 2 FLOP per FMA
    assert flop.value == 2.0 * 4 * sms * 256 * 16 * iters
    rate = flop.value / (e0.elapsed_time(e1) / 1e3) / 1e12
    # below the lanes' bound at the highest clock a GB300 runs (128 lanes x 2 FLOP x 2.1 GHz per SM)
    assert 0.0 < rate <= sms * 128 * 2 * 2.1e9 / 1e12, rate
    assert sink.item() == 0.0  # the kernel's guard store never fires
