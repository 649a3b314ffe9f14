"""The FFMA throughput probe (the denominator of the FFMA-bound roofline)
runs, reports the FMAs it launched, and measures a plausible binary32 rate
for a GPU of this size (tens of TFLOP/s)."""
import pytest

from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu


def test_ffma_probe_counts_and_rate():
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sink = torch.zeros(sms * 4, dtype=torch.float32, device="cuda")
    n = qsa.qsa_probe_ffma(4, 64, sink)
    assert n == sms * 4 * 256 * 64 * 16 * 8
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    n = qsa.qsa_probe_ffma(4, 256, sink)
    e1.record()
    torch.cuda.synchronize()
    tflops = 2 * n / (e0.elapsed_time(e1) * 1e-3) / 1e12
    assert 5.0 < tflops < 500.0, tflops
    assert not sink.any()  # the guard store never fires
