"""The tensor-pipe rate probe (fos_selftest_mma_rate): it runs, reports no
timeout, and its rate for the GEMM's MMA instruction is a plausible FP4
figure for one B300 -- above what the GEMM itself reaches on the same part
and below the nominal dense FP4 peak with margin (13.5 PFLOP/s)."""
import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_cols", [128, 256])
def test_mma_rate_probe(n_cols):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaptive_quantization_fos_b300 as fos

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()
    iters = 4096
    assert fos.fos_selftest_mma_rate(n_cols, 16, sms, status.data_ptr(), s.cuda_stream) == fos.FOS_OK  # warm-up
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    assert fos.fos_selftest_mma_rate(n_cols, iters, sms, status.data_ptr(), s.cuda_stream) == fos.FOS_OK
    e1.record(s)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    flops = 2.0 * 128 * n_cols * 64 * 4 * iters * sms
    tflops = flops / (e0.elapsed_time(e1) * 1e-3) / 1e12
    assert 1000.0 < tflops < 15000.0, tflops
