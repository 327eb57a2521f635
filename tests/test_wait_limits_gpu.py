"""Failure detection without a GPU fault: the kernels' bounded waits.

Every device wait in the library (mbarrier waits of the GEMM pipeline and of
the quantizer's bulk-copy rings, the grid barrier of the one-launch
quantizer) gives up after a time limit and records the failure instead of
spinning forever.  fos_selftest_wait_limits makes two of them run out on
purpose -- a GEMM whose producer never fills a stage, and a grid barrier that
waits for one CTA more than the launch has -- and the kernels must report
FOS_ERR_TIMEOUT and leave the CUDA context usable, which the last part checks
with a normal quantize + GEMM afterwards.
"""
import time

import numpy as np
import pytest

import workloads
from fos_testutil import to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fos():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaptive_quantization_fos_b300 as fos

    return fos


def test_waits_run_out_and_report(fos):
    import torch

    scratch = torch.empty(1 << 17, dtype=torch.uint8, device="cuda")
    result = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    st = fos.fos_selftest_wait_limits(scratch.data_ptr(), scratch.numel(), 20_000_000, result.data_ptr(), stream)
    assert st == fos.FOS_OK
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert result.cpu().tolist() == [fos.FOS_ERR_TIMEOUT, fos.FOS_ERR_TIMEOUT]
    assert elapsed < 5.0, "the waits must give up after their 20 ms limits"


def test_context_usable_after_timeouts(fos):
    import torch

    import oracle

    scratch = torch.empty(1 << 17, dtype=torch.uint8, device="cuda")
    result = torch.zeros(2, dtype=torch.int32, device="cuda")
    fos.fos_selftest_wait_limits(scratch.data_ptr(), scratch.numel(), 10_000_000, result.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    xa = workloads.activations(256, 512, seed=71)
    xw = workloads.student_t(256, 512, seed=72)
    a = fos.quantize(to_device_bf16(xa))
    w = fos.quantize(to_device_bf16(xw))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = fos.gemm(a, w, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    qa = oracle.quantize(xa)
    assert np.array_equal(a.codes[:, :256].cpu().numpy(), qa.codes)
    assert np.float32(a.tensor_scale.item()) == np.float32(qa.tensor_scale)
    ref, bnd = oracle.gemm_rows(oracle.dequantize(qa), oracle.dequantize(oracle.quantize(xw)), np.arange(256))
    c = C.float().cpu().numpy().astype(np.float64)
    assert (np.abs(c - ref) <= 1e-3 * bnd + 2.0 ** -8 * np.abs(ref)).all()


def test_selftest_rejects_bad_arguments(fos):
    assert fos.fos_selftest_wait_limits(0, 1 << 17, 1000, 1 << 20, 0) == fos.FOS_ERR_INVALID_ARG
    assert fos.fos_selftest_wait_limits(1 << 20, 1024, 1000, 1 << 20, 0) == fos.FOS_ERR_INVALID_ARG
    assert fos.fos_selftest_wait_limits(1 << 20, 1 << 17, 0, 1 << 20, 0) == fos.FOS_ERR_INVALID_ARG
