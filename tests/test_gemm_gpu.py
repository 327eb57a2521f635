"""Parity of the block-scaled tcgen05 NVFP4 GEMM with the oracle.

The oracle's reference is the FP32-simulation path of the "Four Over Six" page
(first section): dequantize both operands (x_hat = g * (sf * s_t)), then
multiply, here with FP64 sums.  The bar, per output element:
|C - C_ref| <= 1e-3 * sum_k |a_hat_k| |w_hat_k| + 2^-8 |C_ref|.
The first term bounds the accumulation; the second is the unit roundoff of the
bf16 output (8-bit significand, round to nearest even), which alone exceeds
the first term whenever a few products dominate an output (|C| close to
sum |a||w|), as in rows with outlier channels.

Operands for the GEMM-only cases are quantized by the oracle and uploaded, so
these tests do not depend on the CUDA quantizer; the end-to-end cases quantize
on the GPU and first check those codes against the oracle bit for bit.
"""
import numpy as np
import pytest

import workloads
from fos_testutil import assert_same, gpu_quantize, mixed_bits, oracle_quantize

pytestmark = pytest.mark.gpu

REL_TOL = 1e-3
BF16_UNIT_ROUNDOFF = 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaptive_quantization_fos_b300  # noqa: F401  (fails loudly if libfos.so is missing)


def upload(q):
    """An oracle QResult -> device NVFP4Tensor (rows padded to 16-byte strides)."""
    import torch

    import adaptive_quantization_fos_b300 as fos

    R, C = q.rows, q.cols
    ld = max(16, ((C // 2 + 15) // 16) * 16)
    codes = torch.zeros((R, ld), dtype=torch.uint8)
    codes[:, : C // 2] = torch.from_numpy(np.ascontiguousarray(q.codes[:, : C // 2]))
    return fos.NVFP4Tensor(codes=codes.cuda(), sf=torch.from_numpy(q.sf.copy()).cuda(),
                           tensor_scale=torch.tensor([q.tensor_scale], dtype=torch.float32).cuda(),
                           rows=R, cols=C, sf_layout=q.sf_layout)


def run_gemm(a, w):
    import torch

    import adaptive_quantization_fos_b300 as fos

    C = torch.full((a.rows, w.rows), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fos.gemm(a, w, out=C, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "the kernel reported a wait timeout"
    return C


def check_rows(C, A_hat, W_hat, rows, matmul=False):
    import oracle

    ref, bnd = (oracle.gemm_rows_matmul if matmul else oracle.gemm_rows)(A_hat, W_hat, rows)
    c = C[rows].float().cpu().numpy().astype(np.float64)
    assert np.isfinite(c).all(), "non-finite output"
    err = np.abs(c - ref)
    tol = REL_TOL * bnd + BF16_UNIT_ROUNDOFF * np.abs(ref)
    bad = np.argwhere(err > tol)
    worst = float(np.max(err / np.maximum(tol, 1e-300)))
    assert bad.size == 0, f"{len(bad)} elements outside the bound, first {bad[:4].tolist()}, worst err/tol {worst:.3g}"


SHAPES = [
    (128, 256, 256),    # one 128 x 256 tile, one stage
    (256, 512, 1024),   # 2 x 2 tiles, 4 stages
    (200, 384, 320),    # ragged M; 128-column tiles; K = 5 MMAs (partial last stage)
    (136, 264, 192),    # 128-column tiles with an 8-column tail; K = 3 MMAs
    (72, 456, 64),      # M < 128; 256-column tiles with a 200-column tail; one MMA
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_oracle_operands(M, N, K):
    import oracle

    qa = oracle.quantize(mixed_bits(M, K, seed=M + K))
    qw = oracle.quantize(workloads.student_t(N, K, seed=N + 7 * K))
    C = run_gemm(upload(qa), upload(qw))
    check_rows(C, oracle.dequantize(qa), oracle.dequantize(qw), np.arange(M))


def test_gemm_options_and_zero_rows():
    """Operands from stochastic rounding, 2D tiles and the RHT all feed the same
    GEMM; rows of zeros must give exact zeros."""
    import oracle

    M, N, K = 256, 256, 512
    xa = mixed_bits(M, K, seed=5)
    xa[17] = 0
    qa = oracle.quantize(xa, rounding=oracle.ROUND_SR, sr_seed=99, hadamard=True, hadamard_seed=4)
    qw = oracle.quantize(workloads.student_t(N, K, seed=6), block_2d=True, hadamard=True, hadamard_seed=4)
    C = run_gemm(upload(qa), upload(qw))
    assert not C[17].float().abs().max().item()
    check_rows(C, oracle.dequantize(qa), oracle.dequantize(qw), np.arange(M))


@pytest.mark.parametrize("N,ld,off", [(264, 272, 0), (256, 264, 0), (384, 400, 0), (256, 272, 8)])
def test_gemm_output_inside_wider_rows(N, ld, off):
    """C as a view into wider rows, starting `off` columns in: 32-byte stores
    where C's start and row stride allow them (32-byte aligned, ld % 16 == 0),
    16-byte stores otherwise (off = 8: a 16-byte aligned start) and at a ragged
    right edge; the columns outside C must stay untouched."""
    import torch

    import adaptive_quantization_fos_b300 as fos
    import oracle

    M, K = 200, 256
    qa = oracle.quantize(mixed_bits(M, K, seed=N + ld))
    qw = oracle.quantize(workloads.student_t(N, K, seed=N + 2 * ld))
    full = torch.full((M, ld), float("nan"), dtype=torch.bfloat16, device="cuda")
    C = full[:, off:off + N]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fos.gemm(upload(qa), upload(qw), out=C, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.isnan(full[:, :off]).all() and torch.isnan(full[:, off + N:]).all(), "columns outside C were written"
    check_rows(C, oracle.dequantize(qa), oracle.dequantize(qw), np.arange(M))


def test_gemm_many_tiles_per_cta():
    """More output tiles than SMs: each persistent CTA runs several tiles and
    the accumulator barrier phases wrap."""
    import oracle

    M, N, K = 2048, 2560, 512
    qa = oracle.quantize(workloads.activations(M, K, seed=11))
    qw = oracle.quantize(workloads.student_t(N, K, seed=12))
    C = run_gemm(upload(qa), upload(qw))
    rows = np.unique(np.concatenate([np.arange(0, M, 61), np.arange(M - 130, M)]))
    check_rows(C, oracle.dequantize(qa), oracle.dequantize(qw), rows)


def test_linear_forward_small_end_to_end():
    """GPU quantize (4/6, 1D, RNE) -> GPU GEMM against oracle quantize ->
    dequantize -> FP64 product."""
    import adaptive_quantization_fos_b300 as fos
    import oracle
    from fos_testutil import to_device_bf16

    xa = workloads.activations(384, 1024, seed=21)
    xw = workloads.student_t(768, 1024, seed=22)
    assert_same(gpu_quantize(xa), oracle_quantize(xa), "A")
    assert_same(gpu_quantize(xw), oracle_quantize(xw), "W")
    a = fos.quantize(to_device_bf16(xa))
    w = fos.quantize(to_device_bf16(xw))
    C = run_gemm(a, w)
    check_rows(C, oracle.dequantize(oracle.quantize(xa)), oracle.dequantize(oracle.quantize(xw)), np.arange(384))


def test_linear_forward_full_size_sampled_rows():
    """The 8192 x 12288 x 4096 linear forward: A (activation recipe) and W
    (weight recipe) quantized on the GPU -- codes, scales and s_t bit-exact
    against the oracle -- then the GEMM, checked on 256 seeded rows x all
    12288 columns."""
    import adaptive_quantization_fos_b300 as fos
    import oracle
    from fos_testutil import QOut, to_device_bf16

    xa = workloads.activations(8192, 4096, seed=5001)
    xw = workloads.student_t(12288, 4096, seed=5002)
    a = fos.quantize(to_device_bf16(xa))
    w = fos.quantize(to_device_bf16(xw))
    C = run_gemm(a, w)
    qa, qw = oracle.quantize(xa), oracle.quantize(xw)
    for name, g, o in (("A", a, qa), ("W", w, qw)):
        got = QOut(codes=g.codes[:, : g.cols // 2].cpu().numpy(), sf=g.sf.cpu().numpy(),
                   s_t=np.float32(g.tensor_scale.item()), choice=None)
        want = QOut(codes=np.ascontiguousarray(o.codes), sf=o.sf, s_t=np.float32(o.tensor_scale), choice=None)
        assert_same(got, want, name)
    rows = np.sort(np.random.default_rng(5003).choice(8192, 256, replace=False))
    check_rows(C, oracle.dequantize(qa), oracle.dequantize(qw), rows, matmul=True)
