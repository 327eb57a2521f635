"""Parity of the MXFP4 contraction (fos_gemm_mxfp4) with the oracle.

The reference is the product of the oracle's dequantized MXFP4 operands
(x_hat = g * 2^X, reading R12), summed in FP64: the FP32-simulation path of the
"Four Over Six" page (first section) applied to the FP4 glossary page's MXFP4
format ("FP4 Nasıl Çalışır": 32 values under one power-of-two scale).  The bar
is the NVFP4 GEMM's, per output element:
|C - C_ref| <= 1e-3 * sum_k |a_hat_k| |w_hat_k| + 2^-8 |C_ref|.

The GEMM-only cases upload operands quantized by the oracle, so they do not
depend on the CUDA quantizer; K of 64 or 192 modulo 128 puts half a scale
chunk (128 values of K) in the last stage.  The end-to-end case quantizes on
the GPU and first checks those operands against the oracle bit for bit.
"""
import numpy as np
import pytest

import workloads
from fos_testutil import mixed_bits, to_device_bf16

pytestmark = pytest.mark.gpu

REL_TOL = 1e-3
BF16_UNIT_ROUNDOFF = 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaptive_quantization_fos_b300  # noqa: F401  (fails loudly if libfos.so is missing)


def upload(o):
    """An oracle MXResult -> device MXFP4Tensor: codes in 16-byte rows, scales
    scattered into the 128x4 tiles (pads zero)."""
    import torch

    import adaptive_quantization_fos_b300 as fos
    import oracle

    R, C = o.rows, o.cols
    nb = C // 32
    ld = max(16, ((C // 2 + 15) // 16) * 16)
    codes = np.zeros((R, ld), np.uint8)
    codes[:, : C // 2] = o.codes
    size = oracle.sf_bytes(R, nb)
    where = oracle.sf_to_rowmajor(np.arange(size), R, nb)  # byte offset of each (row, block)
    sf = np.zeros(size, np.uint8)
    sf[where] = o.scales
    return fos.MXFP4Tensor(codes=torch.from_numpy(codes).cuda(), scales=torch.from_numpy(sf).cuda(), rows=R,
                           cols=C, sf_layout=fos.FOS_SF_SWIZZLED_128x4)


def run_gemm(a, w):
    import torch

    import adaptive_quantization_fos_b300 as fos

    C = torch.full((a.rows, w.rows), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fos.gemm_mxfp4(a, w, out=C, status=status)
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
    (128, 256, 256),    # one 128 x 256 tile, one stage (two scale chunks)
    (256, 512, 1024),   # 2 x 2 tiles, 4 stages
    (200, 384, 320),    # ragged M; 128-column tiles; K = 5 MMAs: the last chunk half used
    (136, 264, 192),    # 128-column tiles with an 8-column tail; K = 3 MMAs
    (72, 456, 64),      # M < 128; 256-column tiles with a 200-column tail; one MMA
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_mx_oracle_operands(M, N, K):
    import oracle

    qa = oracle.quantize_mx(mixed_bits(M, K, seed=M + K))
    qw = oracle.quantize_mx(workloads.student_t(N, K, seed=N + 7 * K))
    C = run_gemm(upload(qa), upload(qw))
    check_rows(C, oracle.dequantize_mx(qa), oracle.dequantize_mx(qw), np.arange(M))


def test_gemm_mx_scale_per_32_values():
    """Each 32-value scale must reach both 16-value halves of its block and no
    other block: one row of A with a different power of two in every block
    against B rows that pick out single blocks, and the 6-only / 4-only rules."""
    import oracle

    M, N, K = 128, 256, 512
    x = np.ones((M, K), np.float32)
    x *= (2.0 ** (np.arange(K) // 32 - 8))[None, :].astype(np.float32)  # block b of every row: 2^(b-8)
    x[1::2] *= -1.5
    w = np.zeros((N, K), np.float32)
    for n in range(N):
        k = (7 * n) % K
        w[n, k] = 1.0 + (n % 3)  # a single value: picks out one half of one block of A
    for rule in (0, 1, 2):
        qa = oracle.quantize_mx(workloads.bf16_bits(x), scale_rule=rule)
        qw = oracle.quantize_mx(workloads.bf16_bits(w), scale_rule=rule)
        C = run_gemm(upload(qa), upload(qw))
        A_hat, W_hat = oracle.dequantize_mx(qa), oracle.dequantize_mx(qw)
        check_rows(C, A_hat, W_hat, np.arange(M))
        # these products are exact in bf16: the result must be the FP64 product itself
        ref = A_hat.astype(np.float64) @ W_hat.astype(np.float64).T
        assert np.array_equal(C.float().cpu().numpy(), ref.astype(np.float32)), f"rule {rule}"


@pytest.mark.parametrize("N,ld,off", [(264, 272, 0), (256, 272, 8)])
def test_gemm_mx_output_inside_wider_rows(N, ld, off):
    """The MXFP4 contraction's C as a view into wider rows: the 32-byte stores
    with a ragged last group, and the 16-byte path from a start that is only
    16-byte aligned; the columns outside C stay untouched."""
    import torch

    import adaptive_quantization_fos_b300 as fos
    import oracle

    M, K = 200, 256
    qa = oracle.quantize_mx(mixed_bits(M, K, seed=N + ld + off))
    qw = oracle.quantize_mx(workloads.student_t(N, K, seed=N + 3 * ld))
    full = torch.full((M, ld), float("nan"), dtype=torch.bfloat16, device="cuda")
    C = full[:, off:off + N]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fos.gemm_mxfp4(upload(qa), upload(qw), out=C, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.isnan(full[:, :off]).all() and torch.isnan(full[:, off + N:]).all(), "columns outside C were written"
    check_rows(C, oracle.dequantize_mx(qa), oracle.dequantize_mx(qw), np.arange(M))


def test_gemm_mx_many_tiles_per_cta():
    """More output tiles than SMs: each persistent CTA runs several tiles."""
    import oracle

    M, N, K = 2048, 2560, 512
    qa = oracle.quantize_mx(workloads.activations(M, K, seed=11))
    qw = oracle.quantize_mx(workloads.student_t(N, K, seed=12))
    C = run_gemm(upload(qa), upload(qw))
    rows = np.unique(np.concatenate([np.arange(0, M, 61), np.arange(M - 130, M)]))
    check_rows(C, oracle.dequantize_mx(qa), oracle.dequantize_mx(qw), rows)


def test_gemm_mx_full_size_sampled_rows():
    """The 8192 x 12288 x 4096 contraction from MXFP4 operands quantized on the
    GPU (activation and weight recipes; codes and swizzled scales bit-exact
    against the oracle), checked on 256 seeded rows x all 12288 columns."""
    import adaptive_quantization_fos_b300 as fos
    import oracle

    xa = workloads.activations(8192, 4096, seed=5001)
    xw = workloads.student_t(12288, 4096, seed=5002)
    a = fos.quantize_mxfp4(to_device_bf16(xa))
    w = fos.quantize_mxfp4(to_device_bf16(xw))
    C = run_gemm(a, w)
    qa, qw = oracle.quantize_mx(xa), oracle.quantize_mx(xw)
    for name, g, o in (("A", a, qa), ("W", w, qw)):
        assert np.array_equal(g.codes[:, : g.cols // 2].cpu().numpy(), o.codes), name + " codes differ"
        got = oracle.sf_to_rowmajor(g.scales.cpu().numpy(), g.rows, g.cols // 32)
        assert np.array_equal(got, o.scales), name + " scale bytes differ"
    rows = np.sort(np.random.default_rng(5003).choice(8192, 256, replace=False))
    check_rows(C, oracle.dequantize_mx(qa), oracle.dequantize_mx(qw), rows, matmul=True)
