"""Parity of fos_linear_forward (X quantized, then Y = X W^T against an already
quantized W, the GEMM launched as the quantizer's programmatic dependent).

X's operand inside the workspace must equal the oracle's quantization bit for
bit; Y must lie within the GEMM bound |C - C_ref| <= 1e-3 sum |a||b| +
2^-8 |C_ref| of the FP64 product of the oracle's dequantized operands.
"""
import numpy as np
import pytest

import workloads
from fos_testutil import QOut, assert_same, mixed_bits, to_device_bf16

pytestmark = pytest.mark.gpu

REL_TOL = 1e-3
BF16_UNIT_ROUNDOFF = 2.0 ** -8


@pytest.fixture(scope="module")
def fos():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaptive_quantization_fos_b300 as fos

    return fos


def check(C, ref, bnd, what="Y"):
    c = C.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(c).all(), f"{what}: non-finite output"
    err = np.abs(c - ref)
    tol = REL_TOL * bnd + BF16_UNIT_ROUNDOFF * np.abs(ref)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, f"{what}: {len(bad)} elements outside the bound, first {bad[:4].tolist()}"


def run(fos, x_bits, w_bits, **opts):
    """W quantized first (offline, with the same RHT options along K as X),
    then one fos_linear_forward call; returns (layer, Y, W's oracle result)."""
    import torch

    import oracle

    M, K = x_bits.shape
    w_opts = {k: v for k, v in opts.items() if k in ("hadamard", "hadamard_seed", "scale_rule")}
    w = fos.quantize(to_device_bf16(w_bits), **w_opts)
    layer = fos.LinearForward(M, K, **opts)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = layer(to_device_bf16(x_bits), w, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "a GEMM wait timed out"
    return layer, y, oracle.quantize(w_bits, **w_opts)


def x_operand(layer):
    t = layer.operand()
    return QOut(codes=t.codes[:, : t.cols // 2].cpu().numpy(), sf=t.sf.cpu().numpy(),
                s_t=np.float32(t.tensor_scale.item()), choice=None)


OPTS = [dict(), dict(hadamard=True, hadamard_seed=21), dict(rounding=1, sr_seed=5), dict(block_2d=True),
        dict(scale_rule=1)]


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 136, 320), (64, 512, 1024)])
@pytest.mark.parametrize("opts", OPTS)
def test_forward_matches_oracle(fos, M, N, K, opts):
    import oracle

    x = mixed_bits(M, K, seed=M + K)
    w = workloads.student_t(N, K, seed=N + 3)
    if opts.get("block_2d") and M % 16:
        # 16 x 16 tiles need whole 16-row groups: the call is refused, nothing runs
        with pytest.raises(fos.FosError) as e:
            run(fos, x, w, **opts)
        assert e.value.status == fos.FOS_ERR_INVALID_ARG
        return
    layer, y, qw = run(fos, x, w, **opts)
    qx = oracle.quantize(x, **opts)
    want = QOut(codes=np.ascontiguousarray(qx.codes[:, : K // 2]), sf=qx.sf, s_t=np.float32(qx.tensor_scale),
                choice=None)
    assert_same(x_operand(layer), want, "X")
    ref, bnd = oracle.gemm_rows(oracle.dequantize(qx), oracle.dequantize(qw), np.arange(M))
    check(y, ref, bnd)


def test_forward_delayed_scaling(fos):
    """A supplied tensor amax (delayed scaling) takes the single-pass quantizer."""
    import torch

    import oracle

    M, N, K = 256, 256, 512
    x = workloads.activations(M, K, seed=7)
    w = workloads.student_t(N, K, seed=8)
    amax = 180.0  # a previous step's amax (below this X's own: the largest values saturate)
    amax_dev = torch.tensor([amax], dtype=torch.float32, device="cuda")
    layer, y, qw = run(fos, x, w, tensor_amax=amax_dev)
    qx = oracle.quantize(x, amax=amax)
    assert_same(x_operand(layer), QOut(codes=np.ascontiguousarray(qx.codes[:, : K // 2]), sf=qx.sf,
                                       s_t=np.float32(qx.tensor_scale), choice=None), "X")
    ref, bnd = oracle.gemm_rows(oracle.dequantize(qx), oracle.dequantize(qw), np.arange(M))
    check(y, ref, bnd)


def test_forward_full_size_sampled_rows(fos):
    """The 8192 x 12288 x 4096 layer (activation-recipe X, weight-recipe W),
    4/6 1D RNE: X's operand bit-exact, then 256 seeded rows of Y."""
    import oracle

    M, N, K = 8192, 12288, 4096
    x = workloads.activations(M, K, seed=5001)
    w = workloads.student_t(N, K, seed=5002)
    layer, y, qw = run(fos, x, w)
    qx = oracle.quantize(x)
    assert_same(x_operand(layer), QOut(codes=np.ascontiguousarray(qx.codes[:, : K // 2]), sf=qx.sf,
                                       s_t=np.float32(qx.tensor_scale), choice=None), "X")
    rows = np.sort(np.random.default_rng(5003).choice(M, 256, replace=False))
    ref, bnd = oracle.gemm_rows_matmul(oracle.dequantize(qx), oracle.dequantize(qw), rows)
    check(y[rows], ref, bnd)
