"""Parity of fos_linear_backward (dX = dY W, dW = dY^T X for Y = X W^T) with
the oracle's backward.

The four quantized operands inside the workspace (dY along N, W^T along N,
dY^T and X^T along M) must equal the oracle's quantizations bit for bit
(codes, scale bytes, tensor scale); the two products must lie within the GEMM
bound |C - C_ref| <= 1e-3 sum |a||b| + 2^-8 |C_ref| of the FP64 products of
the oracle's dequantized operands.
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


def qout(t):
    return QOut(codes=t.codes[:, : t.cols // 2].cpu().numpy(), sf=t.sf.cpu().numpy(),
                s_t=np.float32(t.tensor_scale.item()), choice=None)


def oqout(r):
    return QOut(codes=np.ascontiguousarray(r.codes[:, : r.cols // 2]), sf=r.sf, s_t=np.float32(r.tensor_scale),
                choice=None)


def check(C, ref, bnd, what):
    c = C.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(c).all(), f"{what}: non-finite output"
    err = np.abs(c - ref)
    tol = REL_TOL * bnd + BF16_UNIT_ROUNDOFF * np.abs(ref)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, f"{what}: {len(bad)} elements outside the bound, first {bad[:4].tolist()}"


def run(fos, dy, x, w, need_dx=True, need_dw=True, **opts):
    import torch

    M, N = dy.shape
    K = x.shape[1]
    bw = fos.LinearBackward(M, N, K, **opts)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dx, dw = bw(to_device_bf16(dy), to_device_bf16(x), to_device_bf16(w), need_dx=need_dx, need_dw=need_dw,
                status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "a GEMM wait timed out"
    return bw, dx, dw


OPTS = [
    dict(),  # the training recipe: SR on dY, RHT along M for the weight gradient
    dict(grad_rounding=0, wgrad_hadamard=False),
    dict(weight_2d=True, sr_seed=77, hadamard_seed=3),
    dict(scale_rule=1, grad_rounding=0),
    # SR without the RHT, and under the 4-only rule: dY's two SR quantizations
    # share one launch in every SR case with both products
    dict(wgrad_hadamard=False, sr_seed=5),
    dict(scale_rule=2, sr_seed=9, hadamard_seed=4),
]


@pytest.mark.parametrize("M,N,K", [(128, 192, 80), (64, 64, 16), (192, 128, 272)])
@pytest.mark.parametrize("opts", OPTS)
def test_backward_matches_oracle(fos, M, N, K, opts):
    import oracle

    dy = mixed_bits(M, N, seed=M + N + K)
    x = workloads.activations(M, K, seed=K + 1)
    w = workloads.student_t(N, K, seed=N + 2)
    bw, dx, dw = run(fos, dy, x, w, **opts)
    oo = {k: v for k, v in opts.items()}
    ops = oracle.linear_backward_operands(dy, x, w, **oo)
    for name, g, o in zip(("dY", "W^T", "dY^T", "X^T"), bw.operands(), ops):
        assert (g.rows, g.cols) == (o.rows, o.cols), name
        assert_same(qout(g), oqout(o), name)
    (rx, bx), (rw, bwd) = oracle.linear_backward_rows(ops, np.arange(M), np.arange(N))
    check(dx, rx, bx, "dX")
    check(dw, rw, bwd, "dW")


def test_backward_halves_alone(fos):
    """dx or dw may be skipped; the other half is unchanged."""
    import oracle

    M, N, K = 128, 128, 64
    dy, x, w = mixed_bits(M, N, seed=1), workloads.activations(M, K, seed=2), workloads.student_t(N, K, seed=3)
    ops = oracle.linear_backward_operands(dy, x, w)
    (rx, bx), (rw, bwd) = oracle.linear_backward_rows(ops, np.arange(M), np.arange(N))
    _, dx, dw = run(fos, dy, x, w, need_dw=False)
    assert dw is None
    check(dx, rx, bx, "dX alone")
    _, dx, dw = run(fos, dy, x, w, need_dx=False)
    assert dx is None
    check(dw, rw, bwd, "dW alone")


def test_backward_full_size_sampled_rows(fos):
    """The linear layer of the forward case (X 8192 x 4096 activations, W
    12288 x 4096 weights) with dY 8192 x 12288 from the gradient recipe:
    all four operands bit-exact, then 256 seeded rows of dX and of dW."""
    import oracle

    M, N, K = 8192, 12288, 4096
    dy = workloads.gradients(M, N, seed=6001)
    x = workloads.activations(M, K, seed=6002)
    w = workloads.student_t(N, K, seed=6003)
    bw, dx, dw = run(fos, dy, x, w, sr_seed=11, hadamard_seed=12)
    ops = oracle.linear_backward_operands(dy, x, w, sr_seed=11, hadamard_seed=12)
    for name, g, o in zip(("dY", "W^T", "dY^T", "X^T"), bw.operands(), ops):
        assert_same(qout(g), oqout(o), name)
    rng = np.random.default_rng(6004)
    rx_rows = np.sort(rng.choice(M, 256, replace=False))
    rw_rows = np.sort(rng.choice(N, 256, replace=False))
    (rx, bx), (rw, bwd) = oracle.linear_backward_rows(ops, rx_rows, rw_rows, matmul=True)
    check(dx[rx_rows], rx, bx, "dX")
    check(dw[rw_rows], rw, bwd, "dW")
