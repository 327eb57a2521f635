"""Maximum sizes.  The row quantizer at a size where element indices pass
2^34, so the stochastic-rounding Philox counter (i / 4) needs its high word,
and byte offsets pass 2^31: a 262208 x 65536 bf16 gradient (17.2 G values, 34 GB on the
device), quantized with SR through both forms of the row path: the default
two launches (amax pass, then the quantize pass) and the one cooperative launch
(amax pass, grid barrier, quantize pass).  Rows on both sides of index 2^34 are
compared with the oracle's quantization of the same rows at the same source
indices.

The matrix repeats one seeded 64-row block, so its amax is the block's; the
stochastic-rounding words still differ everywhere (they depend on the index).
"""
import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu

ROWS, COLS = 262208, 65536  # ROWS * COLS > 2^34
BLOCK_ROWS = 64


@pytest.fixture(scope="module")
def fos():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < 60 << 30:
        pytest.skip("needs about 50 GB of free device memory")
    import adaptive_quantization_fos_b300 as fos

    return fos


def test_sr_rows_beyond_2_pow_34(fos):
    import torch

    import oracle

    base = workloads.gradients(BLOCK_ROWS, COLS, seed=7001)
    dev_base = torch.from_numpy(base.view(np.int16)).view(torch.bfloat16).cuda()
    x = dev_base.repeat(ROWS // BLOCK_ROWS + 1, 1)[:ROWS]
    assert x.is_contiguous() and x.shape == (ROWS, COLS)
    amax = float(np.abs(workloads.bf16_to_f32(base)).max())
    nb = COLS // 16
    first_beyond = (1 << 34) // COLS  # the first row whose indices reach 2^34
    expect = {}
    for r in (0, 1, first_beyond - 1, first_beyond, ROWS - 1):
        expect[r] = oracle.quantize(base[r % BLOCK_ROWS][None, :], rounding=oracle.ROUND_SR, sr_seed=77, amax=amax,
                                    sf_layout=oracle.SF_ROWMAJOR, src_row0=r, src_cols=COLS)
    for one_launch in (False, True):
        q = fos.quantize(x, rounding=fos.FOS_ROUND_STOCHASTIC, sr_seed=77, sf_layout=fos.FOS_SF_ROWMAJOR,
                         one_launch=one_launch)
        torch.cuda.synchronize()
        form = "one launch" if one_launch else "two launches"
        # the tensor amax is the block's (the matrix repeats it)
        assert np.float32(q.tensor_scale.item()) == np.float32(oracle.quantize(base[:1], amax=amax).tensor_scale), form
        for r, o in expect.items():
            got_codes = q.codes[r, : COLS // 2].cpu().numpy()
            got_sf = q.sf[r * nb:(r + 1) * nb].cpu().numpy()
            assert np.array_equal(got_codes, o.codes[0]), f"{form}, row {r}: codes differ"
            assert np.array_equal(got_sf, o.sf[:nb]), f"{form}, row {r}: scales differ"
        del q
        torch.cuda.empty_cache()
    del x
    torch.cuda.empty_cache()


def test_gemm_output_beyond_2_pow_31(fos):
    """C = A W^T with 49152 x 49152 outputs (2.4 G elements, 4.8 GB of bf16,
    offsets past 2^31), K = 256: sampled rows, the last tile row included,
    within the GEMM bound of the oracle's FP64 product."""
    import torch

    import oracle
    from fos_testutil import to_device_bf16

    M = N = 49152
    K = 256
    xa = workloads.activations(M, K, seed=7101)
    xw = workloads.student_t(N, K, seed=7102)
    a = fos.quantize(to_device_bf16(xa))
    w = fos.quantize(to_device_bf16(xw))
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fos.gemm(a, w, out=C, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "a GEMM wait timed out"
    rows = np.array([0, 1, 24575, M - 129, M - 2, M - 1])
    ref, bnd = oracle.gemm_rows_matmul(oracle.dequantize(oracle.quantize(xa)), oracle.dequantize(oracle.quantize(xw)),
                                       rows)
    c = C[torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
    assert np.isfinite(c).all()
    assert np.all(np.abs(c - ref) <= 1e-3 * bnd + 2.0 ** -8 * np.abs(ref))
    del C
    torch.cuda.empty_cache()
