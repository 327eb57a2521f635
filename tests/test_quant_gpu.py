"""Parity of the CUDA quantizer with the oracle: bit-exact codes, scale bytes,
tensor scale and 4/6 choices, over ragged shapes and every option."""
import numpy as np
import pytest

import workloads
from fos_testutil import assert_same, gpu_quantize, mixed_bits, oracle_quantize

pytestmark = pytest.mark.gpu

RNE, SR = 0, 1
SHAPES_1D = [(1, 16), (3, 48), (300, 1040), (129, 512), (64, 4096), (256, 256)]
# cols / 16 = 1, 5, 6, 7, 65, 256: a 2D row band of 4 tiles ends with 1, 2, 3 or 0 over
SHAPES_16 = [(16, 16), (48, 80), (32, 96), (64, 112), (304, 1040), (128, 4096)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaptive_quantization_fos_b300  # noqa: F401  (fails loudly if libfos.so is missing)


def check(bits, **opts):
    g = gpu_quantize(bits, **{k: v for k, v in opts.items() if k != "ld_x"}, ld=opts.get("ld_x"))
    o = oracle_quantize(bits, **{k: v for k, v in opts.items() if k != "ld_x"})
    assert_same(g, o, repr(opts))
    return g


@pytest.mark.parametrize("shape", SHAPES_1D)
@pytest.mark.parametrize("rule", [0, 1, 2])
def test_rows_rne(shape, rule):
    check(mixed_bits(*shape, seed=shape[0] * 7 + shape[1] + rule), scale_rule=rule)


@pytest.mark.parametrize("shape", SHAPES_1D)
def test_rows_sr(shape):
    check(mixed_bits(*shape, seed=11 + shape[0]), rounding=SR, sr_seed=0x9E3779B97F4A7C15)


@pytest.mark.parametrize("shape", SHAPES_1D)
@pytest.mark.parametrize("rounding", [RNE, SR])
def test_rows_hadamard(shape, rounding):
    check(mixed_bits(*shape, seed=21 + shape[1]), hadamard=True, hadamard_seed=12345, rounding=rounding, sr_seed=3)


@pytest.mark.parametrize("shape", SHAPES_1D)
@pytest.mark.parametrize("kind", [dict(), dict(scale_rule=1), dict(rounding=SR, sr_seed=9),
                                  dict(hadamard=True, hadamard_seed=4, rounding=SR, sr_seed=2)])
def test_rows_one_launch(shape, kind):
    """The cooperative one-launch form of the row quantizer (amax pass, grid
    barrier, quantize pass) against the oracle, like the two-launch default."""
    bits = mixed_bits(*shape, seed=61 + shape[0] + shape[1])
    assert_same(gpu_quantize(bits, one_launch=True, **kind), oracle_quantize(bits, **kind), repr(kind))


@pytest.mark.parametrize("shape", SHAPES_16)
@pytest.mark.parametrize("rounding", [RNE, SR])
@pytest.mark.parametrize("hadamard", [False, True])
def test_transposed(shape, rounding, hadamard):
    check(mixed_bits(*shape, seed=31 + shape[0]), transpose=True, rounding=rounding, sr_seed=77,
          hadamard=hadamard, hadamard_seed=99)


@pytest.mark.parametrize("shape", SHAPES_16)
@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("rounding", [RNE, SR])
@pytest.mark.parametrize("hadamard", [False, True])
def test_2d(shape, transpose, rounding, hadamard):
    check(mixed_bits(*shape, seed=41 + shape[1]), block_2d=True, transpose=transpose, rounding=rounding,
          sr_seed=5, hadamard=hadamard, hadamard_seed=7)


@pytest.mark.parametrize("kind", [dict(), dict(transpose=True), dict(block_2d=True), dict(hadamard=True),
                                  dict(block_2d=True, rounding=SR, sr_seed=5),
                                  dict(transpose=True, rounding=SR, sr_seed=5)])
def test_rowmajor_scale_layout(kind):
    check(mixed_bits(304, 1040, seed=51), sf_layout=1, **kind)


@pytest.mark.parametrize("kind", [dict(), dict(transpose=True), dict(block_2d=True),
                                  dict(block_2d=True, rounding=SR, sr_seed=6)])
def test_padded_source_rows(kind):
    check(mixed_bits(48, 160, seed=61), ld_x=168, **kind)


def test_rule_variants_2d_and_transposed():
    x = mixed_bits(64, 128, seed=71)
    for rule in (1, 2):
        check(x, scale_rule=rule, block_2d=True)
        check(x, scale_rule=rule, transpose=True)


def test_supplied_amax():
    import torch

    import adaptive_quantization_fos_b300 as fos
    import oracle

    x = mixed_bits(128, 256, seed=81)
    amax = torch.tensor([123.5], dtype=torch.float32, device="cuda")
    q = fos.quantize(__import__("fos_testutil").to_device_bf16(x), tensor_amax=amax, with_choice=True)
    torch.cuda.synchronize()
    o = oracle.quantize(x, amax=123.5)
    assert np.array_equal(q.codes.cpu().numpy()[:, :128], o.codes)
    assert np.array_equal(q.sf.cpu().numpy(), o.sf)


def test_tensor_amax_entry_point():
    import torch

    import adaptive_quantization_fos_b300 as fos
    import oracle
    from fos_testutil import to_device_bf16

    x = mixed_bits(304, 1040, seed=91)
    xf = workloads.bf16_to_f32(x)
    assert fos.tensor_amax(to_device_bf16(x)).item() == np.abs(xf).max()
    mask = oracle.rht_sign_mask(17)
    y = oracle.rht16(xf.reshape(-1, 16), mask)
    assert fos.tensor_amax(to_device_bf16(x), hadamard=True, hadamard_seed=17).item() == np.abs(y).max()
    yt = oracle.rht16(np.ascontiguousarray(xf.T).reshape(-1, 16), mask)
    got = fos.tensor_amax(to_device_bf16(x), hadamard=True, transpose=True, hadamard_seed=17).item()
    assert got == np.abs(yt).max()
    torch.cuda.synchronize()


def test_edge_cases():
    check(np.zeros((16, 64), np.uint16))
    check(np.zeros((16, 64), np.uint16), block_2d=True)
    neg_zero = np.full((16, 32), 0x8000, np.uint16)
    check(neg_zero)
    one = np.zeros((1, 16), np.float32)
    one[0, 3] = -7.0
    check(workloads.bf16_bits(one))
    big = np.full((4, 32), 3.0e38, np.float32)
    big[:, ::3] = -1.0e38
    check(workloads.bf16_bits(big))
    tiny = np.full((4, 32), 1.0e-38, np.float32)
    tiny[:, ::5] = 9.0e-41
    check(workloads.bf16_bits(tiny))
    check(workloads.bf16_bits(tiny), rounding=SR, sr_seed=4)


def test_empty_input():
    import torch

    import adaptive_quantization_fos_b300 as fos

    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    q = fos.quantize(x)
    torch.cuda.synchronize()
    assert q.tensor_scale.item() == 0.0


def test_outlier_matrix_matches_and_beats_six_only():
    x = workloads.outlier_matrix()
    g46 = check(x)
    check(x, scale_rule=1)
    assert 0 < g46.choice.mean() < 1


def test_candidate_scales_at_exact_e4m3_ties():
    import oracle

    from fos_testutil import e4m3_tie_blocks

    bits, ties = e4m3_tie_blocks()
    assert len(ties) >= 20
    # the oracle takes the even neighbour on every tie (RNE of the quotient)
    for rule, M in ((2, 4), (1, 6)):
        o = oracle.quantize(bits, scale_rule=rule, sf_layout=1)
        sf = o.sf.reshape(bits.shape[0], 4)
        for r, (_, m, even) in enumerate(ties):
            if m == M:
                assert sf[r, 1] == even, (r, hex(sf[r, 1]), hex(even))
    for rule in (0, 1, 2):
        check(bits, scale_rule=rule)
        check(bits, scale_rule=rule, sf_layout=1)
