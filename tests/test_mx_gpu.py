"""Parity of the MXFP4 4/6 quantizer (fos_quantize_mxfp4) with the oracle
(reading R12): codes, E8M0 scale bytes and choices bit for bit, and the
dequantized values exactly, with the scales row-major and in the 128x4 tiles
the block-scaled MMA reads (pad bytes zero); ragged and edge-case inputs, all
three scale rules, and the full-size gradient and weight shapes."""
import numpy as np
import pytest

import workloads
from fos_testutil import mixed_bits, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fos():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaptive_quantization_fos_b300 as fos

    return fos


def scales_rowmajor(fos, q):
    """The GPU's scale bytes as [rows, cols/32]; for the 128x4 tiles, also
    check that every pad byte is zero."""
    import oracle

    sf = q.scales.cpu().numpy().reshape(-1)
    nb = q.cols // 32
    if q.sf_layout == fos.FOS_SF_ROWMAJOR:
        return sf.reshape(q.rows, nb)
    assert sf.size == oracle.sf_bytes(q.rows, nb)
    real = np.zeros(sf.size, bool)
    r, c = np.meshgrid(np.arange(q.rows), np.arange(nb), indexing="ij")
    real[((r // 128) * ((nb + 3) // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4] = True
    assert not sf[~real].any(), "pad bytes of the 128x4 tiles are not zero"
    return oracle.sf_to_rowmajor(sf, q.rows, nb)


def check(fos, bits, ld=None, scale_rule=0, layouts=None):
    import torch

    import oracle

    x = to_device_bf16(bits, ld)
    o = oracle.quantize_mx(bits, scale_rule=scale_rule)
    want = oracle.dequantize_mx(o)
    rows, cols = bits.shape
    for layout in layouts or (fos.FOS_SF_ROWMAJOR, fos.FOS_SF_SWIZZLED_128x4):
        q = fos.quantize_mxfp4(x, scale_rule=scale_rule, sf_layout=layout, with_choice=True)
        if layout == fos.FOS_SF_SWIZZLED_128x4:
            # again into a buffer of junk: the launch itself writes every byte, pads included
            q.scales.fill_(0xA5)
            assert fos.fos_quantize_mxfp4(x.data_ptr(), rows, cols, x.stride(0), scale_rule, layout,
                                          q.codes.data_ptr(), q.codes.stride(0), q.scales.data_ptr(),
                                          q.choice.data_ptr(), None) == fos.FOS_OK
        d = fos.dequantize_mxfp4(q)
        db = fos.dequantize_mxfp4(q, dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert np.array_equal(q.codes[:, : cols // 2].cpu().numpy(), o.codes), "codes differ"
        assert np.array_equal(scales_rowmajor(fos, q), o.scales), "scale bytes differ"
        assert np.array_equal(q.choice.cpu().numpy(), o.choice), "choices differ"
        assert np.array_equal(d.cpu().numpy(), want), "dequantized values differ"
        assert np.array_equal(db.float().cpu().numpy(), workloads.bf16_to_f32(workloads.bf16_bits(want)))
    return o


@pytest.mark.parametrize("shape", [(1, 32), (3, 96), (300, 1056), (129, 512), (64, 4096)])
@pytest.mark.parametrize("rule", [0, 1, 2])
def test_mx_matches_oracle(fos, shape, rule):
    check(fos, mixed_bits(*shape, seed=shape[0] * 7 + shape[1]), scale_rule=rule)


def test_mx_padded_rows_and_edges(fos):
    check(fos, mixed_bits(40, 160, seed=3), ld=168)
    zeros = np.zeros((2, 64), np.uint16)
    zeros[1, 5] = 0x8000  # -0
    o = check(fos, zeros)
    assert not o.scales.any()
    big = workloads.bf16_bits(np.full((2, 32), 3.0e38, np.float32))
    tiny = workloads.bf16_bits(np.full((2, 32), 1.0e-38, np.float32) * np.arange(1, 33, dtype=np.float32))
    sub = np.full((1, 32), 0x0003, np.uint16)  # bf16 subnormals
    check(fos, np.concatenate([big, tiny]))
    check(fos, sub)
    seven = workloads.bf16_bits(np.array([[7.5] + [0.0] * 31, [6.0, 0.5, -1.5, 3.0] * 8], np.float32))
    o = check(fos, seven)
    assert o.choice[0, 0] == 1 and o.choice[1, 0] == 0


@pytest.mark.parametrize("name,make", [
    ("gradient 8192x12288", lambda: workloads.gradients(8192, 12288, seed=4001)),
    ("gate_proj 12288x4096", lambda: workloads.student_t(12288, 4096, seed=2004)),
])
def test_mx_full_size(fos, name, make):
    o = check(fos, make())
    assert 0 < o.choice.mean() < 0.5, name


@pytest.mark.parametrize("scale_rule", [0, 1, 2])
def test_mx_non_finite_blocks(fos, scale_rule):
    """Blocks holding +inf, -inf or NaN get the E8M0 NaN byte 0xFF with zero
    codes and choice 0 (reading R12) and dequantize to NaN, bit for bit with
    the oracle; the other blocks are unaffected."""
    import torch

    import oracle

    bits = mixed_bits(5, 256, seed=77)
    bits[0, 3] = 0x7F80   # +inf
    bits[1, 100] = 0xFF80  # -inf
    bits[2, 255] = 0x7FC0  # NaN
    bits[3, 32:64] = 0x7F81  # a block of signalling-pattern NaNs
    x = to_device_bf16(bits)
    q = fos.quantize_mxfp4(x, scale_rule=scale_rule, sf_layout=fos.FOS_SF_SWIZZLED_128x4, with_choice=True)
    d = fos.dequantize_mxfp4(q)
    db = fos.dequantize_mxfp4(q, dtype=torch.bfloat16)
    torch.cuda.synchronize()
    o = oracle.quantize_mx(bits, scale_rule=scale_rule)
    assert np.array_equal(q.codes[:, :128].cpu().numpy(), o.codes), "codes differ"
    assert np.array_equal(scales_rowmajor(fos, q), o.scales), "scale bytes differ"
    assert np.array_equal(q.choice.cpu().numpy(), o.choice), "choices differ"
    assert (o.scales == 0xFF).sum() == 4
    want = oracle.dequantize_mx(o)
    assert np.array_equal(d.cpu().numpy(), want, equal_nan=True), "dequantized values differ"
    got_b = db.view(torch.int16).cpu().numpy().view(np.uint16)
    nan_b = (got_b & 0x7F80) == 0x7F80
    assert np.array_equal(nan_b & ((got_b & 0x7F) != 0), np.isnan(want)), "bf16 NaN positions differ"
    fin = ~np.isnan(want)
    assert np.array_equal(got_b[fin], workloads.bf16_bits(want)[fin])
