"""Parity of the NVFP4 dequantizer (fos_dequantize) with the oracle.

The operands are the ORACLE's quantizations, uploaded as they are, so this
tests the dequantizer on its own: x_hat = g * (sf * s_t) with one FP32 rounding
("Four Over Six", first section: the FP32-simulation path multiplies
dequantized operands), f32 output bit for bit, bf16 output as the
round-to-nearest-even bf16 of that FP32 value.  Covered: both scale layouts,
operands from the transposed, 2D, RHT and stochastic-rounding options, output
rows wider than the matrix (ld_out > cols, the pad columns left untouched),
ragged shapes and the full q_proj-shaped weight.
"""
import ctypes

import numpy as np
import pytest

import workloads
from fos_testutil import mixed_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaptive_quantization_fos_b300 as fos
    import oracle

    return torch, fos, oracle


def upload(torch, fos, q):
    """The oracle's result as a device fos_nvfp4_tensor (plus the buffers it points into)."""
    codes = torch.from_numpy(np.ascontiguousarray(q.codes)).cuda()
    sf = torch.from_numpy(np.ascontiguousarray(q.sf)).cuda()
    ts = torch.tensor([q.tensor_scale], dtype=torch.float32, device="cuda")
    t = fos.fos_nvfp4_tensor()
    t.codes, t.sf, t.tensor_scale = codes.data_ptr(), sf.data_ptr(), ts.data_ptr()
    t.rows, t.cols, t.ld_codes, t.sf_layout = q.rows, q.cols, codes.stride(0), q.sf_layout
    return t, (codes, sf, ts)


def run(env, q, dtype, ld_out=None):
    torch, fos, _ = env
    t, keep = upload(torch, fos, q)
    ld = q.cols if ld_out is None else ld_out
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    code = fos.FOS_DTYPE_F32 if dtype == "f32" else fos.FOS_DTYPE_BF16
    canary = float("nan") if dtype == "f32" else 1234.0
    out = torch.full((max(q.rows, 1), max(ld, 8)), canary, dtype=tdt, device="cuda")
    st = fos.fos_dequantize(t, out.data_ptr(), code, ld, torch.cuda.current_stream().cuda_stream)
    assert st == fos.FOS_OK, fos.FosError(st, "fos_dequantize")
    torch.cuda.synchronize()
    got = out.cpu()
    if dtype == "f32":
        g = got.numpy()
    else:
        g = got.view(torch.int16).numpy().view(np.uint16)
    return g[: q.rows], keep


def want_of(oracle, q, dtype):
    d = oracle.dequantize(q)
    return d if dtype == "f32" else workloads.bf16_bits(d)


def check(env, q, dtype, ld_out=None):
    _, _, oracle = env
    got, _ = run(env, q, dtype, ld_out)
    want = want_of(oracle, q, dtype)
    body = got[:, : q.cols]
    if dtype == "f32":
        bad = np.argwhere(body.view(np.uint32) != want.view(np.uint32))
    else:
        bad = np.argwhere(body != want)
    assert bad.size == 0, f"{len(bad)} values differ, first {bad[:4].tolist()}"
    if ld_out is not None and ld_out > q.cols:
        pad = got[:, q.cols: ld_out]
        if dtype == "f32":
            assert np.isnan(pad).all(), "the dequantizer wrote past cols"
        else:
            assert (pad == workloads.bf16_bits(np.float32(1234.0))).all(), "the dequantizer wrote past cols"


SHAPES = [(1, 16), (3, 48), (300, 1040), (129, 512)]
SHAPES_16 = [(16, 16), (48, 80), (304, 1040)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [0, 1])
def test_dequantize_rows(env, shape, dtype, layout):
    _, _, oracle = env
    q = oracle.quantize(mixed_bits(*shape, seed=101 + shape[0]), sf_layout=layout)
    check(env, q, dtype)


@pytest.mark.parametrize("kind", [dict(transpose=True), dict(block_2d=True), dict(block_2d=True, transpose=True),
                                  dict(hadamard=True, hadamard_seed=5), dict(rounding=1, sr_seed=9),
                                  dict(scale_rule=1), dict(scale_rule=2)])
@pytest.mark.parametrize("shape", SHAPES_16)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_dequantize_option_operands(env, kind, shape, dtype):
    _, _, oracle = env
    q = oracle.quantize(mixed_bits(*shape, seed=201 + shape[1]), **kind)
    check(env, q, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [0, 1])
def test_dequantize_wide_output_rows(env, dtype, layout):
    _, _, oracle = env
    q = oracle.quantize(mixed_bits(130, 160, seed=301), sf_layout=layout)
    check(env, q, dtype, ld_out=160 + (8 if dtype == "bf16" else 4) * 3)


def test_dequantize_padded_code_rows(env):
    """Code rows wider than cols/2 bytes (ld_codes > cols/2)."""
    _, _, oracle = env
    q = oracle.quantize(mixed_bits(64, 96, seed=401), ld_codes=64)
    assert q.codes.shape == (64, 64)
    check(env, q, "f32")


def test_dequantize_zero_tensor(env):
    _, _, oracle = env
    q = oracle.quantize(np.zeros((32, 64), np.uint16))
    got, _ = run(env, q, "f32")
    assert not got.view(np.uint32).any()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_dequantize_full_size_weight(env, dtype):
    """The 4096 x 4096 q_proj-shaped weight of the Qwen3-8B layer set."""
    _, _, oracle = env
    q = oracle.quantize(workloads.student_t(4096, 4096, seed=2000))
    check(env, q, dtype)


def test_dequantize_rejects_bad_arguments(env):
    torch, fos, oracle = env
    q = oracle.quantize(mixed_bits(32, 64, seed=501))
    t, keep = upload(torch, fos, q)
    out = torch.empty((32, 64), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert fos.fos_dequantize(t, out.data_ptr(), fos.FOS_DTYPE_F32, 60, s) == fos.FOS_ERR_INVALID_ARG  # ld < cols
    assert fos.fos_dequantize(t, out.data_ptr(), 7, 64, s) == fos.FOS_ERR_INVALID_ARG  # dtype
    assert fos.fos_dequantize(t, out.data_ptr() + 4, fos.FOS_DTYPE_F32, 64, s) == fos.FOS_ERR_INVALID_ARG  # align
    t.cols = 40
    assert fos.fos_dequantize(t, out.data_ptr(), fos.FOS_DTYPE_F32, 64, s) == fos.FOS_ERR_INVALID_ARG  # cols % 16
    del keep
