"""The C-ABI library (no GPU needed): it loads, exports every call that
include/fos.h declares, its structs have the header's layout, and argument
validation rejects bad input without launching anything."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fos.h")


@pytest.fixture(scope="module")
def fos():
    import adaptive_quantization_fos_b300 as fos

    return fos


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fos_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_function(fos):
    lib = ctypes.CDLL(fos.LIB_PATH)
    names = declared_functions()
    assert "fos_quantize" in names and "fos_gemm" in names and "fos_dequantize" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(fos.EXPORTED)


def test_struct_layout_matches_header(fos, tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "fos.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu %zu %zu %zu\\n\", sizeof(fos_quant_options),"
        " offsetof(fos_quant_options, sr_seed), offsetof(fos_quant_options, tensor_amax),"
        " sizeof(fos_nvfp4_tensor), offsetof(fos_nvfp4_tensor, rows), offsetof(fos_nvfp4_tensor, sf_layout),"
        " sizeof(fos_mxfp4_tensor), offsetof(fos_mxfp4_tensor, rows), offsetof(fos_mxfp4_tensor, sf_layout));"
        "return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), "-I", "/usr/local/cuda/include", str(src),
                           "-o", str(exe)])
    got = [int(v) for v in subprocess.check_output([str(exe)]).split()]
    O, T, X = fos.fos_quant_options, fos.fos_nvfp4_tensor, fos.fos_mxfp4_tensor
    assert got == [ctypes.sizeof(O), O.sr_seed.offset, O.tensor_amax.offset, ctypes.sizeof(T), T.rows.offset,
                   T.sf_layout.offset, ctypes.sizeof(X), X.rows.offset, X.sf_layout.offset]


def test_version_and_sizes(fos):
    assert fos.fos_abi_version() == 2
    assert fos.fos_sf_bytes(300, 1040) == 384 * 68
    assert fos.fos_sf_bytes(300, 1040, fos.FOS_SF_ROWMAJOR) == 300 * 65
    assert fos.fos_sf_bytes(0, 0) == 0
    o = fos.options()
    assert fos.fos_quantize_workspace_size(64, 64, o) > 0
    with pytest.raises(fos.FosError):
        fos.fos_sf_bytes(10, 17)


def test_validation_rejects_without_launch(fos):
    INVALID = fos.FOS_ERR_INVALID_ARG
    o = fos.options()
    fake = 1 << 20  # never dereferenced: validation fails first
    ws = fos.fos_quantize_workspace_size(32, 64, o)
    q = lambda **kw: fos.fos_quantize(  # noqa: E731
        kw.get("x", fake), kw.get("rows", 32), kw.get("cols", 64), kw.get("ld", 64), kw.get("opt", o),
        kw.get("codes", fake), kw.get("ldc", 32), kw.get("sf", fake), kw.get("ts", fake), 0,
        kw.get("ws", fake), kw.get("wsb", ws), 0)
    assert q(cols=40, ld=40) == INVALID  # cols % 16
    assert q(ld=60) == INVALID  # ld < cols
    assert q(ld=68) == INVALID  # ld % 8
    assert q(x=fake + 2) == INVALID  # alignment
    assert q(x=0) == INVALID
    assert q(codes=0) == INVALID
    assert q(ldc=16) == INVALID  # ld_codes < C/2
    assert q(ws=0) == INVALID
    assert q(wsb=4) == INVALID
    assert q(rows=-1) == INVALID
    assert q(rows=24, opt=fos.options(transpose=True)) == INVALID  # rows % 16
    assert q(rows=24, opt=fos.options(block_2d=True)) == INVALID
    bad = fos.options()
    bad.scale_rule = 7
    assert q(opt=bad) == INVALID
    bad = fos.options()
    bad.struct_size = 8
    assert q(opt=bad) == INVALID
    bad = fos.options()
    bad.one_launch = 2
    assert q(opt=bad) == INVALID
    t = fos.fos_nvfp4_tensor()
    assert fos.fos_dequantize(t, fake, 0, 64, 0) == INVALID
    assert fos.fos_e2m1_encode(0, 5, 0, 0) == INVALID


def test_batch_validation_rejects_without_launch(fos):
    """fos_quantize_batch refuses before anything is enqueued: a supplied amax
    (unsupported), a transposed or 2D job without whole 16-row groups, an
    output row stride too small for the transposed output."""
    fake = 1 << 20  # never dereferenced: validation fails first
    ws = fos.fos_quantize_batch_workspace_size(2)

    def call(opt, rows=32, cols=64, ldc=None):
        R, C = (cols, rows) if opt.transpose else (rows, cols)
        job = fos.fos_quant_job(fake, rows, cols, cols, fake, C // 2 if ldc is None else ldc, fake, fake, None)
        return fos.fos_quantize_batch([job, job], opt, fake, ws, 0)

    bad = fos.options()
    bad.tensor_amax = fake
    assert call(bad) == fos.FOS_ERR_UNSUPPORTED
    assert call(fos.options(transpose=True), rows=24) == fos.FOS_ERR_INVALID_ARG
    assert call(fos.options(block_2d=True), rows=24) == fos.FOS_ERR_INVALID_ARG
    assert call(fos.options(transpose=True), ldc=8) == fos.FOS_ERR_INVALID_ARG  # C_out / 2 = 16
    assert fos.fos_quantize_batch([], fos.options(transpose=True), 0, 0, 0) == fos.FOS_OK


def test_batch_quantizer_output_shapes_on_host(fos):
    """BatchQuantizer sizes its outputs on the host (nothing launches): a
    transposed job's codes, scales and choices are [cols, rows]-shaped, a row
    job's [rows, cols]-shaped, each scale buffer fos_sf_bytes of that shape."""
    for opts, swap in ((dict(), False), (dict(transpose=True), True), (dict(block_2d=True), False),
                       (dict(transpose=True, sf_layout=fos.FOS_SF_ROWMAJOR), True)):
        shapes = [(64, 256), (48, 80), (16, 4096)]
        bq = fos.BatchQuantizer(shapes, device="cpu", with_choice=True, **opts)
        assert bq.shapes == shapes
        layout = opts.get("sf_layout", fos.FOS_SF_SWIZZLED_128x4)
        for (rows, cols), o in zip(shapes, bq.outs):
            R, C = (cols, rows) if swap else (rows, cols)
            assert (o.rows, o.cols) == (R, C), opts
            assert o.codes.shape[0] == R and o.codes.shape[1] >= C // 2 and o.codes.shape[1] % 16 == 0
            assert o.sf.numel() == fos.fos_sf_bytes(R, C, layout)
            assert tuple(o.choice.shape) == (R, C // 16)
        assert bq.ws_bytes == fos.fos_quantize_batch_workspace_size(len(shapes))


def test_gemm_validation(fos):
    INVALID = fos.FOS_ERR_INVALID_ARG
    fake = 1 << 20
    A = fos.fos_nvfp4_tensor(codes=fake, sf=fake, tensor_scale=fake, rows=128, cols=256, ld_codes=128)
    B = fos.fos_nvfp4_tensor(codes=fake, sf=fake, tensor_scale=fake, rows=256, cols=512, ld_codes=256)
    assert fos.fos_gemm(A, B, fake, 256, 0, 0) == INVALID  # K differs
    B.cols, B.ld_codes = 256, 128
    assert fos.fos_gemm(A, B, fake, 100, 0, 0) == INVALID  # ldc < N
    assert fos.fos_gemm(A, B, fake + 8, 256, 0, 0) == INVALID  # C not 16-byte aligned
    assert fos.fos_gemm(A, B, fake, 260, 0, 0) == INVALID  # ldc % 8
    B.rows = 250
    assert fos.fos_gemm(A, B, fake, 256, 0, 0) == INVALID  # N % 8
    B.rows = 256
    A.cols = B.cols = 96
    assert fos.fos_gemm(A, B, fake, 256, 0, 0) == INVALID  # K % 64
    A.cols = B.cols = 256
    A.ld_codes = 136
    assert fos.fos_gemm(A, B, fake, 256, 0, 0) == INVALID  # ld_codes % 16
    A.ld_codes = 128
    A.sf_layout = fos.FOS_SF_ROWMAJOR
    assert fos.fos_gemm(A, B, fake, 256, 0, 0) == INVALID  # the MMA reads the 128x4 layout only
    A.sf_layout = fos.FOS_SF_SWIZZLED_128x4
    A.rows = 0
    assert fos.fos_gemm(A, B, fake, 256, 0, 0) == fos.FOS_OK  # empty: nothing to launch


def test_linear_backward_validation(fos):
    """Every argument check of fos_linear_backward fails before anything is
    enqueued (fake device addresses; nothing here reaches a launch)."""
    INVALID = fos.FOS_ERR_INVALID_ARG
    fake = 1 << 20
    M, N, K = 128, 192, 80
    ws = fos.fos_linear_backward_workspace_size(M, N, K)
    assert ws > 0
    opt = fos.backward_options()

    def call(M=M, N=N, K=K, dy=fake, ld_dy=N, x=fake, ld_x=K, w=fake, ld_w=K, o=opt, dx=fake, ld_dx=K, dw=fake,
             ld_dw=K, wsp=fake, wsb=ws, status=0):
        return fos.fos_linear_backward(dy, ld_dy, x, ld_x, w, ld_w, M, N, K, o, dx, ld_dx, dw, ld_dw, wsp, wsb,
                                       status, 0)

    assert call(M=96) == INVALID  # M % 64 (the weight-gradient contraction)
    assert call(N=160) == INVALID  # N % 64 (the data-gradient contraction)
    assert call(K=72) == INVALID  # K % 16
    assert call(M=0) == INVALID
    assert call(dy=0) == INVALID
    assert call(ld_dy=N - 8) == INVALID
    assert call(ld_x=K + 4) == INVALID  # ld % 8
    assert call(w=fake + 8) == INVALID  # 16-byte alignment
    assert call(dx=fake + 2) == INVALID
    assert call(ld_dw=K - 16) == INVALID
    assert call(wsb=ws - 1) == INVALID
    assert call(wsp=fake + 128) == INVALID  # workspace 256-byte aligned
    assert call(status=fake + 2) == INVALID
    assert call(x=0) == INVALID  # the weight gradient needs X
    assert call(w=0) == INVALID  # the data gradient needs W
    for field, value in (("scale_rule", 5), ("grad_rounding", 2), ("wgrad_hadamard", 2), ("weight_2d", 3),
                         ("reserved", 1), ("struct_size", 8)):
        bad = fos.backward_options()
        setattr(bad, field, value)
        assert call(o=bad) == INVALID, field
    ops = fos.fos_linear_backward_operands(M, N, K, fake, ws)
    assert [(o.rows, o.cols) for o in ops] == [(M, N), (K, N), (N, M), (K, M)]
    assert all(o.ld_codes % 16 == 0 and o.codes % 256 == 0 and o.sf % 256 == 0 for o in ops)
    with pytest.raises(fos.FosError):
        fos.fos_linear_backward_workspace_size(100, N, K)


def test_linear_forward_validation(fos):
    """fos_linear_forward's argument checks (fake device addresses; nothing here
    reaches a launch)."""
    INVALID = fos.FOS_ERR_INVALID_ARG
    fake = 1 << 20
    M, K, N = 256, 512, 384
    ws = fos.fos_linear_forward_workspace_size(M, K)
    W = fos.fos_nvfp4_tensor(codes=fake, sf=fake, tensor_scale=fake, rows=N, cols=K, ld_codes=K // 2)

    def call(x=fake, ld_x=K, M=M, K=K, o=None, w=W, y=fake, ld_y=N, wsp=fake, wsb=ws, status=0):
        return fos.fos_linear_forward(x, ld_x, M, K, o if o is not None else fos.options(), w, y, ld_y, wsp, wsb,
                                      status, 0)

    assert call(K=480) == INVALID  # K % 64 (one MMA step)
    assert call(M=0) == INVALID
    assert call(o=fos.options(transpose=True)) == INVALID
    assert call(o=fos.options(sf_layout=fos.FOS_SF_ROWMAJOR)) == INVALID
    assert call(ld_y=N - 8) == INVALID
    assert call(y=fake + 4) == INVALID
    assert call(wsb=ws - 1) == INVALID
    assert call(wsp=fake + 64) == INVALID
    assert call(status=fake + 1) == INVALID
    W.cols = K + 64
    assert call() == INVALID  # W's K differs
    W.cols, W.rows = K, N - 4
    assert call() == INVALID  # N % 8
    W.rows, W.ld_codes = N, K // 2 + 8
    assert call() == INVALID  # ld_codes % 16
    W.ld_codes, W.sf_layout = K // 2, fos.FOS_SF_ROWMAJOR
    assert call() == INVALID
    d = fos.fos_linear_forward_operand(M, K, fake, ws)
    assert (d.rows, d.cols, d.ld_codes) == (M, K, K // 2) and d.sf % 256 == 0 and d.tensor_scale % 256 == 0


def test_mxfp4_validation(fos):
    INVALID = fos.FOS_ERR_INVALID_ARG
    fake = 1 << 20
    q = fos.fos_quantize_mxfp4
    assert q(fake, 4, 48, 48, 0, 0, fake, 32, fake, 0, 0) == INVALID  # cols % 32
    assert q(fake, 4, 64, 60, 0, 0, fake, 32, fake, 0, 0) == INVALID  # ld_x < cols
    assert q(fake, 4, 64, 68, 0, 0, fake, 32, fake, 0, 0) == INVALID  # ld_x % 8
    assert q(fake + 8, 4, 64, 64, 0, 0, fake, 32, fake, 0, 0) == INVALID  # x 16-byte aligned
    assert q(fake, 4, 64, 64, 3, 0, fake, 32, fake, 0, 0) == INVALID  # scale rule
    assert q(fake, 4, 64, 64, 0, 2, fake, 32, fake, 0, 0) == INVALID  # scale layout
    assert q(fake, 4, 64, 64, 0, 0, fake, 30, fake, 0, 0) == INVALID  # ld_codes < cols / 2
    assert q(fake, 4, 64, 64, 0, 0, fake + 2, 32, fake, 0, 0) == INVALID  # codes 4-byte aligned
    assert q(fake, 4, 64, 64, 0, 0, fake, 32, 0, 0, 0) == INVALID  # scales
    assert q(fake, 0, 64, 64, 0, 0, 0, 32, 0, 0, 0) == fos.FOS_OK  # empty: nothing to launch
    d = fos.fos_dequantize_mxfp4
    t = fos.fos_mxfp4_tensor(codes=fake, sf=fake, rows=4, cols=48, ld_codes=32)
    assert d(t, fake, 0, 48, 0) == INVALID  # cols % 32
    t.cols = 64
    assert d(t, fake, 7, 64, 0) == INVALID  # dtype
    assert d(t, fake + 2, 0, 64, 0) == INVALID  # f32 output 4-byte aligned
    assert d(t, fake, 0, 48, 0) == INVALID  # ld_out < cols
    t.sf_layout = 5
    assert d(t, fake, 0, 64, 0) == INVALID  # scale layout
    assert fos.fos_mxfp4_sf_bytes(300, 1056) == 384 * 36
    assert fos.fos_mxfp4_sf_bytes(300, 1056, fos.FOS_SF_ROWMAJOR) == 300 * 33
    assert fos.fos_mxfp4_sf_bytes(0, 0) == 0
    with pytest.raises(fos.FosError):
        fos.fos_mxfp4_sf_bytes(10, 48)


def test_gemm_mxfp4_validation(fos):
    INVALID = fos.FOS_ERR_INVALID_ARG
    fake = 1 << 20
    g = fos.fos_gemm_mxfp4
    A = fos.fos_mxfp4_tensor(codes=fake, sf=fake, rows=128, cols=256, ld_codes=128)
    B = fos.fos_mxfp4_tensor(codes=fake, sf=fake, rows=256, cols=512, ld_codes=256)
    assert g(A, B, fake, 256, 0, 0) == INVALID  # K differs
    B.cols, B.ld_codes = 256, 128
    assert g(A, B, fake, 100, 0, 0) == INVALID  # ldc < N
    assert g(A, B, fake + 8, 256, 0, 0) == INVALID  # C not 16-byte aligned
    B.rows = 250
    assert g(A, B, fake, 256, 0, 0) == INVALID  # N % 8
    B.rows = 256
    A.cols = B.cols = 96
    assert g(A, B, fake, 256, 0, 0) == INVALID  # K % 64
    A.cols = B.cols = 256
    A.sf = fake + 4
    assert g(A, B, fake, 256, 0, 0) == INVALID  # scales 16-byte aligned
    A.sf = fake
    A.sf_layout = fos.FOS_SF_ROWMAJOR
    assert g(A, B, fake, 256, 0, 0) == INVALID  # the MMA reads the 128x4 layout only
    A.sf_layout = fos.FOS_SF_SWIZZLED_128x4
    A.rows = 0
    assert g(A, B, fake, 256, 0, 0) == fos.FOS_OK  # empty: nothing to launch


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import importlib.util

    spec = importlib.util.spec_from_file_location(
        "fos_copy", os.path.join(ROOT, "adaptive_quantization_fos_b300", "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    src = open(spec.origin).read().replace('LIB_PATH = os.path.join(_PKG, "libfos.so")',
                                           f'LIB_PATH = {str(tmp_path / "missing.so")!r}')
    with pytest.raises(ImportError):
        exec(compile(src, spec.origin, "exec"), mod.__dict__)


def test_mma_rate_rejects_bad_arguments(fos):
    assert fos.fos_selftest_mma_rate(64, 10, 1, 0, None) == fos.FOS_ERR_INVALID_ARG
    assert fos.fos_selftest_mma_rate(256, 0, 1, 0, None) == fos.FOS_ERR_INVALID_ARG
    assert fos.fos_selftest_mma_rate(256, 1 << 25, 1, 0, None) == fos.FOS_ERR_INVALID_ARG
    assert fos.fos_selftest_mma_rate(128, 10, 0, 0, None) == fos.FOS_ERR_INVALID_ARG
