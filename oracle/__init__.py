"""CPU oracle for Four Over Six NVFP4 quantization (test infrastructure only).

Plain C (``fos_oracle.c``), single-threaded, compiled with
``-ffp-contract=off`` so every FP32 expression is rounded where it is written.
Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the CUDA library never does, and this
package never imports the CUDA library.

Every function cites what it follows; the fixed readings R1-R8 (tensor scale
amax/(6*448), scaled-domain block error, ties to 6, E2M1 RNE with kept sign,
Philox stochastic rounding, the 16-point RHT, 2D tiles, transposed input) are
spelled out at the top of ``fos_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fos_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC"]

SCALE_4OVER6, SCALE_6, SCALE_4 = 0, 1, 2
ROUND_RNE, ROUND_SR = 0, 1
SF_SWIZZLED, SF_ROWMAJOR = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle shared library next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", _LIB, "-lm"])
    return _LIB


class _Opts(ctypes.Structure):
    _fields_ = [
        ("scale_rule", ctypes.c_int32),
        ("rounding", ctypes.c_int32),
        ("block_2d", ctypes.c_int32),
        ("transpose", ctypes.c_int32),
        ("hadamard", ctypes.c_int32),
        ("sf_layout", ctypes.c_int32),
        ("sr_seed", ctypes.c_uint64),
        ("hadamard_seed", ctypes.c_uint64),
        ("use_amax", ctypes.c_int32),
        ("amax", ctypes.c_float),
        ("src_row0", ctypes.c_int64),
        ("src_cols", ctypes.c_int64),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        L = _lib
        vp, i64, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
        L.orc_e2m1_decode.restype = ctypes.c_float
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.orc_e2m1_rne.restype = ctypes.c_uint8
        L.orc_e2m1_rne.argtypes = [ctypes.c_float]
        L.orc_e2m1_sr.restype = ctypes.c_uint8
        L.orc_e2m1_sr.argtypes = [ctypes.c_float, ctypes.c_uint32]
        L.orc_e4m3_decode.restype = ctypes.c_float
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_rne_satfinite.restype = ctypes.c_uint8
        L.orc_e4m3_rne_satfinite.argtypes = [ctypes.c_float]
        L.orc_philox4x32_10.restype = None
        L.orc_philox4x32_10.argtypes = [vp, vp, vp]
        L.orc_sr_word.restype = ctypes.c_uint32
        L.orc_sr_word.argtypes = [u64, u64]
        L.orc_rht_sign_mask.restype = ctypes.c_uint32
        L.orc_rht_sign_mask.argtypes = [u64]
        L.orc_rht16_n.restype = None
        L.orc_rht16_n.argtypes = [vp, i64, ctypes.c_uint32]
        L.orc_sumsq16.restype = ctypes.c_float
        L.orc_sumsq16.argtypes = [vp]
        L.orc_sf_offset.restype = i64
        L.orc_sf_offset.argtypes = [i64, i64, i64, ctypes.c_int]
        L.orc_sf_bytes.restype = i64
        L.orc_sf_bytes.argtypes = [i64, i64, ctypes.c_int]
        L.orc_quantize.restype = ctypes.c_int
        L.orc_quantize.argtypes = [vp, i64, i64, i64, ctypes.POINTER(_Opts), vp, i64, vp, vp, vp]
        L.orc_dequantize.restype = None
        L.orc_dequantize.argtypes = [vp, i64, i64, i64, vp, ctypes.c_int, ctypes.c_float, vp]
        L.orc_gemm_rows.restype = None
        L.orc_gemm_rows.argtypes = [vp, vp, i64, i64, vp, i64, vp, vp]
        L.orc_mae_nearest_grid.restype = ctypes.c_double
        L.orc_mae_nearest_grid.argtypes = [vp, i64, i64]
        L.orc_e2m1_rne_n.restype = None
        L.orc_e2m1_rne_n.argtypes = [vp, i64, vp]
        L.orc_e2m1_sr_n.restype = None
        L.orc_e2m1_sr_n.argtypes = [vp, vp, i64, vp]
        L.orc_e4m3_rne_satfinite_n.restype = None
        L.orc_e4m3_rne_satfinite_n.argtypes = [vp, i64, vp]
        L.orc_sr_words_n.restype = None
        L.orc_sr_words_n.argtypes = [u64, vp, i64, vp]
        L.orc_e8m0_decode.restype = ctypes.c_float
        L.orc_e8m0_decode.argtypes = [ctypes.c_uint8]
        L.orc_mx_exponent.restype = ctypes.c_int
        L.orc_mx_exponent.argtypes = [ctypes.c_float, ctypes.c_int]
        L.orc_quantize_mx.restype = ctypes.c_int
        L.orc_quantize_mx.argtypes = [vp, i64, i64, i64, ctypes.c_int, vp, i64, vp, vp]
        L.orc_dequantize_mx.restype = None
        L.orc_dequantize_mx.argtypes = [vp, vp, i64, i64, i64, vp]
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ----------------------------------------------------------------- formats


def e2m1_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib().orc_e2m1_decode(int(v)) for v in c.ravel()], np.float32).reshape(c.shape)


def e2m1_rne(q) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float32)
    out = np.empty(q.shape, np.uint8)
    lib().orc_e2m1_rne_n(_p(q), q.size, _p(out))
    return out


def e2m1_sr(q, words) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float32)
    w = np.ascontiguousarray(words, dtype=np.uint32)
    assert w.shape == q.shape
    out = np.empty(q.shape, np.uint8)
    lib().orc_e2m1_sr_n(_p(q), _p(w), q.size, _p(out))
    return out


def e4m3_decode(b) -> np.ndarray:
    c = np.asarray(b, dtype=np.uint8)
    return np.array([lib().orc_e4m3_decode(int(v)) for v in c.ravel()], np.float32).reshape(c.shape)


def e4m3_rne_satfinite(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_rne_satfinite_n(_p(x), x.size, _p(out))
    return out


# ------------------------------------------------------------------ Philox


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.empty(4, np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def sr_words(seed: int, idx) -> np.ndarray:
    i = np.ascontiguousarray(idx, dtype=np.uint64)
    out = np.empty(i.shape, np.uint32)
    lib().orc_sr_words_n(seed, _p(i), i.size, _p(out))
    return out


def rht_sign_mask(seed: int) -> int:
    return int(lib().orc_rht_sign_mask(seed))


def rht16(w, sign_mask: int) -> np.ndarray:
    """RHT of each consecutive 16 values (returns a new float32 array)."""
    a = np.array(w, dtype=np.float32, copy=True).reshape(-1)
    assert a.size % 16 == 0
    lib().orc_rht16_n(_p(a), a.size // 16, sign_mask & 0xFFFF)
    return a.reshape(np.shape(w))


def sumsq16(r) -> float:
    a = np.ascontiguousarray(r, dtype=np.float32)
    assert a.size == 16
    return float(lib().orc_sumsq16(_p(a)))


# ----------------------------------------------------------------- layouts


def sf_bytes(rows: int, nb: int, layout: int = SF_SWIZZLED) -> int:
    return int(lib().orc_sf_bytes(rows, nb, layout))


def sf_offset(r: int, c: int, nb: int, layout: int = SF_SWIZZLED) -> int:
    return int(lib().orc_sf_offset(r, c, nb, layout))


def sf_to_rowmajor(sf: np.ndarray, rows: int, nb: int, layout: int = SF_SWIZZLED) -> np.ndarray:
    """Gather a scale buffer in `layout` into a [rows, nb] array."""
    if layout == SF_ROWMAJOR:
        return sf[: rows * nb].reshape(rows, nb).copy()
    r = np.arange(rows)[:, None]
    c = np.arange(nb)[None, :]
    n_ct = (nb + 3) // 4
    off = ((r // 128) * n_ct + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)
    return sf[off]


# ---------------------------------------------------------------- quantize


@dataclass
class QResult:
    codes: np.ndarray  # uint8 [R_out, ld_codes]
    sf: np.ndarray  # uint8 flat, sf_bytes(R_out, nb, layout)
    tensor_scale: float
    choice: np.ndarray  # uint32 [R_out, ceil(nb/32)]
    rows: int  # R_out
    cols: int  # C_out
    sf_layout: int


def quantize(
    x_bf16: np.ndarray,
    *,
    scale_rule: int = SCALE_4OVER6,
    rounding: int = ROUND_RNE,
    block_2d: bool = False,
    transpose: bool = False,
    hadamard: bool = False,
    sf_layout: int = SF_SWIZZLED,
    sr_seed: int = 0,
    hadamard_seed: int = 0,
    amax: float | None = None,
    ld: int | None = None,
    ld_codes: int | None = None,
    src_row0: int = 0,
    src_cols: int = 0,
) -> QResult:
    """Quantize a bf16 matrix given as uint16 bit patterns [rows, cols].

    `ld` > cols quantizes the first `cols` columns of an array whose rows are
    `ld` elements long (pass the full [rows, ld] array)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows = x.shape[0]
    cols = x.shape[1]
    if ld is None:
        ld = cols
    else:
        cols, ld = ld, x.shape[1]
    return _quantize(x, rows, cols, ld, scale_rule, rounding, block_2d, transpose, hadamard,
                     sf_layout, sr_seed, hadamard_seed, amax, ld_codes, src_row0, src_cols)


def quantize_view(x_bf16: np.ndarray, cols: int, **kw) -> QResult:
    """Quantize the first `cols` columns of a [rows, ld] bf16 (uint16) array."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, ld = x.shape
    return _quantize(x, rows, cols, ld, kw.get("scale_rule", SCALE_4OVER6), kw.get("rounding", ROUND_RNE),
                     kw.get("block_2d", False), kw.get("transpose", False), kw.get("hadamard", False),
                     kw.get("sf_layout", SF_SWIZZLED), kw.get("sr_seed", 0), kw.get("hadamard_seed", 0),
                     kw.get("amax", None), kw.get("ld_codes", None), kw.get("src_row0", 0), kw.get("src_cols", 0))


def _quantize(x, rows, cols, ld, scale_rule, rounding, block_2d, transpose, hadamard, sf_layout,
              sr_seed, hadamard_seed, amax, ld_codes, src_row0=0, src_cols=0) -> QResult:
    R, C = (cols, rows) if transpose else (rows, cols)
    nb = C // 16
    ldc = C // 2 if ld_codes is None else ld_codes
    codes = np.zeros((max(R, 1), max(ldc, 1)), np.uint8)
    sf = np.zeros(max(sf_bytes(R, nb, sf_layout), 1), np.uint8)
    nw = (nb + 31) // 32
    choice = np.zeros((max(R, 1), max(nw, 1)), np.uint32)
    ts = np.zeros(1, np.float32)
    o = _Opts(scale_rule, rounding, int(block_2d), int(transpose), int(hadamard), sf_layout,
              sr_seed, hadamard_seed, 0 if amax is None else 1, 0.0 if amax is None else amax, src_row0, src_cols)
    rc = lib().orc_quantize(_p(x), rows, cols, ld, ctypes.byref(o), _p(codes), ldc, _p(sf), _p(ts),
                            _p(choice))
    if rc != 0:
        raise ValueError(f"oracle rejected shape rows={rows} cols={cols} with these options")
    return QResult(codes[:R, :ldc], sf[: sf_bytes(R, nb, sf_layout)], float(ts[0]), choice[:R, :nw], R, C,
                   sf_layout)


def dequantize(q: QResult) -> np.ndarray:
    """x_hat = g * (sf * s_t) as float32 [R_out, C_out]."""
    out = np.empty((q.rows, q.cols), np.float32)
    codes = np.ascontiguousarray(q.codes)
    lib().orc_dequantize(_p(codes), q.rows, q.cols, codes.shape[1], _p(q.sf), q.sf_layout,
                         q.tensor_scale, _p(out))
    return out


def gemm_rows(A_hat: np.ndarray, W_hat: np.ndarray, rows) -> tuple[np.ndarray, np.ndarray]:
    """FP64 reference of (A_hat W_hat^T)[rows, :] and the bound sum_k |a||w|."""
    A = np.ascontiguousarray(A_hat, dtype=np.float32)
    W = np.ascontiguousarray(W_hat, dtype=np.float32)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    N, K = W.shape
    out = np.empty((r.size, N), np.float64)
    bnd = np.empty((r.size, N), np.float64)
    lib().orc_gemm_rows(_p(A), _p(W), N, K, _p(r), r.size, _p(out), _p(bnd))
    return out, bnd


def gemm_rows_matmul(A_hat: np.ndarray, W_hat: np.ndarray, rows) -> tuple[np.ndarray, np.ndarray]:
    """The same FP64 reference as ``gemm_rows`` -- the FP32-simulation fallback
    of "Four Over Six" (first section): dequantize, then multiply -- with the
    K-sums done by numpy's float64 matmul (a library primitive) instead of the
    plain loop, for full-size shapes where the loop takes minutes.  Each sum is
    over exact products of FP32 values in FP64, so it agrees with
    ``gemm_rows`` to FP64 rounding (pinned against it in the CPU tests)."""
    r = np.asarray(rows, dtype=np.int64)
    a = np.asarray(A_hat, dtype=np.float32)[r].astype(np.float64)
    w = np.asarray(W_hat, dtype=np.float32).astype(np.float64)
    return a @ w.T, np.abs(a) @ np.abs(w).T


def mae_nearest_grid(x, block: int) -> float:
    a = np.ascontiguousarray(x, dtype=np.float32)
    assert a.size % block == 0
    return float(lib().orc_mae_nearest_grid(_p(a), a.size, block))


def linear_backward_operands(dy, x, w, *, scale_rule: int = SCALE_4OVER6, grad_rounding: int = ROUND_SR,
                             wgrad_hadamard: bool = True, weight_2d: bool = False, sr_seed: int = 0,
                             hadamard_seed: int = 0) -> list[QResult]:
    """The four quantized operands of the quantized linear layer's backward for
    Y = X W^T (dy [M, N], x [M, K], w [N, K] as bf16 bit patterns).

    "Four Over Six" ("Training") gives its quantized linear layer a backward
    pass; the FP4 glossary page ("FP4 ile Çıkarım ve Eğitim") names the recipe:
    random Hadamard transforms against outliers, stochastic rounding for
    gradients.  Each product contracts over one dimension, and both of its
    operands are blocked along that dimension:
      dX = dY W     over N: [dY along N, W^T along N]
      dW = dY^T X   over M: [dY^T along M, X^T along M] (RHT along M on both)
    Returns [dY, W^T, dY^T, X^T]."""
    return [
        quantize(dy, scale_rule=scale_rule, rounding=grad_rounding, sr_seed=sr_seed),
        quantize(w, scale_rule=scale_rule, transpose=True, block_2d=weight_2d),
        quantize(dy, scale_rule=scale_rule, rounding=grad_rounding, transpose=True, hadamard=wgrad_hadamard,
                 sr_seed=sr_seed, hadamard_seed=hadamard_seed),
        quantize(x, scale_rule=scale_rule, transpose=True, hadamard=wgrad_hadamard, hadamard_seed=hadamard_seed),
    ]


def linear_backward_rows(ops: list[QResult], dx_rows, dw_rows, matmul: bool = False):
    """FP64 references (and the sum |a||b| bounds) of the sampled rows of
    dX = dY_hat W^T_hat^T and dW = dY^T_hat X^T_hat^T from the dequantized
    operands of ``linear_backward_operands``."""
    f = gemm_rows_matmul if matmul else gemm_rows
    dx = f(dequantize(ops[0]), dequantize(ops[1]), dx_rows)
    dw = f(dequantize(ops[2]), dequantize(ops[3]), dw_rows)
    return dx, dw


# ----------------------------------------------------------------- MXFP4


def e8m0_decode(b: int) -> float:
    """R12: E8M0 byte -> 2^(b - 127) (0xFF: NaN)."""
    return float(lib().orc_e8m0_decode(int(b)))


def mx_exponent(a: float, m: int) -> int:
    """R12: the candidate exponent, X6 = floor(log2 a) - 2 (m = 6, the MX
    specification's shared exponent) or X6 + 1 (m = 4), clamped to [-127, 127]."""
    return int(lib().orc_mx_exponent(float(a), int(m)))


@dataclass
class MXResult:
    codes: np.ndarray   # uint8 [rows, cols/2]
    scales: np.ndarray  # uint8 [rows, cols/32], E8M0
    choice: np.ndarray  # uint8 [rows, cols/32], 1 = kept the 4-candidate
    rows: int
    cols: int


def quantize_mx(x_bf16: np.ndarray, scale_rule: int = SCALE_4OVER6) -> MXResult:
    """MXFP4 with the 4/6 choice (reading R12 of ``fos_oracle.c``): 32-value
    blocks along the rows of a bf16 (uint16 bits) matrix, one E8M0 scale each,
    no tensor scale.  The FP4 glossary page ("FP4 Nasıl Çalışır") defines the
    format; the candidate rule is this build's reading."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, cols = x.shape
    assert cols % 32 == 0
    codes = np.zeros((max(rows, 1), max(cols // 2, 1)), np.uint8)
    scales = np.zeros((max(rows, 1), max(cols // 32, 1)), np.uint8)
    choice = np.zeros_like(scales)
    if rows and cols:
        rc = lib().orc_quantize_mx(_p(x), rows, cols, cols, scale_rule, _p(codes), codes.shape[1], _p(scales),
                                   _p(choice))
        assert rc == 0
    return MXResult(codes=codes[:rows, : cols // 2], scales=scales[:rows, : cols // 32],
                    choice=choice[:rows, : cols // 32], rows=rows, cols=cols)


def dequantize_mx(q: MXResult) -> np.ndarray:
    """R12: x_hat = g * 2^X as float32 [rows, cols]."""
    out = np.empty((q.rows, q.cols), np.float32)
    codes = np.ascontiguousarray(q.codes)
    scales = np.ascontiguousarray(q.scales)
    lib().orc_dequantize_mx(_p(codes), _p(scales), q.rows, q.cols, codes.shape[1], _p(out))
    return out
