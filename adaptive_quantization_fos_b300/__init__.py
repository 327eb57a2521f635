"""Python binding of libfos.so -- Four Over Six NVFP4 quantization on B300.

The C ABI (include/fos.h) is called through ctypes with raw device pointers
taken from torch tensors; torch provides device memory and streams only.
Every step of the computation runs in the library's CUDA kernels.  There is
no CPU fallback: importing this package fails loudly when libfos.so is
missing, and every call raises on a non-OK status.

Low-level names mirror the C functions (``fos_quantize``, ``fos_dequantize``,
``fos_gemm``, ...).  ``quantize`` / ``dequantize`` / ``gemm`` are thin
conveniences that allocate the output tensors with torch and call them.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfos.so")

FOS_OK, FOS_ERR_INVALID_ARG, FOS_ERR_UNSUPPORTED, FOS_ERR_CUDA, FOS_ERR_TIMEOUT = 0, 1, 2, 3, 4
FOS_SCALE_4OVER6, FOS_SCALE_6, FOS_SCALE_4 = 0, 1, 2
FOS_ROUND_RNE, FOS_ROUND_STOCHASTIC = 0, 1
FOS_SF_SWIZZLED_128x4, FOS_SF_ROWMAJOR = 0, 1
FOS_DTYPE_F32, FOS_DTYPE_BF16 = 0, 1


class FosError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib.fos_status_string(status).decode()} (status {status})")


class fos_quant_options(ctypes.Structure):
    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("scale_rule", ctypes.c_int32),
        ("rounding", ctypes.c_int32),
        ("block_2d", ctypes.c_int32),
        ("transpose", ctypes.c_int32),
        ("hadamard", ctypes.c_int32),
        ("sf_layout", ctypes.c_int32),
        ("one_launch", ctypes.c_int32),
        ("sr_seed", ctypes.c_uint64),
        ("hadamard_seed", ctypes.c_uint64),
        ("tensor_amax", ctypes.c_void_p),
    ]


class fos_quant_job(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
        ("ld_x", ctypes.c_int64),
        ("codes", ctypes.c_void_p),
        ("ld_codes", ctypes.c_int64),
        ("sf", ctypes.c_void_p),
        ("tensor_scale", ctypes.c_void_p),
        ("choice", ctypes.c_void_p),
    ]


class fos_nvfp4_tensor(ctypes.Structure):
    _fields_ = [
        ("codes", ctypes.c_void_p),
        ("sf", ctypes.c_void_p),
        ("tensor_scale", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
        ("ld_codes", ctypes.c_int64),
        ("sf_layout", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class fos_mxfp4_tensor(ctypes.Structure):
    _fields_ = [
        ("codes", ctypes.c_void_p),
        ("sf", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
        ("ld_codes", ctypes.c_int64),
        ("sf_layout", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class fos_backward_options(ctypes.Structure):
    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("scale_rule", ctypes.c_int32),
        ("grad_rounding", ctypes.c_int32),
        ("wgrad_hadamard", ctypes.c_int32),
        ("weight_2d", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("sr_seed", ctypes.c_uint64),
        ("hadamard_seed", ctypes.c_uint64),
    ]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python adaptive_quantization_fos_b300/build.py` "
            "(there is no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, u64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int32, ctypes.c_size_t
    sig = {
        "fos_abi_version": (i32, []),
        "fos_status_string": (ctypes.c_char_p, [i32]),
        "fos_sf_bytes": (i32, [i64, i64, i32, ctypes.POINTER(sz)]),
        "fos_quantize_workspace_size": (i32, [i64, i64, ctypes.POINTER(fos_quant_options), ctypes.POINTER(sz)]),
        "fos_tensor_amax": (i32, [vp, i64, i64, i64, i32, i32, u64, vp, vp, sz, vp]),
        "fos_quantize": (i32, [vp, i64, i64, i64, ctypes.POINTER(fos_quant_options), vp, i64, vp, vp, vp, vp, sz,
                               vp]),
        "fos_quantize_noalloc": (i32, [vp, i64, i64, i64, ctypes.POINTER(fos_quant_options), vp, i64, vp, vp, vp,
                                       vp]),
        "fos_dequantize": (i32, [ctypes.POINTER(fos_nvfp4_tensor), vp, i32, i64, vp]),
        "fos_gemm": (i32, [ctypes.POINTER(fos_nvfp4_tensor), ctypes.POINTER(fos_nvfp4_tensor), vp, i64, vp, vp]),
        "fos_e2m1_encode": (i32, [vp, i64, vp, vp]),
        "fos_e4m3_encode": (i32, [vp, i64, vp, vp]),
        "fos_philox4x32_10": (i32, [vp, i64, u64, vp, vp]),
        "fos_selftest_wait_limits": (i32, [vp, sz, u64, vp, vp]),
        "fos_selftest_mma_rate": (i32, [i32, i64, i32, vp, vp]),
        "fos_quantize_batch_workspace_size": (i32, [i32, ctypes.POINTER(sz)]),
        "fos_quantize_batch": (i32, [ctypes.POINTER(fos_quant_job), i32, ctypes.POINTER(fos_quant_options), vp, sz,
                                     vp]),
        "fos_linear_backward_workspace_size": (i32, [i64, i64, i64, ctypes.POINTER(sz)]),
        "fos_mxfp4_sf_bytes": (i32, [i64, i64, i32, ctypes.POINTER(sz)]),
        "fos_quantize_mxfp4": (i32, [vp, i64, i64, i64, i32, i32, vp, i64, vp, vp, vp]),
        "fos_dequantize_mxfp4": (i32, [ctypes.POINTER(fos_mxfp4_tensor), vp, i32, i64, vp]),
        "fos_gemm_mxfp4": (i32, [ctypes.POINTER(fos_mxfp4_tensor), ctypes.POINTER(fos_mxfp4_tensor), vp, i64, vp,
                                 vp]),
        "fos_linear_forward_workspace_size": (i32, [i64, i64, ctypes.POINTER(sz)]),
        "fos_linear_forward_operand": (i32, [i64, i64, vp, sz, ctypes.POINTER(fos_nvfp4_tensor)]),
        "fos_linear_forward": (i32, [vp, i64, i64, i64, ctypes.POINTER(fos_quant_options),
                                     ctypes.POINTER(fos_nvfp4_tensor), vp, i64, vp, sz, vp, vp]),
        "fos_linear_backward_operands": (i32, [i64, i64, i64, vp, sz, ctypes.POINTER(fos_nvfp4_tensor)]),
        "fos_linear_backward": (i32, [vp, i64, vp, i64, vp, i64, i64, i64, i64, ctypes.POINTER(fos_backward_options),
                                      vp, i64, vp, i64, vp, sz, vp, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


_lib = _load()
EXPORTED = ("fos_abi_version", "fos_status_string", "fos_sf_bytes", "fos_quantize_workspace_size",
            "fos_tensor_amax", "fos_quantize", "fos_quantize_noalloc", "fos_dequantize", "fos_gemm", "fos_e2m1_encode",
            "fos_e4m3_encode", "fos_philox4x32_10", "fos_selftest_wait_limits", "fos_quantize_batch",
            "fos_quantize_batch_workspace_size", "fos_linear_backward", "fos_linear_backward_workspace_size",
            "fos_linear_backward_operands", "fos_linear_forward", "fos_linear_forward_workspace_size",
            "fos_linear_forward_operand", "fos_mxfp4_sf_bytes", "fos_quantize_mxfp4", "fos_dequantize_mxfp4",
            "fos_gemm_mxfp4", "fos_selftest_mma_rate")


def _check(status: int, what: str) -> None:
    if status != FOS_OK:
        raise FosError(status, what)


# ------------------------------------------------------- C-named wrappers


def fos_abi_version() -> int:
    return int(_lib.fos_abi_version())


def fos_sf_bytes(out_rows: int, out_cols: int, sf_layout: int = FOS_SF_SWIZZLED_128x4) -> int:
    n = ctypes.c_size_t()
    _check(_lib.fos_sf_bytes(out_rows, out_cols, sf_layout, ctypes.byref(n)), "fos_sf_bytes")
    return n.value


def fos_quantize_workspace_size(rows: int, cols: int, opt: fos_quant_options) -> int:
    n = ctypes.c_size_t()
    _check(_lib.fos_quantize_workspace_size(rows, cols, ctypes.byref(opt), ctypes.byref(n)),
           "fos_quantize_workspace_size")
    return n.value


def fos_quantize(x, rows, cols, ld_x, opt, codes, ld_codes, sf, tensor_scale, choice, workspace, workspace_bytes,
                 stream) -> int:
    """Raw call: all buffer arguments are integer device addresses (0 = NULL)."""
    return int(_lib.fos_quantize(x, rows, cols, ld_x, ctypes.byref(opt), codes, ld_codes, sf, tensor_scale,
                                 choice or None, workspace or None, workspace_bytes, stream))


def fos_quantize_noalloc(x, rows, cols, ld_x, opt, codes, ld_codes, sf, tensor_scale, choice, stream) -> int:
    """Raw call of the entry point that needs no workspace (for callers that
    cannot allocate device memory); buffers are integer device addresses."""
    return int(_lib.fos_quantize_noalloc(x, rows, cols, ld_x, ctypes.byref(opt), codes, ld_codes, sf, tensor_scale,
                                         choice or None, stream))


def fos_tensor_amax(x, rows, cols, ld_x, hadamard, transpose, hadamard_seed, amax_out, workspace,
                    workspace_bytes, stream) -> int:
    return int(_lib.fos_tensor_amax(x, rows, cols, ld_x, hadamard, transpose, hadamard_seed, amax_out, workspace,
                                    workspace_bytes, stream))


def fos_dequantize(q: fos_nvfp4_tensor, out, out_dtype, ld_out, stream) -> int:
    return int(_lib.fos_dequantize(ctypes.byref(q), out, out_dtype, ld_out, stream))


def fos_gemm(A: fos_nvfp4_tensor, B: fos_nvfp4_tensor, C, ldc, dev_status, stream) -> int:
    return int(_lib.fos_gemm(ctypes.byref(A), ctypes.byref(B), C, ldc, dev_status or None, stream))


def fos_selftest_wait_limits(scratch, scratch_bytes, timeout_ns, result, stream) -> int:
    return int(_lib.fos_selftest_wait_limits(scratch, scratch_bytes, timeout_ns, result, stream))


def fos_selftest_mma_rate(n_cols, iters, grid, dev_status, stream) -> int:
    return int(_lib.fos_selftest_mma_rate(n_cols, iters, grid, dev_status or None, stream))


def fos_e2m1_encode(x, n, codes, stream) -> int:
    return int(_lib.fos_e2m1_encode(x, n, codes, stream))


def fos_e4m3_encode(x, n, out, stream) -> int:
    return int(_lib.fos_e4m3_encode(x, n, out, stream))


def fos_philox4x32_10(counters, n, key, out, stream) -> int:
    return int(_lib.fos_philox4x32_10(counters, n, key, out, stream))


# -------------------------------------------------------- torch helpers


def _torch():
    import torch

    return torch


def _stream_ptr(stream=None) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def options(*, scale_rule=FOS_SCALE_4OVER6, rounding=FOS_ROUND_RNE, block_2d=False, transpose=False,
            hadamard=False, sf_layout=FOS_SF_SWIZZLED_128x4, sr_seed=0, hadamard_seed=0,
            tensor_amax=None, one_launch=False) -> fos_quant_options:
    o = fos_quant_options()
    o.struct_size = ctypes.sizeof(fos_quant_options)
    o.scale_rule = scale_rule
    o.rounding = rounding
    o.block_2d = int(bool(block_2d))
    o.transpose = int(bool(transpose))
    o.hadamard = int(bool(hadamard))
    o.sf_layout = sf_layout
    o.one_launch = int(bool(one_launch))
    o.sr_seed = sr_seed
    o.hadamard_seed = hadamard_seed
    o.tensor_amax = None if tensor_amax is None else int(tensor_amax.data_ptr())
    return o


@dataclass
class NVFP4Tensor:
    """Device buffers of one quantized matrix (rows x cols values, blocks along cols)."""

    codes: "object"  # uint8 [rows, ld_codes]
    sf: "object"  # uint8 flat, fos_sf_bytes(rows, cols, sf_layout)
    tensor_scale: "object"  # float32 [1]
    rows: int
    cols: int
    sf_layout: int
    choice: "object" = None  # uint8 [rows, cols/16] or None

    def as_c(self) -> fos_nvfp4_tensor:
        t = fos_nvfp4_tensor()
        t.codes = self.codes.data_ptr()
        t.sf = self.sf.data_ptr()
        t.tensor_scale = self.tensor_scale.data_ptr()
        t.rows = self.rows
        t.cols = self.cols
        t.ld_codes = self.codes.stride(0) if self.codes.dim() == 2 else self.cols // 2
        t.sf_layout = self.sf_layout
        return t


class Quantizer:
    """Reusable output/workspace buffers for repeated quantization of one shape."""

    def __init__(self, rows: int, cols: int, *, device="cuda", with_choice=False, **opts):
        torch = _torch()
        self.rows, self.cols = rows, cols
        self.opt_kwargs = dict(opts)
        self.opt = options(**opts)
        tr = bool(opts.get("transpose", False))
        self.R, self.C = (cols, rows) if tr else (rows, cols)
        layout = opts.get("sf_layout", FOS_SF_SWIZZLED_128x4)
        ldc = max(8, ((self.C // 2 + 15) // 16) * 16)
        self.out = NVFP4Tensor(
            codes=torch.empty((self.R, ldc), dtype=torch.uint8, device=device),
            sf=torch.empty(max(1, fos_sf_bytes(self.R, self.C, layout)), dtype=torch.uint8, device=device),
            tensor_scale=torch.empty(1, dtype=torch.float32, device=device),
            rows=self.R, cols=self.C, sf_layout=layout,
            choice=torch.empty((self.R, self.C // 16), dtype=torch.uint8, device=device) if with_choice else None)
        self.ws_bytes = fos_quantize_workspace_size(rows, cols, self.opt)
        self.workspace = torch.empty(max(1, self.ws_bytes), dtype=torch.uint8, device=device)

    def __call__(self, x, stream=None) -> NVFP4Tensor:
        assert x.dtype == _torch().bfloat16 and x.dim() == 2 and x.shape == (self.rows, self.cols)
        assert x.stride(1) == 1
        o = self.out
        st = fos_quantize(x.data_ptr(), self.rows, self.cols, x.stride(0), self.opt, o.codes.data_ptr(),
                          o.codes.stride(0), o.sf.data_ptr(), o.tensor_scale.data_ptr(),
                          o.choice.data_ptr() if o.choice is not None else 0, self.workspace.data_ptr(),
                          self.ws_bytes, _stream_ptr(stream))
        _check(st, "fos_quantize")
        return o


def fos_quantize_batch_workspace_size(n_jobs: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.fos_quantize_batch_workspace_size(n_jobs, ctypes.byref(n)), "fos_quantize_batch_workspace_size")
    return n.value


def fos_quantize_batch(jobs, opt: fos_quant_options, workspace, workspace_bytes, stream) -> int:
    """Raw call: jobs is a sequence of fos_quant_job (or a ctypes array of
    them); buffers are device addresses."""
    arr = jobs if isinstance(jobs, ctypes.Array) else (fos_quant_job * len(jobs))(*jobs)
    return int(_lib.fos_quantize_batch(arr, len(arr), ctypes.byref(opt), workspace or None, workspace_bytes, stream))


class BatchQuantizer:
    """Reusable outputs and workspace for repeated quantization of a fixed set
    of matrices (e.g. one layer's weights) in one batch call.  shapes are the
    sources' [rows, cols]; with transpose=True each output is [cols, rows]."""

    def __init__(self, shapes, *, device="cuda", with_choice=False, **opts):
        torch = _torch()
        self.opt = options(**opts)
        self.shapes = [tuple(s) for s in shapes]
        tr = bool(opts.get("transpose", False))
        layout = opts.get("sf_layout", FOS_SF_SWIZZLED_128x4)
        self.outs = []
        for rows, cols in self.shapes:
            R, C = (cols, rows) if tr else (rows, cols)
            ldc = max(8, ((C // 2 + 15) // 16) * 16)
            self.outs.append(NVFP4Tensor(
                codes=torch.empty((R, ldc), dtype=torch.uint8, device=device),
                sf=torch.empty(max(1, fos_sf_bytes(R, C, layout)), dtype=torch.uint8, device=device),
                tensor_scale=torch.empty(1, dtype=torch.float32, device=device),
                rows=R, cols=C, sf_layout=layout,
                choice=torch.empty((R, C // 16), dtype=torch.uint8, device=device) if with_choice else None))
        self.ws_bytes = fos_quantize_batch_workspace_size(len(self.outs))
        self.workspace = torch.empty(max(1, self.ws_bytes), dtype=torch.uint8, device=device)
        # the job array of the last call, reused while the inputs stay the same
        # tensors (the outputs never change): a repeated call only checks them
        self._key = None
        self._jobs = None

    def __call__(self, xs, stream=None):
        assert len(xs) == len(self.outs)
        bf16 = _torch().bfloat16
        key = tuple((x.data_ptr(), x.stride(0), x.stride(1)) if x.numel() else (0, 0, 0) for x in xs)
        if key != self._key:
            jobs = []
            for x, shape, o in zip(xs, self.shapes, self.outs):
                assert x.dtype == bf16 and tuple(x.shape) == shape
                assert x.numel() == 0 or x.stride(1) == 1
                ld = x.stride(0) if x.numel() else max(shape[1], 8)
                jobs.append(fos_quant_job(x.data_ptr(), shape[0], shape[1], ld, o.codes.data_ptr(),
                                          o.codes.stride(0), o.sf.data_ptr(), o.tensor_scale.data_ptr(),
                                          o.choice.data_ptr() if o.choice is not None else None))
            self._jobs = (fos_quant_job * len(jobs))(*jobs)
            self._key = key
        else:
            for x, shape in zip(xs, self.shapes):
                assert x.dtype == bf16 and tuple(x.shape) == shape
        _check(fos_quantize_batch(self._jobs, self.opt, self.workspace.data_ptr(), self.ws_bytes, _stream_ptr(stream)),
               "fos_quantize_batch")
        return self.outs


def quantize(x, *, with_choice=False, stream=None, **opts) -> NVFP4Tensor:
    """Quantize a bf16 [rows, cols] CUDA tensor (contiguous rows) to NVFP4."""
    q = Quantizer(x.shape[0], x.shape[1], device=x.device, with_choice=with_choice, **opts)
    return q(x, stream=stream)


def tensor_amax(x, *, hadamard=False, transpose=False, hadamard_seed=0, stream=None):
    torch = _torch()
    out = torch.empty(1, dtype=torch.float32, device=x.device)
    ws = torch.empty(fos_quantize_workspace_size(x.shape[0], x.shape[1], options()), dtype=torch.uint8,
                     device=x.device)
    _check(fos_tensor_amax(x.data_ptr(), x.shape[0], x.shape[1], x.stride(0), int(hadamard), int(transpose),
                           hadamard_seed, out.data_ptr(), ws.data_ptr(), ws.numel(), _stream_ptr(stream)),
           "fos_tensor_amax")
    return out


def dequantize(q: NVFP4Tensor, dtype=None, stream=None):
    torch = _torch()
    dtype = torch.float32 if dtype is None else dtype
    out = torch.empty((q.rows, q.cols), dtype=dtype, device=q.codes.device)
    code = FOS_DTYPE_BF16 if dtype == torch.bfloat16 else FOS_DTYPE_F32
    _check(fos_dequantize(q.as_c(), out.data_ptr(), code, q.cols, _stream_ptr(stream)), "fos_dequantize")
    return out


def gemm(A: NVFP4Tensor, B: NVFP4Tensor, out=None, status=None, stream=None):
    """C = A . B^T (bf16) from two NVFP4 operands quantized along K."""
    torch = _torch()
    if out is None:
        out = torch.empty((A.rows, B.rows), dtype=torch.bfloat16, device=A.codes.device)
    _check(fos_gemm(A.as_c(), B.as_c(), out.data_ptr(), out.stride(0),
                    status.data_ptr() if status is not None else 0, _stream_ptr(stream)), "fos_gemm")
    return out


# ------------------------------------------------------- linear backward


def fos_linear_backward_workspace_size(M: int, N: int, K: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.fos_linear_backward_workspace_size(M, N, K, ctypes.byref(n)), "fos_linear_backward_workspace_size")
    return n.value


def fos_linear_backward_operands(M: int, N: int, K: int, workspace, workspace_bytes: int):
    """Raw call: the four fos_nvfp4_tensor descriptors inside a workspace."""
    ops = (fos_nvfp4_tensor * 4)()
    _check(_lib.fos_linear_backward_operands(M, N, K, workspace, workspace_bytes, ops),
           "fos_linear_backward_operands")
    return list(ops)


def fos_linear_backward(dy, ld_dy, x, ld_x, w, ld_w, M, N, K, opt: fos_backward_options, dx, ld_dx, dw, ld_dw,
                        workspace, workspace_bytes, dev_status, stream) -> int:
    return int(_lib.fos_linear_backward(dy, ld_dy, x or None, ld_x, w or None, ld_w, M, N, K, ctypes.byref(opt),
                                        dx or None, ld_dx, dw or None, ld_dw, workspace, workspace_bytes,
                                        dev_status or None, stream))


def backward_options(*, scale_rule=FOS_SCALE_4OVER6, grad_rounding=FOS_ROUND_STOCHASTIC, wgrad_hadamard=True,
                     weight_2d=False, sr_seed=0, hadamard_seed=0) -> fos_backward_options:
    """Defaults follow the FP4 training recipe: stochastic rounding of dY and
    the RHT on the weight-gradient operands."""
    o = fos_backward_options()
    o.struct_size = ctypes.sizeof(fos_backward_options)
    o.scale_rule = scale_rule
    o.grad_rounding = grad_rounding
    o.wgrad_hadamard = int(bool(wgrad_hadamard))
    o.weight_2d = int(bool(weight_2d))
    o.reserved = 0
    o.sr_seed = sr_seed
    o.hadamard_seed = hadamard_seed
    return o


class LinearBackward:
    """dX = dY W and dW = dY^T X for Y = X W^T, through fos_linear_backward,
    with a reusable workspace for one M x N x K shape."""

    def __init__(self, M: int, N: int, K: int, *, device="cuda", **opts):
        torch = _torch()
        self.M, self.N, self.K = M, N, K
        self.opt = backward_options(**opts)
        self.ws_bytes = fos_linear_backward_workspace_size(M, N, K)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)

    def __call__(self, dy, x, w, *, dx=None, dw=None, need_dx=True, need_dw=True, status=None, stream=None):
        torch = _torch()
        M, N, K = self.M, self.N, self.K
        for t, shape in ((dy, (M, N)), (x, (M, K)), (w, (N, K))):
            assert t is None or (t.dtype == torch.bfloat16 and tuple(t.shape) == shape and t.stride(1) == 1)
        dev = dy.device
        if need_dx and dx is None:
            dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        if need_dw and dw is None:
            dw = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
        dx = dx if need_dx else None
        dw = dw if need_dw else None
        st = fos_linear_backward(dy.data_ptr(), dy.stride(0), x.data_ptr() if x is not None else 0,
                                 x.stride(0) if x is not None else 0, w.data_ptr() if w is not None else 0,
                                 w.stride(0) if w is not None else 0, M, N, K, self.opt,
                                 dx.data_ptr() if dx is not None else 0, dx.stride(0) if dx is not None else 0,
                                 dw.data_ptr() if dw is not None else 0, dw.stride(0) if dw is not None else 0,
                                 self.workspace.data_ptr(), self.ws_bytes,
                                 status.data_ptr() if status is not None else 0, _stream_ptr(stream))
        _check(st, "fos_linear_backward")
        return dx, dw

    def operands(self):
        """[dY, W^T, dY^T, X^T] as NVFP4Tensor views into the workspace."""
        torch = _torch()
        base = self.workspace.data_ptr()
        out = []
        for d in fos_linear_backward_operands(self.M, self.N, self.K, base, self.ws_bytes):
            c0 = d.codes - base
            s0 = d.sf - base
            t0 = d.tensor_scale - base
            sfb = fos_sf_bytes(d.rows, d.cols, d.sf_layout)
            out.append(NVFP4Tensor(
                codes=self.workspace[c0:c0 + d.rows * d.ld_codes].view(d.rows, d.ld_codes),
                sf=self.workspace[s0:s0 + sfb], tensor_scale=self.workspace[t0:t0 + 4].view(torch.float32),
                rows=d.rows, cols=d.cols, sf_layout=d.sf_layout))
        return out


# ------------------------------------------------------- linear forward


def fos_linear_forward_workspace_size(M: int, K: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.fos_linear_forward_workspace_size(M, K, ctypes.byref(n)), "fos_linear_forward_workspace_size")
    return n.value


def fos_linear_forward_operand(M: int, K: int, workspace, workspace_bytes: int) -> fos_nvfp4_tensor:
    t = fos_nvfp4_tensor()
    _check(_lib.fos_linear_forward_operand(M, K, workspace, workspace_bytes, ctypes.byref(t)),
           "fos_linear_forward_operand")
    return t


def fos_linear_forward(x, ld_x, M, K, x_opt: fos_quant_options, w: fos_nvfp4_tensor, y, ld_y, workspace,
                       workspace_bytes, dev_status, stream) -> int:
    return int(_lib.fos_linear_forward(x, ld_x, M, K, ctypes.byref(x_opt), ctypes.byref(w), y, ld_y, workspace,
                                       workspace_bytes, dev_status or None, stream))


class LinearForward:
    """Y = X W^T through fos_linear_forward: X [M, K] quantized with the given
    options, then multiplied by W, an NVFP4Tensor quantized beforehand along K
    (with the same RHT seed when hadamard is set)."""

    def __init__(self, M: int, K: int, *, device="cuda", **opts):
        torch = _torch()
        self.M, self.K = M, K
        self.opt = options(**opts)
        self.ws_bytes = fos_linear_forward_workspace_size(M, K)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)

    def __call__(self, x, w: NVFP4Tensor, out=None, status=None, stream=None):
        torch = _torch()
        assert x.dtype == torch.bfloat16 and tuple(x.shape) == (self.M, self.K) and x.stride(1) == 1
        if out is None:
            out = torch.empty((self.M, w.rows), dtype=torch.bfloat16, device=x.device)
        st = fos_linear_forward(x.data_ptr(), x.stride(0), self.M, self.K, self.opt, w.as_c(), out.data_ptr(),
                                out.stride(0), self.workspace.data_ptr(), self.ws_bytes,
                                status.data_ptr() if status is not None else 0, _stream_ptr(stream))
        _check(st, "fos_linear_forward")
        return out

    def operand(self) -> NVFP4Tensor:
        """X's quantized operand as a view into the workspace."""
        torch = _torch()
        base = self.workspace.data_ptr()
        d = fos_linear_forward_operand(self.M, self.K, base, self.ws_bytes)
        c0, s0, t0 = d.codes - base, d.sf - base, d.tensor_scale - base
        sfb = fos_sf_bytes(d.rows, d.cols, d.sf_layout)
        return NVFP4Tensor(codes=self.workspace[c0:c0 + d.rows * d.ld_codes].view(d.rows, d.ld_codes),
                           sf=self.workspace[s0:s0 + sfb], tensor_scale=self.workspace[t0:t0 + 4].view(torch.float32),
                           rows=d.rows, cols=d.cols, sf_layout=d.sf_layout)


# ------------------------------------------------------------------ MXFP4


def fos_mxfp4_sf_bytes(rows: int, cols: int, sf_layout: int = FOS_SF_SWIZZLED_128x4) -> int:
    n = ctypes.c_size_t()
    _check(_lib.fos_mxfp4_sf_bytes(rows, cols, sf_layout, ctypes.byref(n)), "fos_mxfp4_sf_bytes")
    return n.value


def fos_quantize_mxfp4(x, rows, cols, ld_x, scale_rule, sf_layout, codes, ld_codes, scales, choice, stream) -> int:
    return int(_lib.fos_quantize_mxfp4(x or None, rows, cols, ld_x, scale_rule, sf_layout, codes or None, ld_codes,
                                       scales or None, choice or None, stream))


def fos_dequantize_mxfp4(q: fos_mxfp4_tensor, out, out_dtype, ld_out, stream) -> int:
    return int(_lib.fos_dequantize_mxfp4(ctypes.byref(q), out or None, out_dtype, ld_out, stream))


def fos_gemm_mxfp4(A: fos_mxfp4_tensor, B: fos_mxfp4_tensor, C, ldc, dev_status, stream) -> int:
    return int(_lib.fos_gemm_mxfp4(ctypes.byref(A), ctypes.byref(B), C, ldc, dev_status or None, stream))


@dataclass
class MXFP4Tensor:
    """Device buffers of one MXFP4 matrix (rows x cols values, 32-value blocks along cols)."""

    codes: "object"   # uint8 [rows, ld_codes]
    scales: "object"  # uint8 E8M0: [rows, cols/32] (row-major) or flat fos_mxfp4_sf_bytes (swizzled)
    rows: int
    cols: int
    sf_layout: int = FOS_SF_SWIZZLED_128x4
    choice: "object" = None  # uint8 [rows, cols/32] or None

    def as_c(self) -> fos_mxfp4_tensor:
        t = fos_mxfp4_tensor()
        t.codes = self.codes.data_ptr()
        t.sf = self.scales.data_ptr()
        t.rows = self.rows
        t.cols = self.cols
        t.ld_codes = self.codes.stride(0) if self.codes.dim() == 2 else self.cols // 2
        t.sf_layout = self.sf_layout
        return t


def quantize_mxfp4(x, *, scale_rule=FOS_SCALE_4OVER6, sf_layout=FOS_SF_SWIZZLED_128x4, with_choice=False,
                   stream=None) -> MXFP4Tensor:
    """MXFP4 with the 4/6 choice of a bf16 [rows, cols] CUDA tensor (contiguous rows)."""
    torch = _torch()
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    ldc = max(16, ((cols // 2 + 15) // 16) * 16)
    if sf_layout == FOS_SF_ROWMAJOR:
        scales = torch.empty((rows, cols // 32), dtype=torch.uint8, device=x.device)
    else:
        scales = torch.empty(max(1, fos_mxfp4_sf_bytes(rows, cols, sf_layout)), dtype=torch.uint8, device=x.device)
    out = MXFP4Tensor(codes=torch.empty((rows, ldc), dtype=torch.uint8, device=x.device), scales=scales, rows=rows,
                      cols=cols, sf_layout=sf_layout,
                      choice=torch.empty((rows, cols // 32), dtype=torch.uint8, device=x.device) if with_choice
                      else None)
    _check(fos_quantize_mxfp4(x.data_ptr(), rows, cols, x.stride(0), scale_rule, sf_layout, out.codes.data_ptr(),
                              ldc, out.scales.data_ptr(), out.choice.data_ptr() if with_choice else 0,
                              _stream_ptr(stream)), "fos_quantize_mxfp4")
    return out


def dequantize_mxfp4(q: MXFP4Tensor, dtype=None, stream=None):
    torch = _torch()
    dtype = torch.float32 if dtype is None else dtype
    out = torch.empty((q.rows, q.cols), dtype=dtype, device=q.codes.device)
    code = FOS_DTYPE_BF16 if dtype == torch.bfloat16 else FOS_DTYPE_F32
    _check(fos_dequantize_mxfp4(q.as_c(), out.data_ptr(), code, q.cols, _stream_ptr(stream)),
           "fos_dequantize_mxfp4")
    return out


def gemm_mxfp4(A: MXFP4Tensor, B: MXFP4Tensor, out=None, status=None, stream=None):
    """C = A . B^T (bf16) from two MXFP4 operands quantized along K (swizzled scales)."""
    torch = _torch()
    if out is None:
        out = torch.empty((A.rows, B.rows), dtype=torch.bfloat16, device=A.codes.device)
    _check(fos_gemm_mxfp4(A.as_c(), B.as_c(), out.data_ptr(), out.stride(0),
                          status.data_ptr() if status is not None else 0, _stream_ptr(stream)), "fos_gemm_mxfp4")
    return out
