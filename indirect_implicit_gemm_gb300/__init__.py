"""Python binding of libconvgb.so, the sm_103a forward-convolution library.

Argument marshalling only: every step of every call runs in the CUDA kernels
of the shared library (include/convgb.h documents the ABI).  PyTorch supplies
device memory (its caching allocator) and the current CUDA stream.  There is
no CPU fallback: when the library or a GPU is missing, calls raise.

Layouts are channels-last: x [N, H, W, C_in] bf16, w [C_out, KH, KW, C_in]
bf16, bias [C_out] bf16 or None, y [N, H_out, W_out, C_out] bf16 or fp32.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "load", "conv2d_fwd", "conv2d_fwd_path", "conv2d_fwd_indirect", "im2win_transform", "build_indirection_buffer",
    "output_dims", "select_path", "workspace_size", "im2col_bytes", "im2win_bytes",
    "indirection_buffer_bytes", "check_device_errors", "set_wait_timeout_ns",
    "selftest_wait_timeout", "ConvgbError", "PATH_AUTO", "PATH_GATHER", "PATH_DENSE",
    "PATH_STEM", "PATH_WINDOW", "PATH_PLANE", "PATH_IM2WIN", "PATH_STEMWIN", "PATH_WINFOLD",
    "EXPORTED_SYMBOLS",
    "library_path",
    "conv2d_fwd_host", "conv2d_fwd_host_scratch_size", "plan_info", "set_tuning", "Plan",
]

PATH_AUTO, PATH_GATHER, PATH_DENSE, PATH_STEM, PATH_WINDOW, PATH_PLANE, PATH_IM2WIN = (
    0, 1, 2, 3, 4, 5, 6)
PATH_STEMWIN = 7
PATH_WINFOLD = 8
_BF16, _F32 = 0, 1
OK, ERR_INTERNAL = 0, 6

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libconvgb.so")
_lib = None

# Every symbol include/convgb.h declares.
EXPORTED_SYMBOLS = (
    "convgb_status_string", "convgb_output_dims", "convgb_select_path",
    "convgb_conv2d_fwd_workspace_size", "convgb_conv2d_fwd_path_workspace_size",
    "convgb_im2col_bytes", "conv2d_fwd", "conv2d_fwd_path", "conv2d_fwd_indirect",
    "conv2d_fwd_noalloc", "convgb_indirection_buffer_bytes",
    "build_indirection_buffer", "convgb_im2win_bytes", "im2win_transform",
    "convgb_check_device_errors", "convgb_set_wait_timeout_ns", "convgb_selftest_wait_timeout",
    "convgb_version", "convgb_conv2d_fwd_host_scratch_size", "conv2d_fwd_host",
    "convgb_plan_info", "convgb_set_tuning",
)


class Plan(ctypes.Structure):
    """convgb_plan: what conv2d_fwd_path launches for a shape (include/convgb.h)."""
    _fields_ = [(n, ctypes.c_int) for n in (
        "path", "a_mode", "bn", "m_tiles", "tile_rows", "n_tiles", "splits", "k_blocks", "stages",
        "weights_resident", "cta_pair", "tma_store", "epilogue_tiles", "epilogue_c32",
        "stream_k", "segment_outputs", "segment_rows")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class ConvgbError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = load().convgb_status_string(status).decode()
        super().__init__("%s%s (status %d)" % (what + ": " if what else "", msg, status))


def load():
    """Load libconvgb.so (built by __graft_entry__.build()); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise RuntimeError("libconvgb.so is not built (%s); run __graft_entry__.build()"
                           % library_path)
    lib = ctypes.CDLL(library_path)
    I, Z, P, U64 = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_uint64
    shape10 = [I] * 10
    lib.convgb_status_string.argtypes = [I]
    lib.convgb_status_string.restype = ctypes.c_char_p
    lib.convgb_output_dims.argtypes = [I] * 7 + [ctypes.POINTER(I), ctypes.POINTER(I)]
    lib.convgb_output_dims.restype = I
    lib.convgb_select_path.argtypes = shape10
    lib.convgb_select_path.restype = I
    lib.convgb_conv2d_fwd_workspace_size.argtypes = shape10
    lib.convgb_conv2d_fwd_workspace_size.restype = Z
    lib.convgb_conv2d_fwd_path_workspace_size.argtypes = [I] + shape10
    lib.convgb_conv2d_fwd_path_workspace_size.restype = Z
    lib.convgb_im2col_bytes.argtypes = [I] * 9
    lib.convgb_im2col_bytes.restype = Z
    conv_args = [P, P, P] + shape10 + [P, I, P, Z, P]
    lib.conv2d_fwd.argtypes = conv_args
    lib.conv2d_fwd.restype = I
    lib.conv2d_fwd_path.argtypes = [I] + conv_args
    lib.conv2d_fwd_path.restype = I
    lib.conv2d_fwd_indirect.argtypes = [P, P, P] + shape10 + [P, Z, P, I, P]
    lib.conv2d_fwd_indirect.restype = I
    lib.conv2d_fwd_noalloc.argtypes = [P, P, P] + shape10 + [P, I, P]
    lib.conv2d_fwd_noalloc.restype = I
    lib.convgb_conv2d_fwd_host_scratch_size.argtypes = shape10 + [I, I]
    lib.convgb_conv2d_fwd_host_scratch_size.restype = Z
    lib.conv2d_fwd_host.argtypes = conv_args
    lib.conv2d_fwd_host.restype = I
    lib.convgb_indirection_buffer_bytes.argtypes = [I] * 7
    lib.convgb_indirection_buffer_bytes.restype = Z
    lib.build_indirection_buffer.argtypes = [I] * 8 + [P, Z, P]
    lib.build_indirection_buffer.restype = I
    lib.convgb_im2win_bytes.argtypes = [I] * 9
    lib.convgb_im2win_bytes.restype = Z
    lib.im2win_transform.argtypes = [P] + [I] * 9 + [P, Z, P]
    lib.im2win_transform.restype = I
    lib.convgb_check_device_errors.argtypes = [P, ctypes.POINTER(ctypes.c_uint)]
    lib.convgb_check_device_errors.restype = I
    lib.convgb_set_wait_timeout_ns.argtypes = [U64]
    lib.convgb_set_wait_timeout_ns.restype = None
    lib.convgb_selftest_wait_timeout.argtypes = [U64, P]
    lib.convgb_selftest_wait_timeout.restype = I
    lib.convgb_plan_info.argtypes = [I] + shape10 + [I, ctypes.POINTER(Plan)]
    lib.convgb_plan_info.restype = I
    lib.convgb_set_tuning.argtypes = [I, I, I]
    lib.convgb_set_tuning.restype = None
    lib.convgb_version.argtypes = []
    lib.convgb_version.restype = I
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != OK:
        raise ConvgbError(status, what)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need_cuda(t, name, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous (channels-last layout)" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))


def plan_info(N, C_in, H, W, C_out, KH, KW, stride=1, pad=0, dilation=1, path=PATH_AUTO,
              out_dtype=torch.bfloat16) -> dict:
    """The tiling conv2d_fwd_path(path, ...) would launch for this shape (no launch)."""
    p = Plan()
    _check(load().convgb_plan_info(path, N, C_in, H, W, C_out, KH, KW, stride, pad, dilation,
                                   _F32 if out_dtype == torch.float32 else _BF16,
                                   ctypes.byref(p)), "plan_info")
    return p.as_dict()


def set_tuning(bn: int = 0, max_stages: int = 0, stream_k: int = 0):
    """Force the tile width, cap the ring depth and/or allow stream-K in later plans
    (0 = the planner's own choice)."""
    load().convgb_set_tuning(int(bn), int(max_stages), int(stream_k))
    _shape_cache.clear()  # workspace sizes follow the plan


# (path, N, C_in, H, W, C_out, KH, KW, stride, pad, dilation) -> (H_out, W_out,
# workspace bytes): the per-call queries of conv2d_fwd_path, made once per shape
_shape_cache = {}


def _shape_info(lib, key):
    got = _shape_cache.get(key)
    if got is None:
        path, N, C_in, H, W, C_out, KH, KW, stride, pad, dilation = key
        H_out, W_out = output_dims(H, W, KH, KW, stride, pad, dilation)
        need = lib.convgb_conv2d_fwd_path_workspace_size(path, N, C_in, H, W, C_out, KH, KW,
                                                         stride, pad, dilation)
        got = (H_out, W_out, need)
        if len(_shape_cache) > 4096:
            _shape_cache.clear()
        _shape_cache[key] = got
    return got


def output_dims(H, W, KH, KW, stride=1, pad=0, dilation=1):
    ho, wo = ctypes.c_int(), ctypes.c_int()
    _check(load().convgb_output_dims(H, W, KH, KW, stride, pad, dilation, ctypes.byref(ho),
                                     ctypes.byref(wo)), "output_dims")
    return ho.value, wo.value


def select_path(N, C_in, H, W, C_out, KH, KW, stride=1, pad=0, dilation=1) -> int:
    return load().convgb_select_path(N, C_in, H, W, C_out, KH, KW, stride, pad, dilation)


def workspace_size(N, C_in, H, W, C_out, KH, KW, stride=1, pad=0, dilation=1,
                   path=PATH_AUTO) -> int:
    return load().convgb_conv2d_fwd_path_workspace_size(path, N, C_in, H, W, C_out, KH, KW,
                                                        stride, pad, dilation)


def im2col_bytes(N, C_in, H, W, KH, KW, stride=1, pad=0, dilation=1) -> int:
    return load().convgb_im2col_bytes(N, C_in, H, W, KH, KW, stride, pad, dilation)


def im2win_bytes(N, C_in, H, W, KH, KW, stride=1, pad=0, dilation=1) -> int:
    return load().convgb_im2win_bytes(N, C_in, H, W, KH, KW, stride, pad, dilation)


def indirection_buffer_bytes(H, W, KH, KW, stride=1, pad=0, dilation=1) -> int:
    return load().convgb_indirection_buffer_bytes(H, W, KH, KW, stride, pad, dilation)


def conv2d_fwd_path(path, x, w, bias=None, stride=1, pad=0, dilation=1,
                    out_dtype=torch.bfloat16, y=None, workspace=None, stream=None):
    """Forward convolution on the requested path (PATH_* constant); returns y."""
    lib = load()
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(w, "w", torch.bfloat16)
    if bias is not None:
        _need_cuda(bias, "bias", torch.bfloat16)
    N, H, W, C_in = x.shape
    C_out, KH, KW, C_in2 = w.shape
    if C_in2 != C_in:
        raise ValueError("x has %d channels, w expects %d" % (C_in, C_in2))
    if bias is not None and tuple(bias.shape) != (C_out,):
        raise ValueError("bias must have shape [C_out]")
    H_out, W_out, need = _shape_info(lib, (path, N, C_in, H, W, C_out, KH, KW, stride, pad,
                                           dilation))
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out_dtype must be bfloat16 or float32")
    if y is None:
        y = torch.empty((N, H_out, W_out, C_out), dtype=out_dtype, device=x.device)
    else:
        _need_cuda(y, "y", out_dtype)
        if tuple(y.shape) != (N, H_out, W_out, C_out):
            raise ValueError("y has shape %s, expected %s" % (tuple(y.shape),
                                                              (N, H_out, W_out, C_out)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.conv2d_fwd_path(path, _ptr(x), _ptr(w), _ptr(bias), N, C_in, H, W, C_out, KH, KW,
                             stride, pad, dilation, _ptr(y),
                             _F32 if out_dtype == torch.float32 else _BF16, _ptr(workspace),
                             ws_bytes, _stream(stream))
    _check(st, "conv2d_fwd")
    return y


def conv2d_fwd(x, w, bias=None, stride=1, pad=0, dilation=1, out_dtype=torch.bfloat16, y=None,
               workspace=None, stream=None):
    """y = conv(x, w) + bias on the path the library picks; see include/convgb.h."""
    return conv2d_fwd_path(PATH_AUTO, x, w, bias, stride, pad, dilation, out_dtype, y,
                           workspace, stream)


def conv2d_fwd_host_scratch_size(N, C_in, H, W, C_out, KH, KW, stride=1, pad=0, dilation=1,
                                 out_dtype=torch.bfloat16, has_bias=True) -> int:
    return load().convgb_conv2d_fwd_host_scratch_size(
        N, C_in, H, W, C_out, KH, KW, stride, pad, dilation,
        _F32 if out_dtype == torch.float32 else _BF16, 1 if has_bias else 0)


def _need_host(t, name, dtype):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError("%s must be a host (CPU) tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous (channels-last layout)" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))


def conv2d_fwd_host(x, w, bias=None, stride=1, pad=0, dilation=1, out_dtype=torch.bfloat16,
                    y=None, scratch=None, stream=None, device=None):
    """conv2d_fwd with x, w, bias and y in host memory (pinned for overlapped copies):
    the library copies chunks of the batch in, convolves and copies out, all queued
    on `stream`; y is valid once that stream has finished.  See include/convgb.h."""
    lib = load()
    _need_host(x, "x", torch.bfloat16)
    _need_host(w, "w", torch.bfloat16)
    if bias is not None:
        _need_host(bias, "bias", torch.bfloat16)
    N, H, W, C_in = x.shape
    C_out, KH, KW, C_in2 = w.shape
    if C_in2 != C_in:
        raise ValueError("x has %d channels, w expects %d" % (C_in, C_in2))
    if bias is not None and tuple(bias.shape) != (C_out,):
        raise ValueError("bias must have shape [C_out]")
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out_dtype must be bfloat16 or float32")
    H_out, W_out = output_dims(H, W, KH, KW, stride, pad, dilation)
    if y is None:
        y = torch.empty((N, H_out, W_out, C_out), dtype=out_dtype, pin_memory=True)
    else:
        _need_host(y, "y", out_dtype)
        if tuple(y.shape) != (N, H_out, W_out, C_out):
            raise ValueError("y has shape %s, expected %s" % (tuple(y.shape),
                                                              (N, H_out, W_out, C_out)))
    need = conv2d_fwd_host_scratch_size(N, C_in, H, W, C_out, KH, KW, stride, pad, dilation,
                                        out_dtype, bias is not None)
    if scratch is None:
        scratch = torch.empty(need, dtype=torch.uint8, device=device or "cuda")
    elif not scratch.is_cuda:
        raise ValueError("scratch must be a CUDA tensor")
    st = lib.conv2d_fwd_host(_ptr(x), _ptr(w), _ptr(bias), N, C_in, H, W, C_out, KH, KW, stride,
                             pad, dilation, _ptr(y), _F32 if out_dtype == torch.float32 else _BF16,
                             _ptr(scratch), scratch.numel(), _stream(stream))
    _check(st, "conv2d_fwd_host")
    return y


def conv2d_fwd_indirect(x, w, bias, ibuf, stride=1, pad=0, dilation=1, out_dtype=torch.bfloat16,
                        y=None, stream=None):
    """Gather-path convolution reusing an indirection buffer from build_indirection_buffer()."""
    lib = load()
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(w, "w", torch.bfloat16)
    _need_cuda(ibuf, "ibuf", torch.int32)
    if bias is not None:
        _need_cuda(bias, "bias", torch.bfloat16)
    N, H, W, C_in = x.shape
    C_out, KH, KW, _ = w.shape
    H_out, W_out = output_dims(H, W, KH, KW, stride, pad, dilation)
    if y is None:
        y = torch.empty((N, H_out, W_out, C_out), dtype=out_dtype, device=x.device)
    else:
        _need_cuda(y, "y", out_dtype)
    st = lib.conv2d_fwd_indirect(_ptr(x), _ptr(w), _ptr(bias), N, C_in, H, W, C_out, KH, KW,
                                 stride, pad, dilation, _ptr(ibuf), ibuf.numel() * 4, _ptr(y),
                                 _F32 if out_dtype == torch.float32 else _BF16, _stream(stream))
    _check(st, "conv2d_fwd_indirect")
    return y


def im2win_transform(x, KH, KW, stride=1, pad=0, dilation=1, win=None, stream=None):
    """Window-order buffer [N, H_out, W_used, KH, C_in] (bf16) of x [N, H, W, C_in]."""
    lib = load()
    _need_cuda(x, "x", torch.bfloat16)
    N, H, W, C_in = x.shape
    H_out, W_out = output_dims(H, W, KH, KW, stride, pad, dilation)
    W_used = (W_out - 1) * stride + (KW - 1) * dilation + 1
    if win is None:
        win = torch.empty((N, H_out, W_used, KH, C_in), dtype=torch.bfloat16, device=x.device)
    else:
        _need_cuda(win, "win", torch.bfloat16)
    st = lib.im2win_transform(_ptr(x), N, C_in, H, W, KH, KW, stride, pad, dilation, _ptr(win),
                              win.numel() * 2, _stream(stream))
    _check(st, "im2win_transform")
    return win


def build_indirection_buffer(H, W, C_in, KH, KW, stride=1, pad=0, dilation=1, ibuf=None,
                             device=None, stream=None):
    """int32 [H_out*W_out, KH*KW] indirection buffer (element offsets, -1 = padding)."""
    lib = load()
    H_out, W_out = output_dims(H, W, KH, KW, stride, pad, dilation)
    if ibuf is None:
        ibuf = torch.empty((H_out * W_out, KH * KW), dtype=torch.int32,
                           device=device if device is not None else "cuda")
    else:
        _need_cuda(ibuf, "ibuf", torch.int32)
    st = lib.build_indirection_buffer(H, W, C_in, KH, KW, stride, pad, dilation, _ptr(ibuf),
                                      ibuf.numel() * 4, _stream(stream))
    _check(st, "build_indirection_buffer")
    return ibuf


def check_device_errors(stream=None):
    """Synchronise the stream; returns (status, raw device error code) and clears the word."""
    code = ctypes.c_uint()
    st = load().convgb_check_device_errors(_stream(stream), ctypes.byref(code))
    return st, code.value


def set_wait_timeout_ns(ns: int):
    load().convgb_set_wait_timeout_ns(int(ns))


def selftest_wait_timeout(timeout_ns: int, stream=None):
    _check(load().convgb_selftest_wait_timeout(int(timeout_ns), _stream(stream)),
           "selftest_wait_timeout")
