"""Python binding of libfusedwin (ctypes; argument marshalling only).

Each function has the name of the C entry point it calls and takes torch
tensors.  Device tensors are passed straight through (the call is enqueued on
torch's current CUDA stream and returns without synchronising).  Host tensors
are accepted too: they are copied to the device, the C entry point runs there,
and the result is copied back into a host tensor; this is the path an end-to-end
caller with host buffers takes.  Every operator runs in the library's CUDA
kernels; if the library cannot be loaded the call raises -- there is no other
implementation to fall back on.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import build as _build

_lib = None

STATUS = {0: "FW_OK", 1: "FW_ERR_NULL", 2: "FW_ERR_SHAPE", 3: "FW_ERR_PARAM", 4: "FW_ERR_ALIAS",
          5: "FW_ERR_ALIGN", 6: "FW_ERR_UNSUPPORTED", 7: "FW_ERR_LAUNCH", 8: "FW_ERR_TIMEOUT",
          9: "FW_ERR_INTERNAL"}

# Every symbol include/fusedwin.h declares.
EXPORTS = ("fw_status_string", "fw_version", "fw_conv2d_pool_out_shape", "fw_maxpool2d_out_shape",
           "fw_convt_out_shape", "fw_conv2d_tanh_scale_bias_maxpool", "fw_maxpool2d",
           "fw_convtranspose2d_softmax_bias_scale_sigmoid", "fw_convt_workspace_size",
           "fw_check_device_errors", "fw_launch_count", "fw_selftest_bounded_wait",
           "fw_convtranspose2d_softmax_bias_scale_sigmoid_noalloc",
           "fw_conv2d_tanh_scale_bias_maxpool_unfused", "fw_conv2d_pool_unfused_workspace_size",
           "fw_convtranspose2d_softmax_bias_scale_sigmoid_unfused", "fw_convt_unfused_workspace_size",
           "fw_maxpool2d_ex", "fw_maxpool2d_out_shape_ex",
           "fw_conv2d_tanh_scale_bias_maxpool_host", "fw_conv2d_tanh_scale_bias_maxpool_host_workspace_size",
           "fw_maxpool2d_host", "fw_maxpool2d_host_workspace_size",
           "fw_convtranspose2d_softmax_bias_scale_sigmoid_host",
           "fw_convtranspose2d_softmax_bias_scale_sigmoid_host_workspace_size",
           "fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc", "fw_conv2d_tanh_scale_bias_maxpool_tf32",
           "fw_conv2d_tanh_scale_bias_maxpool_ffma", "fw_convtranspose2d_softmax_bias_scale_sigmoid_ffma",
           "fw_maxpool2d_nhwc", "fw_conv2d_tanh_scale_bias_maxpool_nhwc")


class FusedWinError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = lib().fw_status_string(code).decode()
        super().__init__(f"{where}: {msg}")


def checked_build() -> bool:
    """FUSEDWIN_CHECKED=1: load the bounds-checked library (build.py, checked=True)."""
    return os.environ.get("FUSEDWIN_CHECKED") == "1"


def library_path() -> str:
    return _build.LIB_CHECKED if checked_build() else _build.LIB


def lib():
    """Load libfusedwin.so (building it first if the sources are newer)."""
    global _lib
    if _lib is None:
        if os.environ.get("FUSEDWIN_NO_BUILD") is None:
            path = _build.build(checked=checked_build())
        else:
            path = library_path()
        L = C.CDLL(path)
        I, P, F, U64 = C.c_int, C.c_void_p, C.c_float, C.c_ulonglong
        IP = C.POINTER(C.c_int)
        L.fw_status_string.restype = C.c_char_p
        L.fw_status_string.argtypes = [I]
        L.fw_version.restype = I
        L.fw_launch_count.restype = U64
        for name, n in (("fw_conv2d_pool_out_shape", 6), ("fw_maxpool2d_out_shape", 6),
                        ("fw_convt_out_shape", 6)):
            f = getattr(L, name)
            f.restype = I
            f.argtypes = [I] * n + [IP, IP]
        for name in ("fw_conv2d_tanh_scale_bias_maxpool", "fw_conv2d_tanh_scale_bias_maxpool_tf32",
                     "fw_conv2d_tanh_scale_bias_maxpool_ffma", "fw_conv2d_tanh_scale_bias_maxpool_nhwc"):
            getattr(L, name).restype = I
            getattr(L, name).argtypes = [P, I, I, I, I, P, P, I, I, I, F, P, I, I, P, P]
        L.fw_maxpool2d.restype = I
        L.fw_maxpool2d.argtypes = [P, I, I, I, I, I, I, I, I, P, P]
        L.fw_maxpool2d_nhwc.restype = I
        L.fw_maxpool2d_nhwc.argtypes = [P, I, I, I, I, I, I, I, I, P, P]
        for name in ("fw_convtranspose2d_softmax_bias_scale_sigmoid",
                     "fw_convtranspose2d_softmax_bias_scale_sigmoid_ffma"):
            getattr(L, name).restype = I
            getattr(L, name).argtypes = [P, I, I, I, I, P, P, I, I, I, I, I, P, F, P, P, U64, P]
        L.fw_convt_workspace_size.restype = U64
        L.fw_convt_workspace_size.argtypes = [I, I, I, I, I]
        L.fw_check_device_errors.restype = I
        L.fw_check_device_errors.argtypes = [P]
        L.fw_selftest_bounded_wait.restype = I
        L.fw_selftest_bounded_wait.argtypes = [C.c_uint, P]
        L.fw_convtranspose2d_softmax_bias_scale_sigmoid_noalloc.restype = I
        L.fw_convtranspose2d_softmax_bias_scale_sigmoid_noalloc.argtypes = [
            P, I, I, I, I, P, P, I, I, I, I, I, P, F, P, P]
        L.fw_conv2d_tanh_scale_bias_maxpool_unfused.restype = I
        L.fw_conv2d_tanh_scale_bias_maxpool_unfused.argtypes = [
            P, I, I, I, I, P, P, I, I, I, F, P, I, I, P, P, U64, P]
        L.fw_conv2d_pool_unfused_workspace_size.restype = U64
        L.fw_conv2d_pool_unfused_workspace_size.argtypes = [I] * 8
        L.fw_convtranspose2d_softmax_bias_scale_sigmoid_unfused.restype = I
        L.fw_convtranspose2d_softmax_bias_scale_sigmoid_unfused.argtypes = [
            P, I, I, I, I, P, P, I, I, I, I, I, P, F, P, P, U64, P]
        L.fw_convt_unfused_workspace_size.restype = U64
        L.fw_convt_unfused_workspace_size.argtypes = [I] * 9
        L.fw_maxpool2d_ex.restype = I
        L.fw_maxpool2d_ex.argtypes = [P, I, I, I, I, I, I, I, I, I, P, P, P]
        L.fw_maxpool2d_out_shape_ex.restype = I
        L.fw_maxpool2d_out_shape_ex.argtypes = [I] * 7 + [IP, IP]
        L.fw_conv2d_tanh_scale_bias_maxpool_host.restype = I
        L.fw_conv2d_tanh_scale_bias_maxpool_host.argtypes = [P, I, I, I, I, P, P, I, I, I, F, P, I, I, P, P, U64, P]
        L.fw_conv2d_tanh_scale_bias_maxpool_host_workspace_size.restype = U64
        L.fw_conv2d_tanh_scale_bias_maxpool_host_workspace_size.argtypes = [I] * 9
        L.fw_maxpool2d_host.restype = I
        L.fw_maxpool2d_host.argtypes = [P, I, I, I, I, I, I, I, I, P, P, U64, P]
        L.fw_maxpool2d_host_workspace_size.restype = U64
        L.fw_maxpool2d_host_workspace_size.argtypes = [I] * 8
        L.fw_convtranspose2d_softmax_bias_scale_sigmoid_host.restype = I
        L.fw_convtranspose2d_softmax_bias_scale_sigmoid_host.argtypes = [
            P, I, I, I, I, P, P, I, I, I, I, I, P, F, P, P, U64, P]
        L.fw_convtranspose2d_softmax_bias_scale_sigmoid_host_workspace_size.restype = U64
        L.fw_convtranspose2d_softmax_bias_scale_sigmoid_host_workspace_size.argtypes = [I] * 9
        L.fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc.restype = I
        L.fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc.argtypes = [
            P, I, I, I, I, P, P, I, I, I, I, I, P, F, P, P, U64, P]
        _lib = L
    return _lib


def _check(code: int, where: str):
    if code != 0:
        raise FusedWinError(code, where)


def _shape2(fn, *args):
    ho, wo = C.c_int(0), C.c_int(0)
    _check(getattr(lib(), fn)(*args, C.byref(ho), C.byref(wo)), fn)
    return ho.value, wo.value


def fw_conv2d_pool_out_shape(H, W, KH, KW, pool_k, pool_s=0):
    return _shape2("fw_conv2d_pool_out_shape", H, W, KH, KW, pool_k, pool_s)


def fw_maxpool2d_out_shape(H, W, k, s, p, d):
    return _shape2("fw_maxpool2d_out_shape", H, W, k, s, p, d)


def fw_convt_out_shape(H, W, k, s, p, op):
    return _shape2("fw_convt_out_shape", H, W, k, s, p, op)


def fw_convt_workspace_size(Cin, Cout, k, s, p) -> int:
    return int(lib().fw_convt_workspace_size(Cin, Cout, k, s, p))


def fw_launch_count() -> int:
    return int(lib().fw_launch_count())


def fw_selftest_bounded_wait(limit_us, stream=None):
    """Launch the bounded-wait self-test kernel (see include/fusedwin.h)."""
    s = torch.cuda.current_stream() if stream is None else stream
    _check(lib().fw_selftest_bounded_wait(int(limit_us), C.c_void_p(s.cuda_stream)), "fw_selftest_bounded_wait")


def fw_check_device_errors(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    _check(lib().fw_check_device_errors(C.c_void_p(s.cuda_stream)), "fw_check_device_errors")


# ----------------------------------------------------------------- helpers --

def _dev(t, name, device):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32:
        raise TypeError(f"{name} must be a float32 torch.Tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (dense NCHW)")
    if t.device.type != "cuda":
        t = t.to(device, non_blocking=True)
    return t


def _ptr(t):
    return C.c_void_p(0 if t is None else t.data_ptr())


# Shape checks made before any C call: a kernel trusts the sizes it is given, so an
# `out` or a bias smaller than the arguments imply would be written or read past its
# end on the GPU.

def _check_out(out, shape, device_type=None, name="out"):
    """`out` (if given) must be a contiguous float32 tensor of exactly `shape`."""
    if out is None:
        return
    if not isinstance(out, torch.Tensor) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 tensor")
    if tuple(out.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(out.shape)}, the call needs {tuple(shape)}")
    if device_type is not None and out.device.type != device_type:
        raise ValueError(f"{name} must be a {device_type} tensor")


def _check_dims(name, t, ndim):
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")


def _check_vec(name, t, n):
    if t is not None and t.numel() != n:
        raise ValueError(f"{name} must hold {n} values (one per output channel), got {t.numel()}")


def _conv_pool_dims(x, w, conv_b, bias, channels_last=False):
    """(N, Cin, H, W, Cout, KH, KW) of a conv+pool call, checked for consistency."""
    _check_dims("x", x, 4)
    _check_dims("w", w, 4)
    if channels_last:
        N, H, W, Cin = x.shape
    else:
        N, Cin, H, W = x.shape
    Cout, Cw, KH, KW = w.shape
    if Cw != Cin:
        raise ValueError(f"w has {Cw} input channels, x has {Cin}")
    _check_vec("conv_b", conv_b, Cout)
    _check_vec("bias", bias, Cout)
    return N, Cin, H, W, Cout, KH, KW


def _convt_dims(x, w, conv_b, bias, channels_last=False):
    """(N, Cin, H, W, Cout, K) of a conv-transpose call, checked for consistency."""
    _check_dims("x", x, 4)
    _check_dims("w", w, 4)
    if channels_last:
        N, H, W, Cin = x.shape
    else:
        N, Cin, H, W = x.shape
    Cw, Cout, K, K2 = w.shape
    if Cw != Cin:
        raise ValueError(f"w has {Cw} input channels, x has {Cin}")
    if K != K2:
        raise ValueError(f"w must have a square kernel, got {K}x{K2}")
    _check_vec("conv_b", conv_b, Cout)
    _check_vec("bias", bias, Cout)
    return N, Cin, H, W, Cout, K


def _device_of(x):
    if x.device.type == "cuda":
        return x.device
    if not torch.cuda.is_available():
        raise RuntimeError("libfusedwin needs a CUDA device; none is available")
    return torch.device("cuda", torch.cuda.current_device())


def _finish(out_dev, out, host):
    if not host:
        return out_dev
    if out is None:
        out = torch.empty(out_dev.shape, dtype=torch.float32, pin_memory=True)
    out.copy_(out_dev, non_blocking=True)
    torch.cuda.current_stream(out_dev.device).synchronize()
    return out


# --------------------------------------------------------------- operators --

def fw_conv2d_tanh_scale_bias_maxpool(x, w, conv_b, bias, scale, pool_k, pool_s=0, out=None):
    """out = MaxPool2d(pool_k, pool_s)(bias + scale * tanh(conv2d(x, w, conv_b)))."""
    return _conv_pool("fw_conv2d_tanh_scale_bias_maxpool", x, w, conv_b, bias, scale, pool_k, pool_s, out)


def fw_conv2d_tanh_scale_bias_maxpool_tf32(x, w, conv_b, bias, scale, pool_k, pool_s=0, out=None):
    """The same operator with the convolution's products taken once in TF32 on the tensor-core shapes."""
    return _conv_pool("fw_conv2d_tanh_scale_bias_maxpool_tf32", x, w, conv_b, bias, scale, pool_k, pool_s, out)


def fw_conv2d_tanh_scale_bias_maxpool_ffma(x, w, conv_b, bias, scale, pool_k, pool_s=0, out=None):
    """The same operator on the float32 FMA pipe only (no tensor cores)."""
    return _conv_pool("fw_conv2d_tanh_scale_bias_maxpool_ffma", x, w, conv_b, bias, scale, pool_k, pool_s, out)


def _conv_pool(fname, x, w, conv_b, bias, scale, pool_k, pool_s, out):
    host = x.device.type != "cuda"
    N, Cin, H, W, Cout, KH, KW = _conv_pool_dims(x, w, conv_b, bias.reshape(-1))
    Ho, Wo = fw_conv2d_pool_out_shape(H, W, KH, KW, pool_k, pool_s)
    _check_out(out, (N, Cout, Ho, Wo), "cpu" if host else "cuda")
    dev = _device_of(x)
    xd, wd = _dev(x, "x", dev), _dev(w, "w", dev)
    cbd, bd = _dev(conv_b, "conv_b", dev), _dev(bias.reshape(-1), "bias", dev)
    od = out if (out is not None and not host) else torch.empty((N, Cout, Ho, Wo), device=dev,
                                                                 dtype=torch.float32)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        _check(getattr(lib(), fname)(
            _ptr(xd), N, Cin, H, W, _ptr(wd), _ptr(cbd), Cout, KH, KW, float(scale), _ptr(bd),
            pool_k, pool_s, _ptr(od), C.c_void_p(stream)), fname)
    return _finish(od, out, host)


def fw_maxpool2d(x, k, s=None, p=0, d=1, out=None):
    """MaxPool2d(kernel k, stride s (default k), padding p (-inf), dilation d)."""
    s = k if s is None else s
    host = x.device.type != "cuda"
    _check_dims("x", x, 4)
    N, Cc, H, W = x.shape
    Ho, Wo = fw_maxpool2d_out_shape(H, W, k, s, p, d)
    _check_out(out, (N, Cc, Ho, Wo), "cpu" if host else "cuda")
    dev = _device_of(x)
    xd = _dev(x, "x", dev)
    od = out if (out is not None and not host) else torch.empty((N, Cc, Ho, Wo), device=dev,
                                                                 dtype=torch.float32)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        _check(lib().fw_maxpool2d(_ptr(xd), N, Cc, H, W, k, s, p, d, _ptr(od), C.c_void_p(stream)),
               "fw_maxpool2d")
    return _finish(od, out, host)


def fw_maxpool2d_nhwc(x, k, s=None, p=0, d=1, out=None):
    """Channels-last MaxPool2d: x [N, H, W, C] -> out [N, Ho, Wo, C]."""
    s = k if s is None else s
    host = x.device.type != "cuda"
    _check_dims("x", x, 4)
    N, H, W, Cc = x.shape
    Ho, Wo = fw_maxpool2d_out_shape(H, W, k, s, p, d)
    _check_out(out, (N, Ho, Wo, Cc), "cpu" if host else "cuda")
    dev = _device_of(x)
    xd = _dev(x, "x", dev)
    od = out if (out is not None and not host) else torch.empty((N, Ho, Wo, Cc), device=dev,
                                                                 dtype=torch.float32)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        _check(lib().fw_maxpool2d_nhwc(_ptr(xd), N, H, W, Cc, k, s, p, d, _ptr(od), C.c_void_p(stream)),
               "fw_maxpool2d_nhwc")
    return _finish(od, out, host)


def fw_convtranspose2d_softmax_bias_scale_sigmoid(x, w, conv_b, bias, scale, stride=2, padding=1,
                                                  output_padding=1, out=None, workspace=None):
    """out = sigmoid((softmax(conv_transpose2d(x, w, conv_b), dim=1) + bias) * scale)."""
    return _convt("fw_convtranspose2d_softmax_bias_scale_sigmoid", x, w, conv_b, bias, scale, stride, padding,
                  output_padding, out, workspace)


def fw_convtranspose2d_softmax_bias_scale_sigmoid_ffma(x, w, conv_b, bias, scale, stride=2, padding=1,
                                                       output_padding=1, out=None, workspace=None):
    """The same operator on the float32 FMA pipe only (float32 products and sums)."""
    return _convt("fw_convtranspose2d_softmax_bias_scale_sigmoid_ffma", x, w, conv_b, bias, scale, stride, padding,
                  output_padding, out, workspace)


def _convt(fname, x, w, conv_b, bias, scale, stride, padding, output_padding, out, workspace):
    host = x.device.type != "cuda"
    N, Cin, H, W, Cout, K = _convt_dims(x, w, conv_b, bias.reshape(-1))
    Ho, Wo = fw_convt_out_shape(H, W, K, stride, padding, output_padding)
    _check_out(out, (N, Cout, Ho, Wo), "cpu" if host else "cuda")
    dev = _device_of(x)
    xd, wd = _dev(x, "x", dev), _dev(w, "w", dev)
    cbd, bd = _dev(conv_b, "conv_b", dev), _dev(bias.reshape(-1), "bias", dev)
    need = fw_convt_workspace_size(Cin, Cout, K, stride, padding)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty((need + 3) // 4, device=dev, dtype=torch.float32)
    od = out if (out is not None and not host) else torch.empty((N, Cout, Ho, Wo), device=dev,
                                                                 dtype=torch.float32)
    stream = torch.cuda.current_stream(dev).cuda_stream
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        _check(getattr(lib(), fname)(
            _ptr(xd), N, Cin, H, W, _ptr(wd), _ptr(cbd), Cout, K, stride, padding, output_padding,
            _ptr(bd), float(scale), _ptr(od), _ptr(workspace), ws_bytes, C.c_void_p(stream)), fname)
    return _finish(od, out, host)


def fw_convtranspose2d_softmax_bias_scale_sigmoid_noalloc(x, w, conv_b, bias, scale, out, stride=2, padding=1,
                                                          output_padding=1):
    """The conv-transpose model through the allocation-free entry point.

    For callers that cannot allocate device memory: every tensor, `out`
    included, must already be on the device (nothing is copied or allocated
    here), and the library uses its own fixed device array for the weight
    rewrite instead of a workspace.  Calls that overlap on the GPU race on that
    array.
    """
    for name, t in (("x", x), ("w", w), ("bias", bias), ("out", out)) + ((("conv_b", conv_b),) if conv_b is not None else ()):
        if not isinstance(t, torch.Tensor) or t.device.type != "cuda" or t.dtype != torch.float32 \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    N, Cin, H, W, Cout, K = _convt_dims(x, w, conv_b, bias.reshape(-1))
    _check_out(out, (N, Cout) + fw_convt_out_shape(H, W, K, stride, padding, output_padding), "cuda")
    stream = torch.cuda.current_stream(x.device).cuda_stream
    with torch.cuda.device(x.device):
        _check(lib().fw_convtranspose2d_softmax_bias_scale_sigmoid_noalloc(
            _ptr(x), N, Cin, H, W, _ptr(w), _ptr(conv_b), Cout, K, stride, padding, output_padding,
            _ptr(bias), float(scale), _ptr(out), C.c_void_p(stream)),
            "fw_convtranspose2d_softmax_bias_scale_sigmoid_noalloc")
    return out


# ------------------------------------------------------ unfused comparison --

def fw_conv2d_pool_unfused_workspace_size(N, H, W, Cout, KH, KW, pool_k, pool_s=0) -> int:
    return int(lib().fw_conv2d_pool_unfused_workspace_size(N, H, W, Cout, KH, KW, pool_k, pool_s))


def fw_convt_unfused_workspace_size(N, Cin, H, W, Cout, k, s, p, op) -> int:
    return int(lib().fw_convt_unfused_workspace_size(N, Cin, H, W, Cout, k, s, p, op))


def _workspace(need, workspace, dev):
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty((need + 15) // 16 * 4, device=dev, dtype=torch.float32)
    return workspace, workspace.numel() * workspace.element_size()


def fw_conv2d_tanh_scale_bias_maxpool_unfused(x, w, conv_b, bias, scale, pool_k, pool_s=0, out=None,
                                              workspace=None):
    """The conv+pool model the unfused way (conv output to memory, then pool + tanh
    + scale + bias); bit-identical to fw_conv2d_tanh_scale_bias_maxpool."""
    dev = _device_of(x)
    xd, wd = _dev(x, "x", dev), _dev(w, "w", dev)
    cbd, bd = _dev(conv_b, "conv_b", dev), _dev(bias.reshape(-1), "bias", dev)
    N, Cin, H, W, Cout, KH, KW = _conv_pool_dims(xd, wd, cbd, bd)
    Ho, Wo = fw_conv2d_pool_out_shape(H, W, KH, KW, pool_k, pool_s)
    _check_out(out, (N, Cout, Ho, Wo), "cuda")
    workspace, ws_bytes = _workspace(fw_conv2d_pool_unfused_workspace_size(N, H, W, Cout, KH, KW, pool_k, pool_s),
                                     workspace, dev)
    od = out if out is not None else torch.empty((N, Cout, Ho, Wo), device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        _check(lib().fw_conv2d_tanh_scale_bias_maxpool_unfused(
            _ptr(xd), N, Cin, H, W, _ptr(wd), _ptr(cbd), Cout, KH, KW, float(scale), _ptr(bd),
            pool_k, pool_s, _ptr(od), _ptr(workspace), ws_bytes, C.c_void_p(stream)),
            "fw_conv2d_tanh_scale_bias_maxpool_unfused")
    return od


def fw_convtranspose2d_softmax_bias_scale_sigmoid_unfused(x, w, conv_b, bias, scale, stride=2, padding=1,
                                                          output_padding=1, out=None, workspace=None):
    """The conv-transpose model the unfused way (conv-transpose output to memory,
    then an online-softmax pass and an output pass per pixel)."""
    dev = _device_of(x)
    xd, wd = _dev(x, "x", dev), _dev(w, "w", dev)
    cbd, bd = _dev(conv_b, "conv_b", dev), _dev(bias.reshape(-1), "bias", dev)
    N, Cin, H, W, Cout, K = _convt_dims(xd, wd, cbd, bd)
    Ho, Wo = fw_convt_out_shape(H, W, K, stride, padding, output_padding)
    _check_out(out, (N, Cout, Ho, Wo), "cuda")
    workspace, ws_bytes = _workspace(
        fw_convt_unfused_workspace_size(N, Cin, H, W, Cout, K, stride, padding, output_padding), workspace, dev)
    od = out if out is not None else torch.empty((N, Cout, Ho, Wo), device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        _check(lib().fw_convtranspose2d_softmax_bias_scale_sigmoid_unfused(
            _ptr(xd), N, Cin, H, W, _ptr(wd), _ptr(cbd), Cout, K, stride, padding, output_padding,
            _ptr(bd), float(scale), _ptr(od), _ptr(workspace), ws_bytes, C.c_void_p(stream)),
            "fw_convtranspose2d_softmax_bias_scale_sigmoid_unfused")
    return od


# ------------------------------------------------- maxpool extensions --

def fw_maxpool2d_out_shape_ex(H, W, k, s, p, d, ceil_mode=False):
    return _shape2("fw_maxpool2d_out_shape_ex", H, W, k, s, p, d, int(bool(ceil_mode)))


def fw_maxpool2d_ex(x, k, s=None, p=0, d=1, ceil_mode=False, return_indices=False, out=None):
    """MaxPool2d with ceil mode and argmax indices (PyTorch's options; not on the
    pages).  Returns out, or (out, indices int64) with return_indices."""
    s = k if s is None else s
    dev = _device_of(x)
    xd = _dev(x, "x", dev)
    _check_dims("x", xd, 4)
    N, Cc, H, W = xd.shape
    Ho, Wo = fw_maxpool2d_out_shape_ex(H, W, k, s, p, d, ceil_mode)
    _check_out(out, (N, Cc, Ho, Wo), "cuda")
    od = out if out is not None else torch.empty((N, Cc, Ho, Wo), device=dev, dtype=torch.float32)
    idx = torch.empty((N, Cc, Ho, Wo), device=dev, dtype=torch.int64) if return_indices else None
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        _check(lib().fw_maxpool2d_ex(_ptr(xd), N, Cc, H, W, k, s, p, d, int(bool(ceil_mode)), _ptr(od), _ptr(idx),
                                     C.c_void_p(stream)), "fw_maxpool2d_ex")
    return (od, idx) if return_indices else od


# ------------------------------------------------------ host-buffer calls --
# Host (CPU) tensors in and out, pinned for the copies to overlap; the C call
# pipelines chunked copies and kernels.  `workspace` is a device tensor (made here
# when None) of at least the *_host_workspace_size bytes.

def _host(t, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.device.type != "cpu":
        raise TypeError(f"{name} must be a float32 CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (dense NCHW)")
    return t


def _dev_workspace(need, workspace):
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        if not torch.cuda.is_available():
            raise RuntimeError("libfusedwin needs a CUDA device; none is available")
        workspace = torch.empty((need + 15) // 16 * 4, device="cuda", dtype=torch.float32)
    return workspace, workspace.numel() * workspace.element_size()


def fw_conv2d_tanh_scale_bias_maxpool_host(x, w, conv_b, bias, scale, pool_k, pool_s=0, out=None, workspace=None,
                                           stream=None):
    x, w, conv_b, bias = _host(x, "x"), _host(w, "w"), _host(conv_b, "conv_b"), _host(bias.reshape(-1), "bias")
    N, Cin, H, W, Cout, KH, KW = _conv_pool_dims(x, w, conv_b, bias)
    Ho, Wo = fw_conv2d_pool_out_shape(H, W, KH, KW, pool_k, pool_s)
    _check_out(out, (N, Cout, Ho, Wo), "cpu")
    out = torch.empty((N, Cout, Ho, Wo), pin_memory=True) if out is None else _host(out, "out")
    workspace, wsb = _dev_workspace(int(lib().fw_conv2d_tanh_scale_bias_maxpool_host_workspace_size(
        N, Cin, H, W, Cout, KH, KW, pool_k, pool_s)), workspace)
    s = torch.cuda.current_stream(workspace.device) if stream is None else stream
    with torch.cuda.device(workspace.device):
        _check(lib().fw_conv2d_tanh_scale_bias_maxpool_host(
            _ptr(x), N, Cin, H, W, _ptr(w), _ptr(conv_b), Cout, KH, KW, float(scale), _ptr(bias), pool_k, pool_s,
            _ptr(out), _ptr(workspace), wsb, C.c_void_p(s.cuda_stream)), "fw_conv2d_tanh_scale_bias_maxpool_host")
    s.synchronize()
    return out


def fw_maxpool2d_host(x, k, s=None, p=0, d=1, out=None, workspace=None, stream=None):
    s = k if s is None else s
    x = _host(x, "x")
    _check_dims("x", x, 4)
    N, Cc, H, W = x.shape
    Ho, Wo = fw_maxpool2d_out_shape(H, W, k, s, p, d)
    _check_out(out, (N, Cc, Ho, Wo), "cpu")
    out = torch.empty((N, Cc, Ho, Wo), pin_memory=True) if out is None else _host(out, "out")
    workspace, wsb = _dev_workspace(int(lib().fw_maxpool2d_host_workspace_size(N, Cc, H, W, k, s, p, d)), workspace)
    st = torch.cuda.current_stream(workspace.device) if stream is None else stream
    with torch.cuda.device(workspace.device):
        _check(lib().fw_maxpool2d_host(_ptr(x), N, Cc, H, W, k, s, p, d, _ptr(out), _ptr(workspace), wsb,
                                       C.c_void_p(st.cuda_stream)), "fw_maxpool2d_host")
    st.synchronize()
    return out


def fw_convtranspose2d_softmax_bias_scale_sigmoid_host(x, w, conv_b, bias, scale, stride=2, padding=1,
                                                       output_padding=1, out=None, workspace=None, stream=None):
    x, w, conv_b, bias = _host(x, "x"), _host(w, "w"), _host(conv_b, "conv_b"), _host(bias.reshape(-1), "bias")
    N, Cin, H, W, Cout, K = _convt_dims(x, w, conv_b, bias)
    Ho, Wo = fw_convt_out_shape(H, W, K, stride, padding, output_padding)
    _check_out(out, (N, Cout, Ho, Wo), "cpu")
    out = torch.empty((N, Cout, Ho, Wo), pin_memory=True) if out is None else _host(out, "out")
    workspace, wsb = _dev_workspace(int(lib().fw_convtranspose2d_softmax_bias_scale_sigmoid_host_workspace_size(
        N, Cin, H, W, Cout, K, stride, padding, output_padding)), workspace)
    st = torch.cuda.current_stream(workspace.device) if stream is None else stream
    with torch.cuda.device(workspace.device):
        _check(lib().fw_convtranspose2d_softmax_bias_scale_sigmoid_host(
            _ptr(x), N, Cin, H, W, _ptr(w), _ptr(conv_b), Cout, K, stride, padding, output_padding, _ptr(bias),
            float(scale), _ptr(out), _ptr(workspace), wsb, C.c_void_p(st.cuda_stream)),
            "fw_convtranspose2d_softmax_bias_scale_sigmoid_host")
    st.synchronize()
    return out


# -------------------------------------------------------- channels last --

def fw_conv2d_tanh_scale_bias_maxpool_nhwc(x, w, conv_b, bias, scale, pool_k, pool_s=0, out=None):
    """The conv+pool model on channels-last tensors: x [N, H, W, Cin] -> out
    [N, Ho, Wo, Cout] (device tensors; w keeps the [Cout, Cin, KH, KW] layout)."""
    dev = _device_of(x)
    xd, wd = _dev(x, "x", dev), _dev(w, "w", dev)
    cbd, bd = _dev(conv_b, "conv_b", dev), _dev(bias.reshape(-1), "bias", dev)
    N, Cin, H, W, Cout, KH, KW = _conv_pool_dims(xd, wd, cbd, bd, channels_last=True)
    Ho, Wo = fw_conv2d_pool_out_shape(H, W, KH, KW, pool_k, pool_s)
    _check_out(out, (N, Ho, Wo, Cout), "cuda")
    od = out if out is not None else torch.empty((N, Ho, Wo, Cout), device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        _check(lib().fw_conv2d_tanh_scale_bias_maxpool_nhwc(
            _ptr(xd), N, Cin, H, W, _ptr(wd), _ptr(cbd), Cout, KH, KW, float(scale), _ptr(bd),
            pool_k, pool_s, _ptr(od), C.c_void_p(stream)), "fw_conv2d_tanh_scale_bias_maxpool_nhwc")
    return od


def fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc(x, w, conv_b, bias, scale, stride=2, padding=1,
                                                       output_padding=1, out=None, workspace=None):
    """The conv-transpose model on channels-last tensors: x [N, H, W, Cin] ->
    out [N, Ho, Wo, Cout] (device tensors; w keeps the [Cin, Cout, k, k] layout)."""
    dev = _device_of(x)
    xd, wd = _dev(x, "x", dev), _dev(w, "w", dev)
    cbd, bd = _dev(conv_b, "conv_b", dev), _dev(bias.reshape(-1), "bias", dev)
    N, Cin, H, W, Cout, K = _convt_dims(xd, wd, cbd, bd, channels_last=True)
    Ho, Wo = fw_convt_out_shape(H, W, K, stride, padding, output_padding)
    _check_out(out, (N, Ho, Wo, Cout), "cuda")
    need = fw_convt_workspace_size(Cin, Cout, K, stride, padding)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(1, (need + 3) // 4), device=dev, dtype=torch.float32)
    od = out if out is not None else torch.empty((N, Ho, Wo, Cout), device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        _check(lib().fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc(
            _ptr(xd), N, Cin, H, W, _ptr(wd), _ptr(cbd), Cout, K, stride, padding, output_padding, _ptr(bd),
            float(scale), _ptr(od), _ptr(workspace), workspace.numel() * workspace.element_size(),
            C.c_void_p(stream)), "fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc")
    return od
