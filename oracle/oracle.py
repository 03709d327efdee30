"""Python front end of the oracle (``fusedwin_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The CUDA product path never
imports this module.

The C library is built with gcc on first use (``build()``), with
``-ffp-contract=off`` so that no multiply-add is fused and the float64 sums are
the same on x86-64 and aarch64.  Every wrapper takes and returns numpy arrays;
float32 in, float32 (fused operators) or float64 (linear stages) out.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fusedwin_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_LIB_OMP = os.path.join(_HERE, "_build", "liboracle_omp.so")
_lock = threading.Lock()
_lib = None
_lib_omp = None

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_L = C.c_long


def build(force: bool = False, openmp: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (if stale).

    ``openmp=True`` builds the same source with ``-fopenmp`` into
    ``liboracle_omp.so``: its pragmas spread independent images, channels and planes
    over the host cores (used only to time the definition at full size); nothing
    else differs, and the results are bit-identical to the single-threaded build.
    """
    out = _LIB_OMP if openmp else _LIB
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                        *(["-fopenmp"] if openmp else []), "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, out)
    return out


def _ptr_or_null(a):
    return None if a is None else a.ctypes.data_as(C.POINTER(C.c_float))


def load(path: str):
    """Load a compiled oracle library and declare its signatures."""
    L = C.CDLL(path)
    fp = C.POINTER(C.c_float)
    for name in ("oracle_conv2d_out_size", "oracle_pool_out_size"):
        getattr(L, name).restype = _L
    L.oracle_conv2d_out_size.argtypes = [_L] * 4
    L.oracle_pool_out_size.argtypes = [_L] * 5
    L.oracle_convt_out_size.restype = _L
    L.oracle_convt_out_size.argtypes = [_L] * 5
    L.oracle_conv2d.restype = C.c_int
    L.oracle_conv2d.argtypes = [_f32p, _L, _L, _L, _L, _f32p, fp, _L, _L, _L, _L, _L, _f64p]
    L.oracle_conv2d_one.restype = C.c_double
    L.oracle_conv2d_one.argtypes = [_f32p, _L, _L, _L, _f32p, fp, _L, _L, _L, _L, _L, _L, _L, _L]
    L.oracle_maxpool2d.restype = C.c_int
    L.oracle_maxpool2d.argtypes = [_f32p, _L, _L, _L, _L, _L, _L, _L, _L, _f32p]
    L.oracle_maxpool2d_one.restype = C.c_float
    L.oracle_maxpool2d_one.argtypes = [fp, _L, _L, _L, _L, _L, _L, _L, _L]
    L.oracle_pool_out_size_ceil.restype = _L
    L.oracle_pool_out_size_ceil.argtypes = [_L] * 5
    L.oracle_maxpool2d_one_idx.restype = C.c_float
    L.oracle_maxpool2d_one_idx.argtypes = [fp, _L, _L, _L, _L, _L, _L, _L, _L, C.POINTER(_L)]
    L.oracle_maxpool2d_ex.restype = C.c_int
    L.oracle_maxpool2d_ex.argtypes = [_f32p, _L, _L, _L, _L, _L, _L, _L, _L, C.c_int, _f32p, C.c_void_p]
    L.oracle_conv2d_tanh_scale_bias_maxpool.restype = C.c_int
    L.oracle_conv2d_tanh_scale_bias_maxpool.argtypes = [
        _f32p, _L, _L, _L, _L, _f32p, fp, _L, _L, _L, C.c_float, _f32p, _L, _L, _f32p]
    L.oracle_convpool_one.restype = C.c_float
    L.oracle_convpool_one.argtypes = [
        _f32p, _L, _L, _L, _f32p, fp, _L, _L, C.c_float, _f32p, _L, _L, _L, _L, _L, _L]
    L.oracle_convt2d.restype = C.c_int
    L.oracle_convt2d.argtypes = [_f32p, _L, _L, _L, _L, _f32p, fp, _L, _L, _L, _L, _L, _f64p]
    L.oracle_convt2d_one.restype = C.c_double
    L.oracle_convt2d_one.argtypes = [_f32p, _L, _L, _L, _f32p, fp, _L, _L, _L, _L, _L, _L, _L, _L]
    L.oracle_softmax_bias_scale_sigmoid_pixel.restype = None
    L.oracle_softmax_bias_scale_sigmoid_pixel.argtypes = [_f32p, _L, _f32p, C.c_float, _f64p, _f32p]
    L.oracle_convt_fused_pixel.restype = C.c_int
    L.oracle_convt_fused_pixel.argtypes = [
        _f32p, _L, _L, _L, _f32p, fp, _L, _L, _L, _L, _f32p, C.c_float, _L, _L, _L, _f32p]
    L.oracle_convtranspose2d_softmax_bias_scale_sigmoid.restype = C.c_int
    L.oracle_convtranspose2d_softmax_bias_scale_sigmoid.argtypes = [
        _f32p, _L, _L, _L, _L, _f32p, fp, _L, _L, _L, _L, _L, _f32p, C.c_float, _f32p]
    L.oracle_softmax_channels.restype = None
    L.oracle_softmax_channels.argtypes = [_f32p, _L, _f64p, _f32p]
    return L


def lib(openmp: bool = False):
    """The loaded oracle library (``openmp=True``: the multi-threaded build; its
    thread count is fixed by OMP_NUM_THREADS when it is first loaded)."""
    global _lib, _lib_omp
    with _lock:
        if openmp:
            if _lib_omp is None:
                _lib_omp = load(build(openmp=True))
            return _lib_omp
        if _lib is None:
            _lib = load(build())
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _check(rc):
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")


# ----------------------------------------------------------------- sizes --

def conv2d_out_size(H, k, s=1, p=0):
    return int(lib().oracle_conv2d_out_size(H, k, s, p))


def pool_out_size(H, k, s, p=0, d=1):
    return int(lib().oracle_pool_out_size(H, k, s, p, d))


def convt_out_size(H, k, s, p, op):
    return int(lib().oracle_convt_out_size(H, k, s, p, op))


# ---------------------------------------------------------- linear stages --

def conv2d(x, w, cb=None, stride=1, pad=0):
    """Conv2d in float64: x [N,Cin,H,W], w [Cout,Cin,KH,KW] -> [N,Cout,Ho,Wo]."""
    x, w = _f32(x), _f32(w)
    cb = None if cb is None else _f32(cb)
    N, Cin, H, W = x.shape
    Cout, _, KH, KW = w.shape
    Ho, Wo = conv2d_out_size(H, KH, stride, pad), conv2d_out_size(W, KW, stride, pad)
    y = np.empty((N, Cout, max(Ho, 0), max(Wo, 0)), dtype=np.float64)
    _check(lib().oracle_conv2d(x, N, Cin, H, W, w, _ptr_or_null(cb), Cout, KH, KW, stride, pad, y))
    return y


def convt2d(x, w, cb=None, stride=2, pad=1, output_padding=1):
    """ConvTranspose2d in float64 (scatter form): w [Cin,Cout,K,K]."""
    x, w = _f32(x), _f32(w)
    cb = None if cb is None else _f32(cb)
    N, Cin, H, W = x.shape
    _, Cout, K, _ = w.shape
    Ho = convt_out_size(H, K, stride, pad, output_padding)
    Wo = convt_out_size(W, K, stride, pad, output_padding)
    y = np.empty((N, Cout, Ho, Wo), dtype=np.float64)
    _check(lib().oracle_convt2d(x, N, Cin, H, W, w, _ptr_or_null(cb), Cout, K, stride, pad,
                                output_padding, y))
    return y


def convt2d_one(x, w, cb, stride, pad, n, co, oh, ow):
    """One ConvTranspose2d output (gather form), float64."""
    x, w = _f32(x), _f32(w)
    cb = None if cb is None else _f32(cb)
    N, Cin, H, W = x.shape
    _, Cout, K, _ = w.shape
    return float(lib().oracle_convt2d_one(x, Cin, H, W, w, _ptr_or_null(cb), Cout, K, stride, pad,
                                          n, co, oh, ow))


# -------------------------------------------------------------- operators --

def maxpool2d(x, k, s=None, p=0, d=1, openmp=False):
    """MaxPool2d (floor mode, -inf padding): float32 out."""
    x = _f32(x)
    s = k if s is None else s
    N, Cc, H, W = x.shape
    Ho, Wo = pool_out_size(H, k, s, p, d), pool_out_size(W, k, s, p, d)
    out = np.empty((N, Cc, max(Ho, 0), max(Wo, 0)), dtype=np.float32)
    _check(lib(openmp).oracle_maxpool2d(x, N, Cc, H, W, k, s, p, d, out))
    return out


def pool_out_size_ceil(H, k, s, p=0, d=1):
    """MaxPool2d output size in ceil mode (extension beyond the pages)."""
    return int(lib().oracle_pool_out_size_ceil(H, k, s, p, d))


def maxpool2d_ex(x, k, s=None, p=0, d=1, ceil_mode=False):
    """MaxPool2d with ceil mode and argmax indices (extension): (out float32,
    idx int64 = flat ih*W + iw of the chosen tap, -1 for a window with no input tap)."""
    x = _f32(x)
    s = k if s is None else s
    N, Cc, H, W = x.shape
    size = pool_out_size_ceil if ceil_mode else pool_out_size
    Ho, Wo = size(H, k, s, p, d), size(W, k, s, p, d)
    out = np.empty((N, Cc, max(Ho, 0), max(Wo, 0)), dtype=np.float32)
    idx = np.empty(out.shape, dtype=np.int64)
    _check(lib().oracle_maxpool2d_ex(x, N, Cc, H, W, k, s, p, d, int(bool(ceil_mode)), out,
                                     idx.ctypes.data_as(C.c_void_p)))
    return out, idx


def maxpool2d_at(x, k, s, p, d, n, c, oh, ow):
    """One MaxPool2d output of x[n, c] by the definition."""
    N, Cc, H, W = x.shape
    plane = _f32(x[n, c])
    return np.float32(lib().oracle_maxpool2d_one(plane.ctypes.data_as(C.POINTER(C.c_float)),
                                                 H, W, k, s, p, d, oh, ow))


def conv2d_tanh_scale_bias_maxpool(x, w, cb, scale, bias, pool_k, pool_s=None, openmp=False):
    """The conv -> tanh -> *scale -> +bias -> MaxPool2d model, stage by stage."""
    x, w, bias = _f32(x), _f32(w), _f32(bias).reshape(-1)
    cb = None if cb is None else _f32(cb)
    pool_s = pool_k if not pool_s else pool_s
    N, Cin, H, W = x.shape
    Cout, _, KH, KW = w.shape
    Ho = pool_out_size(conv2d_out_size(H, KH), pool_k, pool_s)
    Wo = pool_out_size(conv2d_out_size(W, KW), pool_k, pool_s)
    out = np.empty((N, Cout, max(Ho, 0), max(Wo, 0)), dtype=np.float32)
    _check(lib(openmp).oracle_conv2d_tanh_scale_bias_maxpool(x, N, Cin, H, W, w, _ptr_or_null(cb), Cout,
                                                       KH, KW, scale, bias, pool_k, pool_s, out))
    return out


def convpool_at(x, w, cb, scale, bias, pool_k, pool_s, n, co, i, j):
    """One output of the conv+pool model, computed from its own window."""
    x, w, bias = _f32(x), _f32(w), _f32(bias).reshape(-1)
    cb = None if cb is None else _f32(cb)
    pool_s = pool_k if not pool_s else pool_s
    N, Cin, H, W = x.shape
    Cout, _, KH, KW = w.shape
    return np.float32(lib().oracle_convpool_one(x, Cin, H, W, w, _ptr_or_null(cb), KH, KW, scale,
                                                bias, pool_k, pool_s, n, co, i, j))


def softmax_channels(y):
    """Softmax of one pixel's channel vector y (float32 in, float32 out)."""
    y = _f32(y)
    p = np.empty_like(y)
    e = np.empty(y.shape[0], dtype=np.float64)
    lib().oracle_softmax_channels(y, y.shape[0], e, p)
    return p


def softmax_bias_scale_sigmoid_pixel(y, bias, scale):
    """The post-convT chain for one pixel's channel vector y (float32)."""
    y, bias = _f32(y), _f32(bias).reshape(-1)
    out = np.empty_like(y)
    e = np.empty(y.shape[0], dtype=np.float64)
    lib().oracle_softmax_bias_scale_sigmoid_pixel(y, y.shape[0], bias, scale, e, out)
    return out


def convtranspose2d_softmax_bias_scale_sigmoid(x, w, cb, bias, scale, stride=2, pad=1,
                                               output_padding=1, openmp=False):
    """The convT -> softmax(dim 1) -> +bias -> *scale -> sigmoid model."""
    x, w, bias = _f32(x), _f32(w), _f32(bias).reshape(-1)
    cb = None if cb is None else _f32(cb)
    N, Cin, H, W = x.shape
    _, Cout, K, _ = w.shape
    Ho = convt_out_size(H, K, stride, pad, output_padding)
    Wo = convt_out_size(W, K, stride, pad, output_padding)
    out = np.empty((N, Cout, Ho, Wo), dtype=np.float32)
    _check(lib(openmp).oracle_convtranspose2d_softmax_bias_scale_sigmoid(
        x, N, Cin, H, W, w, _ptr_or_null(cb), Cout, K, stride, pad, output_padding, bias, scale, out))
    return out


def convt_fused_pixel(x, w, cb, bias, scale, stride, pad, n, oh, ow):
    """All channels of the convT model at one pixel (gather form)."""
    x, w, bias = _f32(x), _f32(w), _f32(bias).reshape(-1)
    cb = None if cb is None else _f32(cb)
    N, Cin, H, W = x.shape
    _, Cout, K, _ = w.shape
    out = np.empty(Cout, dtype=np.float32)
    _check(lib().oracle_convt_fused_pixel(x, Cin, H, W, w, _ptr_or_null(cb), Cout, K, stride, pad,
                                          bias, scale, n, oh, ow, out))
    return out


def convtranspose2d_softmax_bias_scale_sigmoid_nhwc(x_nhwc, w, cb, bias, scale, stride=2, pad=1, output_padding=1):
    """Channels-last layout of the same model: x [N, H, W, Cin] -> out [N, Ho, Wo, Cout].
    A layout change only -- the definition is the NCHW function above, with the
    activations transposed in and out."""
    x = np.ascontiguousarray(np.transpose(np.asarray(x_nhwc, dtype=np.float32), (0, 3, 1, 2)))
    out = convtranspose2d_softmax_bias_scale_sigmoid(x, w, cb, bias, scale, stride, pad, output_padding)
    return np.ascontiguousarray(np.transpose(out, (0, 2, 3, 1)))
