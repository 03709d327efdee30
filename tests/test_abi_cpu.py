"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol the header declares, computes output shapes like the oracle, and rejects
bad arguments on the host with the documented status before any launch."""
import ctypes as C
import os
import re

import numpy as np
import pytest
import torch

from oracle import oracle as O
from pooling_sliding_window_gb300 import fusedwin as FW

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fusedwin.h")
P = C.c_void_p


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fw_[a-z0-9_]+)\s*\(", text)))


def test_header_and_exports():
    names = declared_functions()
    assert set(names) == set(FW.EXPORTS)
    L = FW.lib()
    for n in names:
        assert hasattr(L, n), n
    assert L.fw_version() >= 100
    for code, name in FW.STATUS.items():
        assert L.fw_status_string(code).decode().startswith(name)


def test_library_is_in_tree_and_sm103a_only():
    assert FW.library_path().startswith(os.path.join(ROOT, "pooling_sliding_window_gb300"))
    from pooling_sliding_window_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


@pytest.mark.parametrize("H,k,s,p,d", [(512, 4, 1, 1, 1), (13, 3, 2, 1, 2), (7, 5, 3, 2, 1), (1, 1, 1, 1, 1)])
def test_maxpool_shape_matches_oracle(H, k, s, p, d):
    assert FW.fw_maxpool2d_out_shape(H, H + 1, k, s, p, d) == (O.pool_out_size(H, k, s, p, d),
                                                              O.pool_out_size(H + 1, k, s, p, d))


@pytest.mark.parametrize("H,pk,ps", [(256, 4, 0), (127, 2, 2), (255, 4, 4), (64, 4, 0), (20, 3, 2)])
def test_convpool_shape_matches_oracle(H, pk, ps):
    hc = O.conv2d_out_size(H, 3)
    want = O.pool_out_size(hc, pk, ps or pk)
    assert FW.fw_conv2d_pool_out_shape(H, H, 3, 3, pk, ps) == (want, want)


@pytest.mark.parametrize("H,k,s,p,op", [(64, 4, 2, 1, 1), (5, 3, 2, 0, 1), (9, 5, 3, 2, 2), (4, 4, 2, 1, 0)])
def test_convt_shape_matches_oracle(H, k, s, p, op):
    want = O.convt_out_size(H, k, s, p, op)
    assert FW.fw_convt_out_shape(H, H, k, s, p, op) == (want, want)


@pytest.mark.parametrize("H,k,s,p,d", [(5, 2, 2, 0, 1), (4, 2, 3, 1, 1), (13, 3, 2, 1, 2), (6, 3, 2, 1, 1),
                                       (1, 2, 2, 0, 1), (512, 4, 1, 1, 1), (7, 4, 3, 2, 1)])
def test_maxpool_ceil_shape_matches_oracle(H, k, s, p, d):
    assert FW.fw_maxpool2d_out_shape_ex(H, H + 2, k, s, p, d, True) == (O.pool_out_size_ceil(H, k, s, p, d),
                                                                         O.pool_out_size_ceil(H + 2, k, s, p, d))
    if H + 2 * p - d * (k - 1) - 1 >= 0:  # floor mode has a window
        assert FW.fw_maxpool2d_out_shape_ex(H, H, k, s, p, d, False) == FW.fw_maxpool2d_out_shape(H, H, k, s, p, d)


def test_shape_errors():
    L = FW.lib()
    a, b = C.c_int(), C.c_int()
    assert L.fw_maxpool2d_out_shape(512, 512, 4, 1, 1, 1, None, None) == 1  # NULL out pointers
    assert L.fw_maxpool2d_out_shape(0, 5, 2, 1, 0, 1, C.byref(a), C.byref(b)) == 2
    assert L.fw_maxpool2d_out_shape(5, 5, 0, 1, 0, 1, C.byref(a), C.byref(b)) == 3
    assert L.fw_maxpool2d_out_shape(5, 5, 2, 0, 0, 1, C.byref(a), C.byref(b)) == 3
    assert L.fw_maxpool2d_out_shape(5, 5, 2, 1, -1, 1, C.byref(a), C.byref(b)) == 3
    assert L.fw_maxpool2d_out_shape(2, 2, 3, 1, 0, 1, C.byref(a), C.byref(b)) == 2  # window > input
    assert L.fw_conv2d_pool_out_shape(4, 4, 3, 3, 4, 4, C.byref(a), C.byref(b)) == 2
    assert L.fw_convt_out_shape(4, 4, 4, 2, 1, 2, C.byref(a), C.byref(b)) == 3  # op >= s


def test_operator_argument_errors_without_launch():
    """Every check runs on the host before a launch; none of these calls needs a GPU."""
    L = FW.lib()
    x, w, b, o = P(0x10000), P(0x20000), P(0x30000), P(0x40000000)
    # maxpool
    assert L.fw_maxpool2d(None, 1, 1, 8, 8, 2, 2, 0, 1, o, None) == 1
    assert L.fw_maxpool2d(x, 0, 1, 8, 8, 2, 2, 0, 1, o, None) == 2
    assert L.fw_maxpool2d(x, 1, 1, 8, 8, 2, 2, 0, 0, o, None) == 3
    assert L.fw_maxpool2d(P(0x10002), 1, 1, 8, 8, 2, 2, 0, 1, o, None) == 5
    assert L.fw_maxpool2d(x, 1, 1, 8, 8, 2, 2, 0, 1, P(0x10000 + 64), None) == 4  # out inside x
    # channels-last maxpool: (x, N, H, W, C, k, s, p, d, out, stream)
    assert L.fw_maxpool2d_nhwc(None, 1, 8, 8, 4, 2, 2, 0, 1, o, None) == 1
    assert L.fw_maxpool2d_nhwc(x, 1, 8, 8, 0, 2, 2, 0, 1, o, None) == 2
    assert L.fw_maxpool2d_nhwc(x, 1, 8, 8, 4, 2, 2, 0, 0, o, None) == 3
    assert L.fw_maxpool2d_nhwc(P(0x10002), 1, 8, 8, 4, 2, 2, 0, 1, o, None) == 5
    assert L.fw_maxpool2d_nhwc(x, 1, 8, 8, 4, 2, 2, 0, 1, P(0x10000 + 64), None) == 4  # out inside x
    # conv+pool
    args = lambda **kw: dict(dict(x=x, N=1, Cin=8, H=16, W=16, w=w, cb=None, Cout=4, KH=3, KW=3,
                                  scale=2.0, bias=b, pk=4, ps=0, out=o), **kw)
    for fname in ("fw_conv2d_tanh_scale_bias_maxpool", "fw_conv2d_tanh_scale_bias_maxpool_tf32",
                  "fw_conv2d_tanh_scale_bias_maxpool_ffma"):
        f = getattr(L, fname)
        call = lambda a: f(a["x"], a["N"], a["Cin"], a["H"], a["W"], a["w"], a["cb"], a["Cout"], a["KH"], a["KW"],
                           a["scale"], a["bias"], a["pk"], a["ps"], a["out"], None)
        assert call(args(bias=None)) == 1
        assert call(args(Cout=0)) == 2
        assert call(args(H=4)) == 2
        assert call(args(scale=float("inf"))) == 3
        assert call(args(scale=float("nan"))) == 3
        assert call(args(pk=0)) == 3
        assert call(args(out=P(0x20000 + 16))) == 4  # out overlaps w
        assert call(args(out=b)) == 4
        assert call(args(w=P(0x20001))) == 5
    # channels-last conv+pool: the same checks, x and out 16-byte aligned, tensor-core shapes only
    f = L.fw_conv2d_tanh_scale_bias_maxpool_nhwc
    call = lambda a: f(a["x"], a["N"], a["Cin"], a["H"], a["W"], a["w"], a["cb"], a["Cout"], a["KH"], a["KW"],
                       a["scale"], a["bias"], a["pk"], a["ps"], a["out"], None)
    assert call(args(bias=None)) == 1
    assert call(args(H=4)) == 2
    assert call(args(scale=float("nan"))) == 3
    assert call(args(Cout=16, x=P(0x10004))) == 5
    assert call(args(Cout=16, out=P(0x40000008))) == 5
    assert call(args(Cout=4)) == 6                 # no tensor-core kernel for Cout 4
    assert call(args(Cout=16, Cin=4)) == 6
    assert call(args(Cout=16, pk=3, ps=2)) == 6
    assert call(args(Cout=16, out=P(0x20000 + 16))) == 4
    # conv-transpose
    need = FW.fw_convt_workspace_size(64, 128, 4, 2, 1)
    assert need == 16 * 64 * 128 * 4
    ws = P(0x80000000)
    ct = lambda **kw: L.fw_convtranspose2d_softmax_bias_scale_sigmoid(
        kw.get("x", x), 1, 64, 8, 8, w, None, kw.get("Cout", 128), 4, 2, 1, kw.get("op", 1), b, 2.0,
        kw.get("out", o), kw.get("ws", ws), kw.get("wsb", need), None)
    assert ct(ws=None) == 1          # workspace required for the tiled path
    assert ct(wsb=need - 4) == 1     # too small
    assert ct(ws=P(0x80000004)) == 5  # workspace not 16-byte aligned
    assert ct(op=2) == 3
    assert ct(Cout=2048) == 6
    assert ct(out=P(0x80000000 + 4096)) == 4  # out overlaps workspace
    # the weight rewrite would overwrite bias / conv_b before the main kernel reads them
    ctb = lambda cb, bias: L.fw_convtranspose2d_softmax_bias_scale_sigmoid(
        x, 1, 64, 8, 8, w, cb, 128, 4, 2, 1, 1, bias, 2.0, o, ws, need, None)
    assert ctb(None, P(0x80000000 + 256)) == 4
    assert ctb(P(0x80000000 + need - 4), b) == 4
    # the FP32-FMA conv-transpose entry takes the same arguments and checks
    ff = lambda **kw: L.fw_convtranspose2d_softmax_bias_scale_sigmoid_ffma(
        kw.get("x", x), 1, 64, 8, 8, w, None, 128, 4, 2, 1, kw.get("op", 1), b, kw.get("scale", 2.0),
        kw.get("out", o), kw.get("ws", ws), need, None)
    assert ff(ws=None) == 1
    assert ff(op=2) == 3
    assert ff(scale=float("nan")) == 3
    assert ff(out=P(0x80000000 + 64)) == 4
    # unfused comparison path: workspace, alignment, support and aliasing checks
    cpn = FW.fw_conv2d_pool_unfused_workspace_size(2, 64, 64, 64, 3, 3, 4)
    assert cpn == 4 * 2 * 64 * 60 * 60
    big = P(0x100000000)
    cpu = lambda **kw: L.fw_conv2d_tanh_scale_bias_maxpool_unfused(
        x, 2, kw.get("Cin", 8), 64, 64, w, None, 64, 3, 3, 2.0, b, 4, 0, kw.get("out", o), kw.get("ws", big),
        kw.get("wsb", cpn), None)
    assert cpu(ws=None) == 1
    assert cpu(wsb=cpn - 1) == 1
    assert cpu(ws=P(0x100000008)) == 5
    assert cpu(Cin=4) == 6
    assert cpu(out=P(0x100000000 + 64)) == 4
    ctn = FW.fw_convt_unfused_workspace_size(1, 64, 8, 8, 128, 4, 2, 1, 1)
    assert ctn == ((16 * 64 * 128 * 4 + 255) // 256) * 256 + 4 * 128 * 17 * 17
    ctu = lambda **kw: L.fw_convtranspose2d_softmax_bias_scale_sigmoid_unfused(
        x, 1, kw.get("Cin", 64), 8, 8, w, None, 128, 4, kw.get("s", 2), 1, 1, b, 2.0, o, kw.get("ws", big),
        kw.get("wsb", ctn), None)
    assert ctu(ws=None) == 1
    assert ctu(wsb=ctn - 4) == 1
    assert ctu(Cin=12) == 6
    assert ctu(s=3) == 6
    assert FW.fw_convt_unfused_workspace_size(1, 64, 8, 8, 128, 4, 2, 1, 2) == 0  # op >= s
    # maxpool with ceil mode / indices
    assert L.fw_maxpool2d_ex(x, 1, 1, 8, 8, 2, 2, 0, 1, 1, o, P(0x50000004), None) == 5  # indices not 8-aligned
    assert L.fw_maxpool2d_ex(x, 1, 1, 8, 8, 2, 2, 0, 1, 1, o, P(0x40000000 + 8), None) == 4  # indices overlap out
    assert L.fw_maxpool2d_ex(x, 1, 1, 8, 8, 2, 2, 0, 1, 1, o, P(0x10000 + 8), None) == 4  # indices overlap x
    assert L.fw_maxpool2d_ex(x, 1, 1, 2, 2, 4, 2, 0, 1, 1, o, None, None) == 2  # output size < 1
    assert L.fw_maxpool2d_ex(None, 1, 1, 8, 8, 2, 2, 0, 1, 0, o, None, None) == 1
    # host-buffer calls: workspace checks before anything is enqueued
    hn = L.fw_maxpool2d_host_workspace_size(2, 3, 16, 16, 2, 2, 0, 1)
    assert hn == 2 * 3 * 16 * 16 * 4 + 2 * 3 * 8 * 8 * 4  # both parts already 256-byte multiples
    assert L.fw_maxpool2d_host(x, 2, 3, 16, 16, 2, 2, 0, 1, o, None, hn, None) == 1
    assert L.fw_maxpool2d_host(x, 2, 3, 16, 16, 2, 2, 0, 1, o, big, hn - 1, None) == 1
    assert L.fw_maxpool2d_host(x, 2, 3, 16, 16, 2, 2, 0, 1, o, P(0x100000010), hn, None) == 5
    assert L.fw_maxpool2d_host(x, 2, 3, 1, 1, 2, 2, 0, 1, o, big, hn, None) == 2
    assert L.fw_conv2d_tanh_scale_bias_maxpool_host_workspace_size(1, 8, 2, 2, 4, 3, 3, 4, 4) == 0
    assert L.fw_convtranspose2d_softmax_bias_scale_sigmoid_host_workspace_size(1, 4, 4, 4, 8, 4, 2, 1, 2) == 0
    # the bounded-wait self-test checks its limit before launching
    assert L.fw_selftest_bounded_wait(0, None) == 3
    assert L.fw_selftest_bounded_wait(2_000_001, None) == 3


def test_product_path_fails_loudly_without_gpu():
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    x = torch.zeros(1, 1, 8, 8)
    with pytest.raises(RuntimeError, match="CUDA"):
        FW.fw_maxpool2d(x, 2)


def test_binding_rejects_wrong_sizes_before_any_call():
    """The binding checks `out` and the per-channel vectors against the shapes the
    call implies (a kernel would otherwise write or read past their ends).  Host
    tensors exercise the checks without a GPU: they run before anything is moved."""
    x = torch.zeros(2, 8, 16, 16)
    w = torch.zeros(4, 8, 3, 3)
    b = torch.zeros(4)
    n0 = FW.fw_launch_count()
    with pytest.raises(ValueError, match="shape"):
        FW.fw_conv2d_tanh_scale_bias_maxpool(x, w, None, b, 2.0, 4, out=torch.zeros(2, 4, 3, 4))
    with pytest.raises(ValueError, match="one per output channel"):
        FW.fw_conv2d_tanh_scale_bias_maxpool(x, w, None, torch.zeros(3), 2.0, 4)
    with pytest.raises(ValueError, match="one per output channel"):
        FW.fw_conv2d_tanh_scale_bias_maxpool(x, w, torch.zeros(5), b, 2.0, 4)
    with pytest.raises(ValueError, match="input channels"):
        FW.fw_conv2d_tanh_scale_bias_maxpool(x, torch.zeros(4, 6, 3, 3), None, b, 2.0, 4)
    with pytest.raises(ValueError, match="shape"):
        FW.fw_maxpool2d(x, 2, 2, 0, 1, out=torch.zeros(2, 8, 8, 7))
    with pytest.raises(ValueError, match="shape"):
        FW.fw_maxpool2d_host(x, 2, 2, 0, 1, out=torch.zeros(2, 8, 8, 9))
    xt = torch.zeros(1, 64, 8, 8)
    wt = torch.zeros(64, 128, 4, 4)
    bt = torch.zeros(128)
    with pytest.raises(ValueError, match="shape"):
        FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(xt, wt, None, bt, 2.0, out=torch.zeros(1, 128, 16, 17))
    with pytest.raises(ValueError, match="shape"):
        FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_ffma(xt, wt, None, bt, 2.0, out=torch.zeros(1, 127, 17, 17))
    with pytest.raises(ValueError, match="one per output channel"):
        FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(xt, wt, torch.zeros(64), bt, 2.0)
    with pytest.raises(ValueError, match="square"):
        FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(xt, torch.zeros(64, 128, 4, 3), None, bt, 2.0)
    with pytest.raises(ValueError, match="input channels"):
        FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_host(xt, torch.zeros(32, 128, 4, 4), None, bt, 2.0)
    with pytest.raises(ValueError, match="shape"):
        FW.fw_conv2d_tanh_scale_bias_maxpool_host(x, w, None, b, 2.0, 4, out=torch.zeros(2, 4, 4, 4, 1))
    assert FW.fw_launch_count() == n0
