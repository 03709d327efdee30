"""Fused conv3x3+tanh+scale+bias+maxpool, plain-TF32 variant: CUDA path vs the oracle
(max abs err <= 5e-3), and vs the oracle evaluated on TF32-rounded x and w (<= 1e-5),
which pins what the variant computes: products of TF32 operands, float32 sums."""
import numpy as np
import pytest
import torch

from tests.parity import (FW, O, TOL_FFMA, TOL_TF32, assert_close, dev, host, pmap, sample_indices, synth,
                          tf32_round)

pytestmark = pytest.mark.gpu


def run_gpu(d, scale, pk, cb=True):
    return host(FW.fw_conv2d_tanh_scale_bias_maxpool_tf32(dev(d["x"]), dev(d["w"]),
                                                          dev(d["conv_b"]) if cb else None, dev(d["bias"]),
                                                          scale, pk))


def run_oracle(d, scale, pk, cb=True, rounded=False):
    x, w = (tf32_round(d["x"]), tf32_round(d["w"])) if rounded else (d["x"], d["w"])
    return O.conv2d_tanh_scale_bias_maxpool(x, w, d["conv_b"] if cb else None, scale, d["bias"], pk, pk)


def test_tiny_config_full():
    """x [2,8,64,64], Conv 8->64 k3, tanh, *2, +bias, MaxPool2d(4) -> [2,64,15,15]."""
    d = synth.convpool_inputs(2, 8, 64, 64, 64, seed=0)
    got = run_gpu(d, 2.0, 4)
    assert got.shape == (2, 64, 15, 15)
    assert_close(got, run_oracle(d, 2.0, 4), TOL_TF32, "tiny")
    assert_close(got, run_oracle(d, 2.0, 4, rounded=True), TOL_FFMA, "tiny, TF32-rounded operands")


# (N, H, W, Cout, pk, scale): tensor-core shapes (several column blocks, ragged tails) and
# shapes that take the float32 FMA kernels.
CASES = [
    (1, 37, 70, 64, 4, 2.0),
    (2, 41, 33, 16, 2, 2.0),
    (1, 36, 68, 32, 4, 2.0),
    (2, 20, 132, 48, 2, 2.0),
    (1, 30, 260, 48, 4, -1.5),   # negative scale: window minimum
    (1, 26, 26, 64, 4, 0.0),     # zero scale: out == bias
    (1, 6, 6, 16, 4, 2.0),       # a single window
    (1, 22, 19, 20, 4, 2.0),     # Cout 20: not a tensor-core shape
]


@pytest.mark.parametrize("case", CASES)
def test_small_shapes(case):
    N, H, W, Cout, pk, scale = case
    d = synth.convpool_inputs(N, 8, H, W, Cout, seed=N + H + W)
    got = run_gpu(d, scale, pk)
    assert_close(got, run_oracle(d, scale, pk), TOL_TF32, str(case))
    tc = Cout in (16, 32, 48, 64)
    assert_close(got, run_oracle(d, scale, pk, rounded=tc), TOL_FFMA, str(case) + " exact-operand model")


def test_no_conv_bias():
    d = synth.convpool_inputs(1, 8, 40, 40, 16, seed=10)
    assert_close(run_gpu(d, 2.0, 4, cb=False), run_oracle(d, 2.0, 4, cb=False, rounded=True), TOL_FFMA, "no-cb")


@pytest.mark.parametrize("N,H,Cout,pk", [(n, h, c, p) for n in (1, 16) for h in (127, 255, 256)
                                         for c in (16, 64) for p in (2, 4)])
def test_sweep(N, H, Cout, pk):
    """batch {1,16} x H=W {127,255,256} x Cout {16,64} x pool {2,4}: first and last image."""
    d = synth.convpool_inputs(N, 8, H, H, Cout, seed=H + Cout)
    got = run_gpu(d, 2.0, pk)
    for n in sorted({0, N - 1}):
        sub = dict(d, x=d["x"][n:n + 1])
        assert_close(got[n:n + 1], run_oracle(sub, 2.0, pk), TOL_TF32, f"image {n}")
        assert_close(got[n:n + 1], run_oracle(sub, 2.0, pk, rounded=True), TOL_FFMA, f"image {n} model")


def test_full_size_sampled():
    """x [128,8,256,256], Conv 8->64 k3, MaxPool2d(4) -> [128,64,63,63]: the benchmarked launch."""
    d = synth.convpool_inputs(128, 8, 256, 256, 64, seed=0)
    got = run_gpu(d, 2.0, 4)
    FW.fw_check_device_errors()
    assert got.shape == (128, 64, 63, 63)
    idx = sample_indices(got.shape, 2000, seed=3)
    g = np.array([got[t] for t in idx])
    want = pmap(lambda t: O.convpool_at(d["x"], d["w"], d["conv_b"], 2.0, d["bias"], 4, 4, *t), idx)
    assert_close(g, np.array(want), TOL_TF32, "samples")
    xr, wr = tf32_round(d["x"]), tf32_round(d["w"])
    want_r = pmap(lambda t: O.convpool_at(xr, wr, d["conv_b"], 2.0, d["bias"], 4, 4, *t), idx)
    assert_close(g, np.array(want_r), TOL_FFMA, "samples, exact-operand model")
    sub = dict(d, x=d["x"][127:128])
    assert_close(got[127:128], run_oracle(sub, 2.0, 4), TOL_TF32, "last image")
    b = d["bias"][None, :, None, None]
    assert np.all(got >= b - 2) and np.all(got <= b + 2)


def test_unaligned_rows_and_errors():
    d = synth.convpool_inputs(2, 8, 40, 64, 64, seed=11)
    flat = torch.zeros(d["x"].size + 1, dtype=torch.float32, device="cuda")
    x = flat[1:].view(d["x"].shape)
    x.copy_(torch.from_numpy(d["x"]))
    assert x.data_ptr() % 16 == 4
    got = host(FW.fw_conv2d_tanh_scale_bias_maxpool_tf32(x, dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]), 2.0, 4))
    assert_close(got, run_oracle(d, 2.0, 4, rounded=True), TOL_FFMA, "unaligned rows")
    with pytest.raises(FW.FusedWinError, match="FW_ERR_PARAM"):
        FW.fw_conv2d_tanh_scale_bias_maxpool_tf32(x, dev(d["w"]), None, dev(d["bias"]), float("nan"), 4)
