"""The unfused comparison path (conv output to memory, then a second kernel): conv+pool
bit-identical to the fused operator, conv-transpose within 1e-5 of the oracle."""
import numpy as np
import pytest
import torch

from tests.parity import FW, O, TOL_FFMA, assert_bits_equal, assert_close, dev, host, pmap, sample_indices, synth

pytestmark = pytest.mark.gpu


def cp_both(d, scale, pk):
    args = (dev(d["x"]), dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]), scale, pk)
    return host(FW.fw_conv2d_tanh_scale_bias_maxpool(*args)), host(FW.fw_conv2d_tanh_scale_bias_maxpool_unfused(*args))


@pytest.mark.parametrize("N,H,W,Cout,pk,scale", [(2, 64, 64, 64, 4, 2.0), (1, 41, 33, 16, 2, 2.0),
                                                 (1, 37, 70, 48, 4, -1.5), (2, 20, 132, 32, 2, 0.5),
                                                 (1, 131, 259, 64, 4, 2.0)])
def test_convpool_unfused_equals_fused(N, H, W, Cout, pk, scale):
    d = synth.convpool_inputs(N, 8, H, W, Cout, seed=H + W)
    fused, unfused = cp_both(d, scale, pk)
    assert_bits_equal(unfused, fused, str((N, H, W, Cout, pk)))
    want = O.conv2d_tanh_scale_bias_maxpool(d["x"], d["w"], d["conv_b"], scale, d["bias"], pk)
    assert_close(unfused, want, TOL_FFMA, "vs oracle")


def test_convpool_unfused_full_size():
    """x [128,8,256,256]: the 2.08 GB intermediate path gives the fused result bit for bit."""
    d = synth.convpool_inputs(128, 8, 256, 256, 64, seed=0)
    fused, unfused = cp_both(d, 2.0, 4)
    FW.fw_check_device_errors()
    assert unfused.shape == (128, 64, 63, 63)
    assert_bits_equal(unfused, fused, "full size")


def ct_unfused(d, scale):
    return host(FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_unfused(
        dev(d["x"]), dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]), scale))


@pytest.mark.parametrize("N,Cin,H,W", [(2, 64, 9, 10), (1, 64, 17, 33), (2, 8, 11, 3), (1, 32, 12, 12),
                                       (1, 16, 7, 9)])
def test_convt_unfused_matches_oracle(N, Cin, H, W):
    d = synth.convt_inputs(N, Cin, H, W, 128, seed=H + W)
    for scale in (2.0, -3.0):
        want = O.convtranspose2d_softmax_bias_scale_sigmoid(d["x"], d["w"], d["conv_b"], d["bias"], scale, 2, 1, 1)
        assert_close(ct_unfused(d, scale), want, TOL_FFMA, str((N, Cin, H, W, scale)))


def test_convt_unfused_full_size_sampled():
    """x [128,64,64,64] -> [128,128,129,129] through the 1.09 GB intermediate."""
    d = synth.convt_inputs(128, 64, 64, 64, 128, seed=0)
    got = ct_unfused(d, 2.0)
    FW.fw_check_device_errors()
    assert got.shape == (128, 128, 129, 129)
    pix = sample_indices((128, 129, 129), 600, seed=5)
    want = pmap(lambda t: O.convt_fused_pixel(d["x"], d["w"], d["conv_b"], d["bias"], 2.0, 2, 1, *t), pix)
    assert_close(np.stack([got[n, :, oh, ow] for n, oh, ow in pix]), np.stack(want), TOL_FFMA, "pixels")


def test_unsupported_shapes_raise():
    x = torch.zeros(1, 4, 16, 16, device="cuda")
    w = torch.zeros(8, 4, 3, 3, device="cuda")
    b = torch.zeros(8, device="cuda")
    with pytest.raises(FW.FusedWinError, match="FW_ERR_UNSUPPORTED"):
        FW.fw_conv2d_tanh_scale_bias_maxpool_unfused(x, w, None, b, 2.0, 4)
    xt = torch.zeros(1, 4, 4, 4, device="cuda")
    wt = torch.zeros(4, 8, 4, 4, device="cuda")
    with pytest.raises(FW.FusedWinError, match="FW_ERR_UNSUPPORTED"):
        FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_unfused(xt, wt, None, b, 2.0)
