"""Channels-last conv-transpose model: x [N,H,W,Cin] -> out [N,Ho,Wo,128], against the
oracle (1e-5) and bit-for-bit against the NCHW kernel's result transposed."""
import numpy as np
import pytest
import torch

from tests.parity import FW, O, TOL_FFMA, assert_bits_equal, assert_close, dev, host, pmap, sample_indices, synth

pytestmark = pytest.mark.gpu


def nhwc(a):
    return np.ascontiguousarray(np.transpose(a, (0, 2, 3, 1)))


@pytest.mark.parametrize("N,Cin,H,W", [(2, 64, 9, 10), (1, 64, 17, 33), (2, 8, 11, 3), (1, 32, 12, 12),
                                       (1, 16, 7, 9), (1, 64, 40, 70)])
def test_nhwc_matches_oracle_and_nchw(N, Cin, H, W):
    d = synth.convt_inputs(N, Cin, H, W, 128, seed=H * W)
    for scale in (2.0, -3.0):
        got = host(FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc(
            dev(nhwc(d["x"])), dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]), scale))
        want = O.convtranspose2d_softmax_bias_scale_sigmoid_nhwc(nhwc(d["x"]), d["w"], d["conv_b"], d["bias"], scale)
        assert got.shape == want.shape
        assert_close(got, want, TOL_FFMA, str((N, Cin, H, W, scale)))
        nchw = host(FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(dev(d["x"]), dev(d["w"]), dev(d["conv_b"]),
                                                                     dev(d["bias"]), scale))
        assert_bits_equal(got, nhwc(nchw), "same arithmetic as the NCHW kernel")


def test_nhwc_full_size_sampled():
    d = synth.convt_inputs(128, 64, 64, 64, 128, seed=0)
    got = host(FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc(
        dev(nhwc(d["x"])), dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]), 2.0))
    FW.fw_check_device_errors()
    assert got.shape == (128, 129, 129, 128)
    pix = sample_indices((128, 129, 129), 600, seed=9)
    want = pmap(lambda t: O.convt_fused_pixel(d["x"], d["w"], d["conv_b"], d["bias"], 2.0, 2, 1, *t), pix)
    assert_close(np.stack([got[n, oh, ow, :] for n, oh, ow in pix]), np.stack(want), TOL_FFMA, "pixels")


def test_nhwc_alignment_and_support_errors():
    x = torch.zeros(1, 8, 8, 64, device="cuda")
    w = torch.zeros(64, 128, 4, 4, device="cuda")
    b = torch.zeros(128, device="cuda")
    flat = torch.zeros(1 * 17 * 17 * 128 + 4, device="cuda")
    with pytest.raises(FW.FusedWinError, match="FW_ERR_ALIGN"):
        FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc(x, w, None, b, 2.0, out=flat[4:].view(1, 17, 17, 128))
    with pytest.raises(FW.FusedWinError, match="FW_ERR_UNSUPPORTED"):
        FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc(torch.zeros(1, 8, 8, 4, device="cuda"),
                                                              torch.zeros(4, 8, 4, 4, device="cuda"), None,
                                                              torch.zeros(8, device="cuda"), 2.0)


def test_nchw_tiles_match_channels_last_on_random_shapes():
    """The NCHW call (CTA pairs, both column phases per tile) and the channels-last call
    (one phase per CTA) run the same products in the same order: bit-identical results on
    random shapes, including tiles whose second half lies past the last pixel."""
    rng = np.random.default_rng(11)
    for _ in range(40):
        N, Cin = int(rng.integers(1, 5)), int(rng.choice([8, 16, 32, 64]))
        H, W = int(rng.integers(1, 40)), int(rng.integers(1, 130))
        scale = float(rng.choice([2.0, -3.0, 0.5]))
        d = synth.convt_inputs(N, Cin, H, W, 128, seed=int(rng.integers(0, 1 << 30)))
        nchw = FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(dev(d["x"]), dev(d["w"]), dev(d["conv_b"]),
                                                               dev(d["bias"]), scale)
        cl = FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc(dev(nhwc(d["x"])), dev(d["w"]), dev(d["conv_b"]),
                                                                  dev(d["bias"]), scale)
        FW.fw_check_device_errors()
        assert torch.equal(nchw.permute(0, 2, 3, 1), cl), (N, Cin, H, W, scale)


def test_full_size_repeat_calls_identical():
    """Full config D called repeatedly: the same bits every time (no race between the pair's CTAs)."""
    d = synth.convt_inputs(128, 64, 64, 64, 128, seed=0)
    args = (dev(d["x"]), dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]), 2.0)
    ref = FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(*args)
    for _ in range(5):
        assert torch.equal(FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(*args), ref)
    FW.fw_check_device_errors()
