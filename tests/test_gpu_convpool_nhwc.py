"""Channels-last conv3x3+tanh+scale+bias+maxpool: x [N,H,W,8] -> out [N,Ho,Wo,Cout], against
the oracle through a layout wrapper (the oracle runs on the NCHW tensor; its result is
transposed) within 1e-5, and bit for bit against the NCHW call's result transposed."""
import numpy as np
import pytest
import torch

from tests.parity import FW, O, TOL_FFMA, assert_bits_equal, assert_close, dev, guarded_call, host, pmap, \
    sample_indices, synth

pytestmark = pytest.mark.gpu


def nhwc(a):
    return np.ascontiguousarray(np.transpose(a, (0, 2, 3, 1)))


def oracle_nhwc(d, scale, pk):
    return nhwc(O.conv2d_tanh_scale_bias_maxpool(d["x"], d["w"], d["conv_b"], scale, d["bias"], pk, pk))


def run_nhwc(d, scale, pk):
    N, Cout = d["x"].shape[0], d["w"].shape[0]
    Ho, Wo = FW.fw_conv2d_pool_out_shape(d["x"].shape[2], d["x"].shape[3], 3, 3, pk, 0)
    return guarded_call(FW.fw_conv2d_tanh_scale_bias_maxpool_nhwc, (N, Ho, Wo, Cout), dev(nhwc(d["x"])),
                        dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]), scale, pk)


def run_nchw(d, scale, pk):
    return host(FW.fw_conv2d_tanh_scale_bias_maxpool(dev(d["x"]), dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]),
                                                     scale, pk))


# (N, H, W, Cout, pool_k, scale): every tensor-core Cout and pool size, ragged rows and
# column blocks, one-item launches, and the min (scale < 0) and scale = 0 paths.
CASES = [
    (2, 64, 64, 64, 4, 2.0),
    (1, 37, 70, 64, 4, 2.0),      # ragged: 2 column blocks, last one partial
    (2, 41, 33, 16, 2, 2.0),
    (1, 36, 68, 32, 4, -1.5),     # negative scale: window min
    (2, 20, 132, 48, 2, 2.0),     # 2 column blocks of 64 pooled pixels, the second partial
    (1, 30, 260, 48, 4, 0.0),     # zero scale: out == bias
    (1, 6, 6, 16, 4, 2.0),        # a single window, one item
    (3, 11, 11, 32, 2, 0.5),      # odd sizes: input columns past the last used one
    (1, 9, 131, 64, 2, 2.0),      # 64 pooled pixels + 1: a tail of one
]


@pytest.mark.parametrize("case", CASES)
def test_nhwc_matches_oracle_and_nchw(case):
    N, H, W, Cout, pk, scale = case
    d = synth.convpool_inputs(N, 8, H, W, Cout, seed=N + H + W + Cout)
    got = run_nhwc(d, scale, pk)
    assert_close(got, oracle_nhwc(d, scale, pk), TOL_FFMA, str(case))
    assert_bits_equal(got, nhwc(run_nchw(d, scale, pk)), "same arithmetic as the NCHW kernel")


def test_nhwc_without_conv_bias():
    """conv_b omitted (NULL): the same as a zero conv bias, against the oracle and the NCHW call."""
    d = synth.convpool_inputs(2, 8, 30, 70, 48, seed=5)
    d = dict(d, conv_b=np.zeros_like(d["conv_b"]))
    got = host(FW.fw_conv2d_tanh_scale_bias_maxpool_nhwc(dev(nhwc(d["x"])), dev(d["w"]), None, dev(d["bias"]),
                                                         -2.0, 2))
    assert_close(got, oracle_nhwc(d, -2.0, 2), TOL_FFMA, "no conv_b")
    ref = host(FW.fw_conv2d_tanh_scale_bias_maxpool(dev(d["x"]), dev(d["w"]), None, dev(d["bias"]), -2.0, 2))
    assert_bits_equal(got, nhwc(ref), "same arithmetic as the NCHW kernel")


def test_random_shapes_bit_identical_to_nchw():
    """Random tensor-core shapes: the channels-last call and the NCHW call run the same
    products in the same order, so the results agree bit for bit."""
    rng = np.random.default_rng(23)
    for _ in range(30):
        N, Cout, pk = int(rng.integers(1, 4)), int(rng.choice([16, 32, 48, 64])), int(rng.choice([2, 4]))
        H, W = int(rng.integers(pk + 2, 60)), int(rng.integers(pk + 2, 300))
        scale = float(rng.choice([2.0, -3.0, 0.5]))
        d = synth.convpool_inputs(N, 8, H, W, Cout, seed=int(rng.integers(0, 1 << 30)))
        cl = FW.fw_conv2d_tanh_scale_bias_maxpool_nhwc(dev(nhwc(d["x"])), dev(d["w"]), dev(d["conv_b"]),
                                                       dev(d["bias"]), scale, pk)
        ref = FW.fw_conv2d_tanh_scale_bias_maxpool(dev(d["x"]), dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]),
                                                   scale, pk)
        FW.fw_check_device_errors()
        assert torch.equal(ref.permute(0, 2, 3, 1), cl), (N, H, W, Cout, pk, scale)


def test_nhwc_full_size_sampled_and_equal_to_nchw():
    """x [128,256,256,8] (the benchmarked conv+pool as NHWC) -> [128,63,63,64]: sampled
    outputs against the oracle, and every output against the NCHW call transposed."""
    d = synth.convpool_inputs(128, 8, 256, 256, 64, seed=0)
    x = dev(nhwc(d["x"]))
    args = (dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]), 2.0, 4)
    got = FW.fw_conv2d_tanh_scale_bias_maxpool_nhwc(x, *args)
    FW.fw_check_device_errors()
    assert got.shape == (128, 63, 63, 64)
    ref = FW.fw_conv2d_tanh_scale_bias_maxpool(dev(d["x"]), *args)
    assert torch.equal(ref.permute(0, 2, 3, 1), got)
    got = host(got)
    idx = sample_indices((128, 64, 63, 63), 1500, seed=3)
    want = pmap(lambda t: O.convpool_at(d["x"], d["w"], d["conv_b"], 2.0, d["bias"], 4, 4, *t), idx)
    assert_close(np.array([got[n, i, j, co] for n, co, i, j in idx]), np.array(want), TOL_FFMA, "samples")


def test_nhwc_errors():
    x = torch.zeros(1, 16, 16, 8, device="cuda")
    w = torch.zeros(16, 8, 3, 3, device="cuda")
    b = torch.zeros(16, device="cuda")
    flat = torch.zeros(16 * 16 * 8 + 4, device="cuda")
    with pytest.raises(FW.FusedWinError, match="FW_ERR_ALIGN"):  # x 4-byte but not 16-byte aligned
        FW.fw_conv2d_tanh_scale_bias_maxpool_nhwc(flat[1:1 + 16 * 16 * 8].view(1, 16, 16, 8), w, None, b, 2.0, 4)
    out = torch.zeros(1 * 3 * 3 * 16 + 4, device="cuda")
    with pytest.raises(FW.FusedWinError, match="FW_ERR_ALIGN"):
        FW.fw_conv2d_tanh_scale_bias_maxpool_nhwc(x, w, None, b, 2.0, 4, out=out[2:2 + 144].view(1, 3, 3, 16))
    with pytest.raises(FW.FusedWinError, match="FW_ERR_UNSUPPORTED"):  # Cin 4: no tensor-core kernel
        FW.fw_conv2d_tanh_scale_bias_maxpool_nhwc(torch.zeros(1, 16, 16, 4, device="cuda"),
                                                  torch.zeros(16, 4, 3, 3, device="cuda"), None, b, 2.0, 4)
    with pytest.raises(FW.FusedWinError, match="FW_ERR_UNSUPPORTED"):  # overlapping pool windows
        FW.fw_conv2d_tanh_scale_bias_maxpool_nhwc(x, w, None, b, 2.0, 3, 2)
    with pytest.raises(FW.FusedWinError, match="FW_ERR_PARAM"):
        FW.fw_conv2d_tanh_scale_bias_maxpool_nhwc(x, w, None, b, float("nan"), 4)
