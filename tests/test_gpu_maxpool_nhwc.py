"""Channels-last MaxPool2d: x [N,H,W,C] -> out [N,Ho,Wo,C], bit for bit against the oracle
through a layout wrapper (the oracle pools the NCHW tensor; its result is transposed), and
against the NCHW kernels at the full size."""
import numpy as np
import pytest
import torch

from tests.parity import FW, O, assert_bits_equal, dev, guarded_call, host, synth

pytestmark = pytest.mark.gpu


def nhwc(a):
    return np.ascontiguousarray(np.transpose(a, (0, 2, 3, 1)))


def oracle_nhwc(x_nchw, k, s, p, d):
    return nhwc(O.maxpool2d(x_nchw, k, s, p, d))


# (N, C, H, W, k, s, p, d): band kernel cases (s = d = 1, C % 4 == 0) and direct ones
CASES = [
    (2, 64, 37, 40, 4, 1, 1, 1),    # the page's (k4 s1 p1 d1), ragged band
    (1, 16, 70, 33, 4, 1, 1, 1),    # several bands of 32 output rows, odd width
    (1, 8, 45, 19, 3, 1, 1, 1),
    (2, 4, 20, 21, 5, 1, 2, 1),
    (1, 12, 17, 9, 2, 1, 1, 1),     # output wider than input
    (1, 20, 9, 10, 1, 1, 0, 1),     # identity; 20 channels: 5 groups of 4
    (1, 48, 33, 14, 4, 1, 2, 1),    # 256 % 48 != 0: the block's last threads idle
    (1, 1024, 6, 5, 3, 1, 1, 1),    # one output column per block
    (1, 1028, 5, 4, 2, 1, 1, 1),    # C > 1024 -> direct kernel
    (2, 3, 13, 14, 4, 1, 1, 1),     # C % 4 != 0 -> direct kernel
    (1, 8, 30, 30, 3, 2, 1, 1),     # stride 2 -> direct kernel
    (1, 4, 25, 27, 3, 1, 1, 2),     # dilation 2 -> direct kernel
    (1, 6, 6, 8, 2, 1, 2, 1),       # windows of padding only -> -inf
]


@pytest.mark.parametrize("case", CASES)
def test_nhwc_small_bit_exact(case):
    N, C, H, W, k, s, p, d = case
    x = synth.maxpool_inputs(N, C, H, W, seed=sum(case))["x"]
    Ho, Wo = FW.fw_maxpool2d_out_shape(H, W, k, s, p, d)
    got = guarded_call(FW.fw_maxpool2d_nhwc, (N, Ho, Wo, C), dev(nhwc(x)), k, s, p, d)
    assert_bits_equal(got, oracle_nhwc(x, k, s, p, d), str(case))


def test_nhwc_special_values():
    """Signed zeros, NaN, +-inf: ties keep the first tap in row-major order, NaN propagates."""
    rng = np.random.default_rng(17)
    vals = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 0.5], np.float32)
    for (C, k, p) in ((16, 4, 1), (8, 3, 1), (6, 4, 2)):
        x = rng.choice(vals, size=(1, C, 23, 19), p=[.3, .3, .1, .1, .04, .04, .02, .1]).astype(np.float32)
        got = host(FW.fw_maxpool2d_nhwc(dev(nhwc(x)), k, 1, p, 1))
        assert_bits_equal(got, oracle_nhwc(x, k, 1, p, 1), str((C, k, p)))


def test_nhwc_full_size_equals_nchw_kernel():
    """x [32,64,512,512] (as NHWC) k4 s1 p1: the same bits as the NCHW call, transposed."""
    x = torch.from_numpy(synth.maxpool_inputs(32, 64, 512, 512, seed=0)["x"]).cuda()
    ref = FW.fw_maxpool2d(x, 4, 1, 1, 1)
    xn = x.permute(0, 2, 3, 1).contiguous()
    del x
    got = FW.fw_maxpool2d_nhwc(xn, 4, 1, 1, 1)
    FW.fw_check_device_errors()
    assert torch.equal(got, ref.permute(0, 2, 3, 1)), "channels-last result differs from the NCHW kernel's"


def test_nhwc_errors():
    x = torch.zeros(1, 8, 8, 4, device="cuda")
    with pytest.raises(FW.FusedWinError, match="FW_ERR_ALIAS"):
        FW.fw_maxpool2d_nhwc(x, 1, 1, 0, 1, out=x)
    with pytest.raises(ValueError):
        FW.fw_maxpool2d_nhwc(x, 3, 1, 1, 1, out=torch.empty(1, 8, 8, 5, device="cuda"))
