"""MaxPool2d: CUDA path (through the C ABI) vs the oracle, bit for bit."""
import numpy as np
import pytest
import torch

from tests.parity import FW, O, assert_bits_equal, dev, guarded_call, host, pmap, sample_indices, synth

pytestmark = pytest.mark.gpu

# (N, C, H, W, k, s, p, d): streaming-kernel cases (s=1, d=1, W%4==0) and direct ones.
CASES = [
    (2, 3, 37, 64, 4, 1, 1, 1),     # the page's (k4 s1 p1 d1), ragged height
    (1, 2, 300, 512, 4, 1, 1, 1),   # several row bands of one plane
    (3, 2, 129, 128, 4, 1, 2, 1),
    (2, 2, 41, 36, 4, 1, 0, 1),     # W % 128 != 0: partial warp of threads
    (1, 3, 33, 32, 3, 1, 1, 1),
    (1, 1, 20, 44, 5, 1, 2, 1),
    (2, 1, 17, 40, 2, 1, 1, 1),     # output wider than input (Wo = W + 1)
    (1, 2, 9, 32, 1, 1, 0, 1),      # identity
    (1, 2, 12, 48, 5, 1, 0, 1),
    (2, 3, 37, 61, 4, 1, 1, 1),     # W odd -> direct kernel
    (2, 2, 30, 30, 3, 2, 1, 1),     # stride 2
    (1, 2, 25, 27, 3, 2, 1, 2),     # dilation 2
    (1, 1, 19, 23, 4, 3, 2, 2),
    (1, 2, 6, 8, 2, 1, 2, 1),       # p > k/2: windows of padding only -> -inf
    (1, 1, 5, 5000, 4, 1, 1, 1),    # row too wide for one CTA -> direct kernel
]


@pytest.mark.parametrize("case", CASES)
def test_maxpool_small_bit_exact(case):
    N, C, H, W, k, s, p, d = case
    x = synth.maxpool_inputs(N, C, H, W, seed=sum(case))["x"]
    got = guarded_call(FW.fw_maxpool2d, (N, C) + FW.fw_maxpool2d_out_shape(H, W, k, s, p, d), dev(x), k, s, p, d)
    want = O.maxpool2d(x, k, s, p, d)
    assert got.shape == want.shape
    assert_bits_equal(got, want, str(case))


# (k, s, d, p) with a strided / dilated streaming kernel
SD = [(2, 2, 1, 0), (2, 2, 1, 1), (3, 2, 1, 0), (3, 2, 1, 1), (4, 2, 1, 1), (5, 2, 1, 2), (3, 3, 1, 0), (3, 3, 1, 1),
      (4, 4, 1, 0), (3, 1, 2, 1), (3, 1, 2, 2), (2, 1, 2, 1)]


@pytest.mark.parametrize("k,s,d,p", SD)
def test_strided_dilated_stream_bit_exact(k, s, d, p):
    for N, C, H, W in ((1, 2, 301, 512), (2, 1, 37, 64), (1, 1, 23, 132)):
        x = synth.maxpool_inputs(N, C, H, W, seed=k + 10 * s + 100 * d + p + W)["x"]
        got = guarded_call(FW.fw_maxpool2d, (N, C) + FW.fw_maxpool2d_out_shape(H, W, k, s, p, d), dev(x), k, s, p, d)
        assert_bits_equal(got, O.maxpool2d(x, k, s, p, d), str((N, C, H, W, k, s, p, d)))
    rng = np.random.default_rng(k + s + d + p)
    x = rng.choice(np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 0.5], np.float32),
                   size=(1, 2, 29, 64), p=[.3, .3, .1, .1, .04, .04, .02, .1]).astype(np.float32)
    assert_bits_equal(host(FW.fw_maxpool2d(dev(x), k, s, p, d)), O.maxpool2d(x, k, s, p, d), "special values")


def test_maxpool_special_values():
    """Signed zeros, NaN, +-inf: ties keep the first tap, NaN propagates."""
    rng = np.random.default_rng(7)
    for W in (64, 61):
        x = rng.choice(np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 0.5], np.float32),
                       size=(2, 2, 23, W), p=[.3, .3, .1, .1, .04, .04, .02, .1]).astype(np.float32)
        got = host(FW.fw_maxpool2d(dev(x), 4, 1, 1, 1))
        assert_bits_equal(got, O.maxpool2d(x, 4, 1, 1, 1), f"special W={W}")
        got = host(FW.fw_maxpool2d(dev(x), 3, 2, 1, 1))
        assert_bits_equal(got, O.maxpool2d(x, 3, 2, 1, 1), f"special s2 W={W}")


def test_maxpool_all_padding_window_is_minus_inf():
    x = synth.maxpool_inputs(1, 1, 4, 8, seed=3)["x"]
    got = host(FW.fw_maxpool2d(dev(x), 1, 1, 1, 1))  # k=1, p=1: the border ring sees only padding
    want = O.maxpool2d(x, 1, 1, 1, 1)
    assert_bits_equal(got, want)
    assert np.isneginf(got[0, 0, 0, 0]) and np.isneginf(got[0, 0, -1, -1])


def test_maxpool_host_buffers_roundtrip():
    x = synth.maxpool_inputs(2, 2, 40, 64, seed=5)["x"]
    got = FW.fw_maxpool2d(torch.from_numpy(x).pin_memory(), 4, 1, 1, 1)
    assert got.device.type == "cpu"
    assert_bits_equal(got.numpy(), O.maxpool2d(x, 4, 1, 1, 1))


def test_maxpool_errors_raise():
    x = torch.zeros(1, 1, 4, 4, device="cuda")
    with pytest.raises(FW.FusedWinError, match="FW_ERR_PARAM"):
        FW.fw_maxpool2d(x, 2, 1, 0, 0)
    with pytest.raises(FW.FusedWinError, match="FW_ERR_SHAPE"):
        FW.fw_maxpool2d(x, 5, 1, 0, 1)
    with pytest.raises(FW.FusedWinError, match="FW_ERR_ALIAS"):
        FW.fw_maxpool2d(x, 1, 1, 0, 1, out=x)
    FW.fw_check_device_errors()


def test_maxpool_full_size_bit_exact_sampled():
    """x [32,64,512,512], k4 s1 p1 d1 -> [32,64,511,511]: whole planes and random
    outputs against the oracle, in the launch configuration the benchmark times."""
    N, C, H, W = 32, 64, 512, 512
    x = synth.maxpool_inputs(N, C, H, W, seed=0)["x"]
    xd = dev(x)
    out = FW.fw_maxpool2d(xd, 4, 1, 1, 1)
    FW.fw_check_device_errors()
    assert tuple(out.shape) == (32, 64, 511, 511)
    planes = [(0, 0), (31, 63), (17, 5), (3, 40)]
    for n, c in planes:
        got = out[n, c].cpu().numpy()
        want = O.maxpool2d(x[n:n + 1, c:c + 1], 4, 1, 1, 1)[0, 0]
        assert_bits_equal(got, want, f"plane {(n, c)}")
    idx = sample_indices((N, C, 511, 511), 4000, seed=11)
    got = out.cpu().numpy()
    want = pmap(lambda t: O.maxpool2d_at(x, 4, 1, 1, 1, *t), idx)
    assert_bits_equal(np.array([got[t] for t in idx]), np.array(want), "samples")
    # invariants on everything: out >= its window's centre tap and finite
    assert np.all(np.isfinite(got))
    assert np.all(got >= x[:, :, :511, :511]) and np.all(got >= x[:, :, 1:, 1:])
