"""MaxPool2d with ceil mode and argmax indices (PyTorch's options, an extension beyond
the pages): values bit-exact and indices exact against the oracle."""
import numpy as np
import pytest
import torch

from tests.parity import FW, O, assert_bits_equal, dev, host, synth

pytestmark = pytest.mark.gpu

GRID = [(k, s, p, d) for k in (1, 2, 3, 4, 5) for s in (1, 2, 3) for p in range(0, k // 2 + 1) for d in (1, 2)]


def inputs(shape, seed, ties=False, nans=0):
    rng = np.random.default_rng(seed)
    x = rng.integers(-3, 4, size=shape).astype(np.float32) if ties else rng.standard_normal(shape).astype(np.float32)
    flat = x.reshape(-1)
    if nans:
        flat[rng.choice(flat.size, nans, replace=False)] = np.nan
    return x


@pytest.mark.parametrize("ceil_mode", [False, True])
@pytest.mark.parametrize("ties,nans", [(False, 0), (True, 0), (False, 9)])
def test_grid_against_oracle(ceil_mode, ties, nans):
    x = inputs((2, 3, 17, 13), seed=int(ceil_mode) + 2 * int(ties) + nans, ties=ties, nans=nans)
    xd = dev(x)
    for k, s, p, d in GRID:
        if 13 + 2 * p - d * (k - 1) - 1 < 0:
            continue
        want, want_idx = O.maxpool2d_ex(x, k, s, p, d, ceil_mode)
        got, idx = FW.fw_maxpool2d_ex(xd, k, s, p, d, ceil_mode=ceil_mode, return_indices=True)
        assert_bits_equal(host(got), want, str((k, s, p, d, ceil_mode)))
        np.testing.assert_array_equal(host(idx), want_idx, err_msg=str((k, s, p, d, ceil_mode)))
        if not ceil_mode or s == 1:  # without indices: the same values as fw_maxpool2d
            assert_bits_equal(host(FW.fw_maxpool2d_ex(xd, k, s, p, d, ceil_mode=ceil_mode)), want, "no indices")


def test_window_without_input_tap():
    x = inputs((1, 1, 5, 6), seed=4)
    out, idx = FW.fw_maxpool2d_ex(dev(x), 1, 1, 1, 1, return_indices=True)
    want, want_idx = O.maxpool2d_ex(x, 1, 1, 1, 1, False)
    np.testing.assert_array_equal(host(idx), want_idx)
    assert host(idx)[0, 0, 0, 0] == -1 and np.isneginf(host(out)[0, 0, 0, 0])


def test_streaming_workload_with_indices_sampled():
    """x [32,64,512,512], k4 s1 p1 d1 with indices: the index picks the value, and sampled outputs match."""
    x = synth.maxpool_inputs(32, 64, 512, 512, seed=1)["x"]
    out, idx = FW.fw_maxpool2d_ex(dev(x), 4, 1, 1, 1, return_indices=True)
    FW.fw_check_device_errors()
    o, i = host(out), host(idx)
    plain = host(FW.fw_maxpool2d(dev(x), 4, 1, 1, 1))
    assert_bits_equal(o, plain, "values vs streaming kernel")
    flat = x.reshape(32 * 64, -1)
    picked = np.take_along_axis(flat, i.reshape(32 * 64, -1), axis=1).reshape(o.shape)
    assert_bits_equal(picked, o, "x[idx] == out")
    rng = np.random.default_rng(2)
    for _ in range(200):
        n, c, oh, ow = (int(rng.integers(0, m)) for m in (32, 64, 511, 511))
        v, at = O.maxpool2d_ex(x[n:n + 1, c:c + 1], 4, 1, 1, 1, False)
        assert i[n, c, oh, ow] == at[0, 0, oh, ow]
