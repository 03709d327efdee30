"""Seeded random shapes for every operator and entry point, against the oracle: conv+pool
through the default, plain-TF32 and FP32-FMA calls (tensor-core, tiled-FMA and direct
kernels by shape), maxpool bit for bit over random (k, s, p, d), conv-transpose through the
tensor-core, tiled-FMA and direct kernels.  Sizes stay small enough for the oracle."""
import numpy as np
import pytest

from tests.parity import FW, O, TOL_FFMA, TOL_TF32, assert_bits_equal, assert_close, dev, host, synth

pytestmark = pytest.mark.gpu


def _convpool_cases(count, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(count):
        tc = i % 2 == 0  # every other case on a tensor-core shape
        Cin = 8 if tc else int(rng.integers(1, 17))
        Cout = int(rng.choice([16, 32, 48, 64])) if tc else int(rng.integers(1, 70))
        pk = int(rng.choice([2, 4])) if tc else int(rng.integers(1, 5))
        ps = pk if (tc or rng.random() < 0.7) else int(rng.integers(1, pk + 1))
        H = int(rng.integers(pk + 2, 90)); W = int(rng.integers(pk + 2, 140))
        N = int(rng.integers(1, 4))
        scale = float(rng.choice([2.0, -1.5, 0.5, 0.0]))
        cases.append((N, Cin, H, W, Cout, pk, ps, scale, 100 + i))
    return cases


@pytest.mark.parametrize("case", _convpool_cases(16, 1))
def test_convpool_random(case):
    N, Cin, H, W, Cout, pk, ps, scale, seed = case
    d = synth.convpool_inputs(N, Cin, H, W, Cout, seed=seed)
    want = O.conv2d_tanh_scale_bias_maxpool(d["x"], d["w"], d["conv_b"], scale, d["bias"], pk, ps)
    args = (dev(d["x"]), dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]), scale, pk, ps)
    assert_close(host(FW.fw_conv2d_tanh_scale_bias_maxpool(*args)), want, TOL_FFMA, f"default {case}")
    assert_close(host(FW.fw_conv2d_tanh_scale_bias_maxpool_ffma(*args)), want, TOL_FFMA, f"ffma {case}")
    assert_close(host(FW.fw_conv2d_tanh_scale_bias_maxpool_tf32(*args)), want, TOL_TF32, f"tf32 {case}")


def _maxpool_cases(count, seed):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < count:
        k = int(rng.integers(1, 6)); s = int(rng.integers(1, 4)); d = int(rng.integers(1, 4))
        p = int(rng.integers(0, k // 2 + 2))
        H = int(rng.integers(1, 70)); W = int(rng.choice([int(rng.integers(1, 70)), 4 * int(rng.integers(8, 40))]))
        span = d * (k - 1) + 1
        if H + 2 * p < span or W + 2 * p < span:
            continue
        cases.append((int(rng.integers(1, 3)), int(rng.integers(1, 5)), H, W, k, s, p, d, 200 + len(cases)))
    return cases


@pytest.mark.parametrize("case", _maxpool_cases(24, 2))
def test_maxpool_random(case):
    N, C, H, W, k, s, p, d, seed = case
    x = synth.maxpool_inputs(N, C, H, W, seed=seed)["x"]
    got = host(FW.fw_maxpool2d(dev(x), k, s, p, d))
    assert_bits_equal(got, O.maxpool2d(x, k, s, p, d), str(case))


def _convt_cases(count, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(count):
        kind = i % 3
        if kind == 0:    # tensor-core shapes: k4 s2 p1, Cout 128
            Cin, Cout, k, s, p = int(rng.choice([8, 16, 32, 64])), 128, 4, 2, 1
        elif kind == 1:  # tiled FMA kernel: k4 s2 p1, Cout 128, other Cin
            Cin, Cout, k, s, p = int(rng.integers(1, 40)), 128, 4, 2, 1
        else:            # direct kernel: any k, s, p
            k = int(rng.integers(1, 6)); s = int(rng.integers(1, 4)); p = int(rng.integers(0, k))
            Cin, Cout = int(rng.integers(1, 24)), int(rng.integers(1, 200))
        op = int(rng.integers(0, s))
        H = int(rng.integers(1, 20)); W = int(rng.integers(1, 24))
        if (H - 1) * s - 2 * p + k + op < 1 or (W - 1) * s - 2 * p + k + op < 1:
            p = 0
        cases.append((int(rng.integers(1, 3)), Cin, H, W, Cout, k, s, p, op, float(rng.choice([2.0, -1.0])), 300 + i))
    return cases


@pytest.mark.parametrize("case", _convt_cases(15, 3))
def test_convt_random(case):
    N, Cin, H, W, Cout, k, s, p, op, scale, seed = case
    d = synth.convt_inputs(N, Cin, H, W, Cout, k=k, seed=seed)
    got = host(FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(dev(d["x"]), dev(d["w"]), dev(d["conv_b"]),
                                                                dev(d["bias"]), scale, s, p, op))
    want = O.convtranspose2d_softmax_bias_scale_sigmoid(d["x"], d["w"], d["conv_b"], d["bias"], scale, s, p, op)
    assert_close(got, want, TOL_FFMA, str(case))
