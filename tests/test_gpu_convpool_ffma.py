"""Fused conv3x3+tanh+scale+bias+maxpool on the float32 FMA pipe only
(fw_conv2d_tanh_scale_bias_maxpool_ffma): CUDA path vs the oracle (max abs err <= 1e-5)."""
import numpy as np
import pytest

from tests.parity import FW, O, TOL_FFMA, assert_close, dev, host, pmap, sample_indices, synth

pytestmark = pytest.mark.gpu


def run_gpu(d, scale, pk, ps=0, cb=True):
    return host(FW.fw_conv2d_tanh_scale_bias_maxpool_ffma(dev(d["x"]), dev(d["w"]), dev(d["conv_b"]) if cb else None,
                                                          dev(d["bias"]), scale, pk, ps))


def run_oracle(d, scale, pk, ps=0, cb=True):
    return O.conv2d_tanh_scale_bias_maxpool(d["x"], d["w"], d["conv_b"] if cb else None, scale, d["bias"], pk,
                                            ps or pk)


# (N, Cin, H, W, Cout, pool_k, pool_s, scale): tiled FMA kernel (the tensor-core shapes among them)
# and the direct kernel.
CASES = [
    (2, 8, 64, 64, 64, 4, 0, 2.0),     # the tiny workload
    (1, 8, 37, 70, 64, 4, 0, 2.0),
    (2, 8, 41, 33, 16, 2, 0, 2.0),
    (1, 3, 22, 19, 20, 4, 0, 2.0),
    (1, 16, 18, 35, 8, 2, 0, 1.0),
    (2, 5, 30, 30, 6, 4, 0, -1.5),     # negative scale: window minimum
    (1, 8, 26, 26, 12, 4, 0, 0.0),     # zero scale: out == bias
    (3, 8, 70, 130, 40, 4, 0, 2.0),    # several items per CTA, ragged edges, two channel blocks
    (1, 17, 20, 20, 8, 4, 0, 2.0),     # Cin > 16 -> direct kernel
    (2, 4, 21, 23, 8, 3, 2, 2.0),      # overlapping pool -> direct kernel
]


@pytest.mark.parametrize("case", CASES)
def test_shapes(case):
    N, Cin, H, W, Cout, pk, ps, scale = case
    d = synth.convpool_inputs(N, Cin, H, W, Cout, seed=N + H + W + Cin)
    assert_close(run_gpu(d, scale, pk, ps), run_oracle(d, scale, pk, ps), TOL_FFMA, str(case))


def test_no_conv_bias_and_unaligned_width():
    d = synth.convpool_inputs(2, 8, 33, 67, 32, seed=5)   # W % 4 != 0: 4-byte staging copies
    assert_close(run_gpu(d, 2.0, 4, cb=False), run_oracle(d, 2.0, 4, cb=False), TOL_FFMA, "W=67 no-cb")


def test_full_size_sampled():
    """x [128,8,256,256], Conv 8->64 k3, MaxPool2d(4) -> [128,64,63,63] on the FMA pipe."""
    d = synth.convpool_inputs(128, 8, 256, 256, 64, seed=0)
    got = run_gpu(d, 2.0, 4)
    FW.fw_check_device_errors()
    assert got.shape == (128, 64, 63, 63)
    idx = sample_indices(got.shape, 1500, seed=7)
    want = pmap(lambda t: O.convpool_at(d["x"], d["w"], d["conv_b"], 2.0, d["bias"], 4, 4, *t), idx)
    assert_close(np.array([got[t] for t in idx]), np.array(want), TOL_FFMA, "samples")
    sub = dict(d, x=d["x"][127:128])
    assert_close(got[127:128], run_oracle(sub, 2.0, 4), TOL_FFMA, "last image")
