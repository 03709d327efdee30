"""The OpenMP build of the oracle (the same C source compiled with -fopenmp, used
only to time the definition at full size on the host cores) gives bit-identical
results to the single-threaded oracle: its pragmas only spread independent images,
channels and planes over threads."""
import os

import numpy as np
import pytest

os.environ.setdefault("OMP_NUM_THREADS", "4")

from oracle import oracle as O  # noqa: E402
from pooling_sliding_window_gb300 import synth  # noqa: E402


def _same(a, b):
    return np.array_equal(np.asarray(a).view(np.uint32), np.asarray(b).view(np.uint32))


@pytest.mark.parametrize("N,H,Cout,pool", [(3, 20, 16, 2), (2, 31, 64, 4)])
def test_convpool_openmp_bit_identical(N, H, Cout, pool):
    d = synth.convpool_inputs(N, 8, H, H + 3, Cout, seed=N + H)
    a = O.conv2d_tanh_scale_bias_maxpool(d["x"], d["w"], d["conv_b"], 2.0, d["bias"], pool)
    b = O.conv2d_tanh_scale_bias_maxpool(d["x"], d["w"], d["conv_b"], 2.0, d["bias"], pool, openmp=True)
    assert _same(a, b)


@pytest.mark.parametrize("k,s,p,d", [(4, 1, 1, 1), (3, 2, 1, 2)])
def test_maxpool_openmp_bit_identical(k, s, p, d):
    x = synth.maxpool_inputs(3, 5, 33, 40, seed=k)["x"]
    assert _same(O.maxpool2d(x, k, s, p, d), O.maxpool2d(x, k, s, p, d, openmp=True))


def test_convt_openmp_bit_identical():
    d = synth.convt_inputs(3, 16, 7, 9, 128, seed=4)
    a = O.convtranspose2d_softmax_bias_scale_sigmoid(d["x"], d["w"], d["conv_b"], d["bias"], 2.0)
    b = O.convtranspose2d_softmax_bias_scale_sigmoid(d["x"], d["w"], d["conv_b"], d["bias"], 2.0, openmp=True)
    assert _same(a, b)
    a = O.convtranspose2d_softmax_bias_scale_sigmoid(d["x"][:1], d["w"][:, :32, :3, :3], None, d["bias"][:32],
                                                     -1.5, 2, 0, 1)
    b = O.convtranspose2d_softmax_bias_scale_sigmoid(d["x"][:1], d["w"][:, :32, :3, :3], None, d["bias"][:32],
                                                     -1.5, 2, 0, 1, openmp=True)
    assert _same(a, b)
