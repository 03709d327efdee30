"""Fused conv3x3+tanh+scale+bias+maxpool: CUDA path vs the oracle (max abs err <= 1e-5)."""
import itertools

import numpy as np
import pytest
import torch

from tests.parity import FW, O, TOL_FFMA, assert_close, dev, guarded_call, host, pmap, sample_indices, synth

pytestmark = pytest.mark.gpu


def run_gpu(d, scale, pk, ps=0, cb=True):
    """The fused call into an output with canary guards on both sides."""
    N, Cout, KH = d["x"].shape[0], d["w"].shape[0], d["w"].shape[2]
    Ho, Wo = FW.fw_conv2d_pool_out_shape(d["x"].shape[2], d["x"].shape[3], KH, d["w"].shape[3], pk, ps)
    return guarded_call(FW.fw_conv2d_tanh_scale_bias_maxpool, (N, Cout, Ho, Wo), dev(d["x"]), dev(d["w"]),
                        dev(d["conv_b"]) if cb else None, dev(d["bias"]), scale, pk, ps)


def run_oracle(d, scale, pk, ps=0, cb=True):
    return O.conv2d_tanh_scale_bias_maxpool(d["x"], d["w"], d["conv_b"] if cb else None, scale, d["bias"],
                                            pk, ps or pk)


def test_tiny_config_full():
    """x [2,8,64,64], Conv 8->64 k3, tanh, *2, +bias, MaxPool2d(4) -> [2,64,15,15]."""
    d = synth.convpool_inputs(2, 8, 64, 64, 64, seed=0)
    got = run_gpu(d, 2.0, 4)
    assert got.shape == (2, 64, 15, 15)
    assert_close(got, run_oracle(d, 2.0, 4), TOL_FFMA, "tiny")


# (N, Cin, H, W, Cout, pool_k, pool_s, scale): tiled kernel and direct kernel cases.
CASES = [
    (1, 8, 37, 70, 64, 4, 0, 2.0),
    (2, 8, 41, 33, 16, 2, 0, 2.0),
    (1, 3, 22, 19, 20, 4, 0, 2.0),     # Cout not a multiple of the 32-channel block
    (1, 16, 18, 35, 8, 2, 0, 1.0),
    (2, 5, 30, 30, 6, 4, 0, -1.5),     # negative scale: window min
    (1, 8, 26, 26, 12, 4, 0, 0.0),     # zero scale: out == bias
    (1, 8, 6, 6, 4, 4, 0, 2.0),        # a single window
    (1, 8, 30, 70, 64, 4, 0, 2.0),     # 7 items on the tensor kernel
    (1, 8, 6, 6, 16, 4, 0, 2.0),       # one item on the tensor kernel
    (1, 17, 20, 20, 8, 4, 0, 2.0),     # Cin > 16 -> direct kernel
    (2, 4, 21, 23, 8, 3, 2, 2.0),      # overlapping pool -> direct kernel
    (1, 4, 15, 16, 8, 4, 4, 2.0),
]


@pytest.mark.parametrize("case", CASES)
def test_small_shapes(case):
    N, Cin, H, W, Cout, pk, ps, scale = case
    d = synth.convpool_inputs(N, Cin, H, W, Cout, seed=N + H + W)
    got = run_gpu(d, scale, pk, ps)
    assert_close(got, run_oracle(d, scale, pk, ps), TOL_FFMA, str(case))


def test_other_kernel_sizes_and_no_conv_bias():
    d = synth.convpool_inputs(2, 4, 19, 17, 8, k=5, seed=9)
    got = run_gpu(d, 2.0, 2, cb=False)
    assert_close(got, run_oracle(d, 2.0, 2, cb=False), TOL_FFMA, "k5 no-cb")
    d = synth.convpool_inputs(1, 8, 40, 40, 16, seed=10)
    assert_close(run_gpu(d, 2.0, 4, cb=False), run_oracle(d, 2.0, 4, cb=False), TOL_FFMA, "k3 no-cb")


def _check_images(d, got, images, pk, scale=2.0):
    for n in images:
        sub = dict(d, x=d["x"][n:n + 1])
        assert_close(got[n:n + 1], run_oracle(sub, scale, pk), TOL_FFMA, f"image {n}")


def _check_samples(d, got, count, pk, seed, scale=2.0):
    idx = sample_indices(got.shape, count, seed)
    want = pmap(lambda t: O.convpool_at(d["x"], d["w"], d["conv_b"], scale, d["bias"], pk, pk, *t), idx)
    assert_close(np.array([got[t] for t in idx]), np.array(want), TOL_FFMA, "samples")


SWEEP = list(itertools.product((1, 16, 128), (127, 255, 256), (16, 64), (2, 4), (0, 1, 2)))


@pytest.mark.parametrize("N,H,Cout,pk,seed", SWEEP)
def test_sweep(N, H, Cout, pk, seed):
    """batch {1,16,128} x H=W {127,255,256} x Cout {16,64} x pool {2,4} x seeds 0-2."""
    d = synth.convpool_inputs(N, 8, H, H, Cout, seed=seed)
    got = run_gpu(d, 2.0, pk)
    ho = O.pool_out_size(O.conv2d_out_size(H, 3), pk, pk)
    assert got.shape == (N, Cout, ho, ho)
    _check_images(d, got, sorted({0, N - 1}), pk)
    if N > 2:
        _check_samples(d, got, 200, pk, seed=N * 1000 + H + Cout + pk + seed)


def test_full_size_sampled():
    """x [128,8,256,256], Conv 8->64 k3, MaxPool2d(4) -> [128,64,63,63], the benchmarked launch."""
    d = synth.convpool_inputs(128, 8, 256, 256, 64, seed=0)
    got = run_gpu(d, 2.0, 4)
    FW.fw_check_device_errors()
    assert got.shape == (128, 64, 63, 63)
    _check_images(d, got, [0, 127], 4)
    _check_samples(d, got, 3000, 4, seed=1)
    b = d["bias"][None, :, None, None]
    assert np.all(got >= b - 2) and np.all(got <= b + 2)


def test_errors_raise():
    x = torch.zeros(1, 8, 16, 16, device="cuda")
    w = torch.zeros(4, 8, 3, 3, device="cuda")
    b = torch.zeros(4, device="cuda")
    with pytest.raises(FW.FusedWinError, match="FW_ERR_PARAM"):
        FW.fw_conv2d_tanh_scale_bias_maxpool(x, w, None, b, float("nan"), 4)
    with pytest.raises(FW.FusedWinError, match="FW_ERR_SHAPE"):
        FW.fw_conv2d_tanh_scale_bias_maxpool(x[:, :, :4, :4].contiguous(), w, None, b, 2.0, 4)


@pytest.mark.parametrize("N,H,W,Cout,pk", [(1, 36, 68, 32, 4), (2, 20, 132, 48, 2), (1, 30, 260, 48, 4)])
def test_tensor_kernel_cout_32_48(N, H, W, Cout, pk):
    """Cout 32 and 48 on the tensor-core kernel, W % 4 == 0 (float4 input rows), several column blocks."""
    d = synth.convpool_inputs(N, 8, H, W, Cout, seed=W)
    assert_close(run_gpu(d, 2.0, pk), run_oracle(d, 2.0, pk), TOL_FFMA, str((N, H, W, Cout, pk)))


def test_input_rows_not_16_byte_aligned():
    """x 4-byte aligned but not 16-byte aligned with W % 4 == 0: the tensor-core kernel
    must take its scalar-load path and give the same result."""
    d = synth.convpool_inputs(2, 8, 40, 64, 64, seed=11)
    flat = torch.zeros(d["x"].size + 1, dtype=torch.float32, device="cuda")
    x = flat[1:].view(d["x"].shape)
    x.copy_(torch.from_numpy(d["x"]))
    assert x.data_ptr() % 16 == 4
    got = host(FW.fw_conv2d_tanh_scale_bias_maxpool(x, dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]), -1.5, 4))
    assert_close(got, run_oracle(d, -1.5, 4), TOL_FFMA, "unaligned rows")


def test_ffma_kernel_when_forced():
    """The FP32-FMA tiled kernel (selected with FUSEDWIN_CONVPOOL_FFMA=1) on shapes the
    tensor-core kernel takes, in a fresh process."""
    import os
    import subprocess
    import sys
    import textwrap
    code = textwrap.dedent("""
        from tests.parity import FW, O, TOL_FFMA, assert_close, dev, host, synth
        for (N, H, W, Cout, pk) in ((2, 64, 64, 64, 4), (1, 41, 33, 16, 2)):
            d = synth.convpool_inputs(N, 8, H, W, Cout, seed=H)
            got = host(FW.fw_conv2d_tanh_scale_bias_maxpool(dev(d["x"]), dev(d["w"]), dev(d["conv_b"]),
                                                            dev(d["bias"]), 2.0, pk))
            want = O.conv2d_tanh_scale_bias_maxpool(d["x"], d["w"], d["conv_b"], 2.0, d["bias"], pk)
            assert_close(got, want, TOL_FFMA, str((N, H, W, Cout, pk)))
        print("ok")
    """)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       env=dict(os.environ, FUSEDWIN_CONVPOOL_FFMA="1"), timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr

