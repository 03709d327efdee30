"""ConvTranspose2d+softmax+bias+scale+sigmoid: CUDA path vs the oracle (max abs err <= 1e-5)."""
import numpy as np
import pytest
import torch

from tests.parity import FW, O, TOL_FFMA, assert_close, dev, guarded_call, host, pmap, sample_indices, synth

pytestmark = pytest.mark.gpu


def run_gpu(d, scale, s=2, p=1, op=1, cb=True, lead=0):
    """The fused call into an output with canary guards on both sides."""
    N, _, H, W = d["x"].shape
    Cout, K = d["w"].shape[1], d["w"].shape[2]
    return guarded_call(FW.fw_convtranspose2d_softmax_bias_scale_sigmoid,
                        (N, Cout) + FW.fw_convt_out_shape(H, W, K, s, p, op), dev(d["x"]), dev(d["w"]),
                        dev(d["conv_b"]) if cb else None, dev(d["bias"]), scale, s, p, op, lead=lead)


def run_oracle(d, scale, s=2, p=1, op=1, cb=True):
    return O.convtranspose2d_softmax_bias_scale_sigmoid(d["x"], d["w"], d["conv_b"] if cb else None,
                                                        d["bias"], scale, s, p, op)


# (N, Cin, H, W, Cout, k, s, p, op)
CASES = [
    (2, 64, 9, 10, 128, 4, 2, 1, 1),    # the page's layer on a small image (tiled kernel)
    (1, 64, 16, 16, 128, 4, 2, 1, 1),
    (1, 20, 5, 7, 128, 4, 2, 1, 1),     # Cin not a multiple of the 16-channel chunk
    (2, 8, 11, 3, 128, 4, 2, 1, 0),     # output_padding 0
    (1, 64, 17, 33, 128, 4, 2, 1, 1),   # several tiles, ragged in both directions
    (1, 64, 3, 100, 128, 4, 2, 1, 1),   # wide rows: one vertical tap per slab (two slabs per tile)
    (1, 16, 3, 100, 128, 4, 2, 1, 1),   # a slab wider than the producer threads
    (2, 16, 6, 5, 64, 4, 2, 1, 1),      # Cout != 128 -> direct kernel
    (1, 8, 5, 6, 32, 3, 2, 0, 1),
    (1, 6, 4, 5, 16, 5, 3, 2, 2),
    (1, 4, 6, 6, 8, 3, 1, 1, 0),
]


@pytest.mark.parametrize("case", CASES)
def test_small_shapes(case):
    N, Cin, H, W, Cout, k, s, p, op = case
    d = synth.convt_inputs(N, Cin, H, W, Cout, k=k, seed=H + W)
    got = run_gpu(d, 2.0, s, p, op)
    want = run_oracle(d, 2.0, s, p, op)
    assert got.shape == want.shape
    assert_close(got, want, TOL_FFMA, str(case))


@pytest.mark.parametrize("N,Cin,H,W,op", [(2, 64, 9, 10, 1), (1, 64, 17, 33, 1), (1, 16, 3, 100, 1),
                                         (2, 8, 11, 3, 0), (1, 32, 6, 64, 1)])
def test_output_one_float_into_its_buffer(N, Cin, H, W, op):
    """An output starting 4 bytes past an 8-byte boundary: the tiled kernel picks its 8-byte
    stores by the parity of each channel's first element, which this start flips."""
    d = synth.convt_inputs(N, Cin, H, W, 128, seed=N + H + W)
    got = run_gpu(d, 2.0, op=op, lead=1)
    assert_close(got, run_oracle(d, 2.0, op=op), TOL_FFMA, str((N, Cin, H, W, op)))


def test_no_conv_bias_and_negative_scale():
    d = synth.convt_inputs(1, 64, 8, 8, 128, seed=3)
    assert_close(run_gpu(d, 2.0, cb=False), run_oracle(d, 2.0, cb=False), TOL_FFMA, "no-cb")
    assert_close(run_gpu(d, -3.0), run_oracle(d, -3.0), TOL_FFMA, "scale -3")


def test_full_size_sampled():
    """x [128,64,64,64] -> ConvTranspose2d(64->128, k4, s2, p1, op1) -> [128,128,129,129]."""
    d = synth.convt_inputs(128, 64, 64, 64, 128, seed=0)
    got = run_gpu(d, 2.0)
    FW.fw_check_device_errors()
    assert got.shape == (128, 128, 129, 129)
    sub = dict(d, x=d["x"][:1])
    assert_close(got[:1], run_oracle(sub, 2.0), TOL_FFMA, "image 0")
    pix = sample_indices((128, 129, 129), 1500, seed=2)
    want = pmap(lambda t: O.convt_fused_pixel(d["x"], d["w"], d["conv_b"], d["bias"], 2.0, 2, 1, *t), pix)
    assert_close(np.stack([got[n, :, oh, ow] for n, oh, ow in pix]), np.stack(want), TOL_FFMA, "pixels")
    assert np.all((got > 0) & (got < 1))


def test_errors_raise():
    x = torch.zeros(1, 4, 4, 4, device="cuda")
    w = torch.zeros(4, 8, 4, 4, device="cuda")
    b = torch.zeros(8, device="cuda")
    with pytest.raises(FW.FusedWinError, match="FW_ERR_PARAM"):
        FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(x, w, None, b, 2.0, 2, 1, 2)


def test_ffma_kernel_when_forced():
    """The FP32-FMA tiled kernel (selected with FUSEDWIN_CONVT_FFMA=1) on the same
    shapes the tensor-core kernel takes, in a fresh process."""
    import subprocess
    import sys
    import textwrap
    code = textwrap.dedent("""
        import numpy as np, torch
        from tests.parity import FW, O, TOL_FFMA, assert_close, dev, host, synth
        for (N, Cin, H, W) in ((2, 64, 9, 10), (1, 32, 17, 33)):
            d = synth.convt_inputs(N, Cin, H, W, 128, seed=H)
            got = host(FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(
                dev(d["x"]), dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]), 2.0))
            want = O.convtranspose2d_softmax_bias_scale_sigmoid(d["x"], d["w"], d["conv_b"], d["bias"], 2.0)
            assert_close(got, want, TOL_FFMA, str((N, Cin, H, W)))
        print("ok")
    """)
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       env=dict(os.environ, FUSEDWIN_CONVT_FFMA="1"), timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr

