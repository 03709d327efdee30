"""The allocation-free conv-transpose entry point, called through the C ABI.

It serves callers that cannot allocate device memory (plugins handed only
input and output buffers by a framework that owns all device memory, real-time
loops that may not allocate after start-up, code where an allocation would
synchronise the device): instead of a caller workspace it uses a fixed device
array inside the library.  This file is collected last on purpose; it must pass
alone in a fresh process and after the other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from oracle import oracle as O
from pooling_sliding_window_gb300 import fusedwin as FW
from pooling_sliding_window_gb300 import synth
from tests.parity import TOL_FFMA

pytestmark = pytest.mark.gpu


def _noalloc(L, t, out, Cin, Cout, H, W, N):
    stream = torch.cuda.current_stream().cuda_stream
    return L.fw_convtranspose2d_softmax_bias_scale_sigmoid_noalloc(
        C.c_void_p(t["x"].data_ptr()), N, Cin, H, W, C.c_void_p(t["w"].data_ptr()),
        C.c_void_p(t["conv_b"].data_ptr()), Cout, 4, 2, 1, 1, C.c_void_p(t["bias"].data_ptr()), 2.0,
        C.c_void_p(out.data_ptr()), C.c_void_p(stream))


def test_noalloc_matches_workspace_entry_point_twice():
    L = FW.lib()
    N, Cin, H, W, Cout = 2, 64, 9, 10, 128
    assert FW.fw_convt_workspace_size(Cin, Cout, 4, 2, 1) > 0  # the path that needs scratch
    for call, seed in enumerate((31, 32)):  # two calls in a row, different weights
        d = synth.convt_inputs(N, Cin, H, W, Cout, seed=seed)
        t = {k: torch.from_numpy(v).cuda() for k, v in d.items()}
        ref = FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(t["x"], t["w"], t["conv_b"], t["bias"], 2.0)
        out = torch.full_like(ref, float("nan"))
        rc = _noalloc(L, t, out, Cin, Cout, H, W, N)
        assert rc == 0, FW.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        err = float((out - ref).abs().max())
        assert np.isfinite(err) and err <= TOL_FFMA, f"call {call}: max abs diff {err}"
        # and against the oracle itself, on the same inputs
        want = O.convtranspose2d_softmax_bias_scale_sigmoid(d["x"], d["w"], d["conv_b"], d["bias"], 2.0)
        got = out.cpu().numpy().astype(np.float64)
        err_o = float(np.abs(got - want).max())
        assert got.shape == want.shape and np.isfinite(err_o) and err_o <= TOL_FFMA, \
            f"call {call}: max abs err vs oracle {err_o}"
    FW.fw_check_device_errors()


def test_noalloc_rejects_rewrite_larger_than_the_array():
    L = FW.lib()
    # Cin = 256 at Cout = 128 needs 16*256*128*4 = 2 MiB > 1 MiB: refused before any launch.
    N, Cin, H, W, Cout = 1, 256, 4, 4, 128
    assert FW.fw_convt_workspace_size(Cin, Cout, 4, 2, 1) > (1 << 20)
    t = {"x": torch.zeros(N, Cin, H, W, device="cuda"), "w": torch.zeros(Cin, Cout, 4, 4, device="cuda"),
         "conv_b": torch.zeros(Cout, device="cuda"), "bias": torch.zeros(Cout, device="cuda")}
    out = torch.zeros(N, Cout, 9, 9, device="cuda")
    n0 = FW.fw_launch_count()
    assert _noalloc(L, t, out, Cin, Cout, H, W, N) == 6  # FW_ERR_UNSUPPORTED
    assert FW.fw_launch_count() == n0
