"""The bounds-checked build (FW_CHECKED): every kernel tests the address range of
its memory accesses, skips an access outside its buffer and records it in the
device error word.  The small-shape parity suite -- every kernel of the library,
on ragged and unaligned shapes -- runs against that library in a fresh process;
each test must still match the oracle, keep its output's canary guards intact and
leave fw_check_device_errors at FW_OK (tests/conftest.py checks the last after
every test).  This replaces a memory checker, which is not available here."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SELECTION = [
    "tests/test_gpu_random_shapes.py",
    "tests/test_gpu_convpool.py::test_small_shapes",
    "tests/test_gpu_convpool.py::test_tiny_config_full",
    "tests/test_gpu_convpool.py::test_other_kernel_sizes_and_no_conv_bias",
    "tests/test_gpu_convpool.py::test_input_rows_not_16_byte_aligned",
    "tests/test_gpu_convpool.py::test_tensor_kernel_cout_32_48",
    "tests/test_gpu_convpool_tf32.py::test_small_shapes",
    "tests/test_gpu_convpool_tf32.py::test_tiny_config_full",
    "tests/test_gpu_convpool_ffma.py::test_shapes",
    "tests/test_gpu_maxpool.py::test_maxpool_small_bit_exact",
    "tests/test_gpu_maxpool.py::test_strided_dilated_stream_bit_exact",
    "tests/test_gpu_maxpool.py::test_maxpool_special_values",
    "tests/test_gpu_maxpool.py::test_maxpool_all_padding_window_is_minus_inf",
    "tests/test_gpu_maxpool_ex.py::test_grid_against_oracle",
    "tests/test_gpu_maxpool_ex.py::test_window_without_input_tap",
    "tests/test_gpu_maxpool_nhwc.py::test_nhwc_small_bit_exact",
    "tests/test_gpu_maxpool_nhwc.py::test_nhwc_special_values",
    "tests/test_gpu_convpool_nhwc.py::test_nhwc_matches_oracle_and_nchw",
    "tests/test_gpu_convt.py::test_small_shapes",
    "tests/test_gpu_convt.py::test_no_conv_bias_and_negative_scale",
    "tests/test_gpu_convt.py::test_output_one_float_into_its_buffer",
    "tests/test_gpu_convt_nhwc.py::test_nhwc_matches_oracle_and_nchw",
    "tests/test_gpu_convt_accuracy.py::test_ffma_call_matches_forced_ffma_kernel_shapes",
    "tests/test_gpu_unfused.py::test_convpool_unfused_equals_fused",
    "tests/test_gpu_unfused.py::test_convt_unfused_matches_oracle",
    "tests/test_gpu_host.py",
]


def test_small_shape_parity_suite_under_the_checked_build():
    from pooling_sliding_window_gb300 import build
    build.build(checked=True)
    env = dict(os.environ, FUSEDWIN_CHECKED="1", FUSEDWIN_NO_BUILD="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        *SELECTION], cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = (r.stdout[-4000:] + "\n" + r.stderr[-2000:])
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "failed" not in r.stdout, tail
