"""Host-buffer entry points (chunked, pipelined copies): results bit-identical to the
device calls, for batches split into several chunks, pinned and pageable memory."""
import numpy as np
import pytest
import torch

from tests.parity import FW, assert_bits_equal, dev, host, synth

pytestmark = pytest.mark.gpu


def cpu(a, pin=True):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory() if pin else t


@pytest.mark.parametrize("N,pin", [(1, True), (3, True), (13, True), (9, False)])
def test_convpool_host(N, pin):
    d = synth.convpool_inputs(N, 8, 40, 36, 64, seed=N)
    want = host(FW.fw_conv2d_tanh_scale_bias_maxpool(dev(d["x"]), dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]),
                                                     2.0, 4))
    got = FW.fw_conv2d_tanh_scale_bias_maxpool_host(cpu(d["x"], pin), cpu(d["w"], pin), cpu(d["conv_b"], pin),
                                                    cpu(d["bias"], pin), 2.0, 4)
    assert_bits_equal(got.numpy(), want, f"N={N}")
    got = FW.fw_conv2d_tanh_scale_bias_maxpool_host(cpu(d["x"]), cpu(d["w"]), None, cpu(d["bias"]), -1.0, 2)
    want = host(FW.fw_conv2d_tanh_scale_bias_maxpool(dev(d["x"]), dev(d["w"]), None, dev(d["bias"]), -1.0, 2))
    assert_bits_equal(got.numpy(), want, "no conv_b")


@pytest.mark.parametrize("N,pin", [(2, True), (11, True), (5, False)])
def test_maxpool_host(N, pin):
    x = synth.maxpool_inputs(N, 3, 64, 64, seed=N)["x"]
    want = host(FW.fw_maxpool2d(dev(x), 4, 1, 1, 1))
    assert_bits_equal(FW.fw_maxpool2d_host(cpu(x, pin), 4, 1, 1, 1).numpy(), want, f"N={N}")
    want = host(FW.fw_maxpool2d(dev(x), 3, 2, 1, 2))
    assert_bits_equal(FW.fw_maxpool2d_host(cpu(x, pin), 3, 2, 1, 2).numpy(), want, "direct kernel")


@pytest.mark.parametrize("N,pin", [(1, True), (10, True), (4, False)])
def test_convt_host(N, pin):
    d = synth.convt_inputs(N, 64, 9, 10, 128, seed=N)
    want = host(FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(dev(d["x"]), dev(d["w"]), dev(d["conv_b"]),
                                                                 dev(d["bias"]), 2.0))
    got = FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_host(cpu(d["x"], pin), cpu(d["w"], pin),
                                                                cpu(d["conv_b"], pin), cpu(d["bias"], pin), 2.0)
    assert_bits_equal(got.numpy(), want, f"N={N}")


def test_host_call_orders_after_and_before_caller_stream():
    """Work queued on the caller's stream before the call finishes first; a
    synchronisation of that stream after the call sees the complete output."""
    d = synth.convpool_inputs(16, 8, 64, 64, 64, seed=7)
    x = cpu(d["x"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        busy = torch.randn(4096, 4096, device="cuda")
        for _ in range(20):
            busy = busy @ busy.T / 4096.0  # keep the stream busy before the call
        out = FW.fw_conv2d_tanh_scale_bias_maxpool_host(x, cpu(d["w"]), cpu(d["conv_b"]), cpu(d["bias"]), 2.0, 4,
                                                        stream=s)
    want = host(FW.fw_conv2d_tanh_scale_bias_maxpool(dev(d["x"]), dev(d["w"]), dev(d["conv_b"]), dev(d["bias"]),
                                                     2.0, 4))
    assert_bits_equal(out.numpy(), want, "ordered")
    FW.fw_check_device_errors()
