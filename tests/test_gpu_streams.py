"""Calls on several CUDA streams at once: each operator's result on a side stream, with
other operators running concurrently on others, equals its result on the default stream
bit for bit (the kernels keep no state between calls beyond the caller's buffers)."""
import pytest
import torch

from tests.parity import FW, dev, synth

pytestmark = pytest.mark.gpu


def test_concurrent_streams_give_the_same_bits():
    cp = synth.convpool_inputs(8, 8, 96, 96, 64, seed=1)
    mp = synth.maxpool_inputs(4, 16, 128, 128, seed=2)
    ct = synth.convt_inputs(4, 64, 24, 24, 128, seed=3)
    cpd = {k: dev(v) for k, v in cp.items()}
    mpx = dev(mp["x"])
    ctd = {k: dev(v) for k, v in ct.items()}

    def run_all(outs, ws):
        FW.fw_conv2d_tanh_scale_bias_maxpool(cpd["x"], cpd["w"], cpd["conv_b"], cpd["bias"], 2.0, 4, out=outs[0])
        FW.fw_maxpool2d(mpx, 4, 1, 1, 1, out=outs[1])
        FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(ctd["x"], ctd["w"], ctd["conv_b"], ctd["bias"], 2.0,
                                                         out=outs[2], workspace=ws)
        FW.fw_conv2d_tanh_scale_bias_maxpool_nhwc(cpd["x"].permute(0, 2, 3, 1).contiguous(), cpd["w"], cpd["conv_b"],
                                                  cpd["bias"], 2.0, 4, out=outs[3])

    def new_outs():
        return [torch.empty(8, 64, 23, 23, device="cuda"), torch.empty(4, 16, 127, 127, device="cuda"),
                torch.empty(4, 128, 49, 49, device="cuda"), torch.empty(8, 23, 23, 64, device="cuda")]

    ws_size = FW.fw_convt_workspace_size(64, 128, 4, 2, 1)
    ref = new_outs()
    run_all(ref, torch.empty(ws_size // 4, device="cuda"))
    torch.cuda.synchronize()

    streams = [torch.cuda.Stream() for _ in range(3)]
    results = [new_outs() for _ in streams]
    workspaces = [torch.empty(ws_size // 4, device="cuda") for _ in streams]
    for _ in range(3):
        for s, outs, ws in zip(streams, results, workspaces):
            with torch.cuda.stream(s):
                run_all(outs, ws)
    torch.cuda.synchronize()
    FW.fw_check_device_errors()
    for outs in results:
        for got, want in zip(outs, ref):
            assert torch.equal(got, want)
