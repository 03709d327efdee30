"""Host logic of bench.py that needs no GPU: algorithmic work counts, the
max-over-ranks reduction and the weak-scaling value with 2 gloo ranks on CPU,
and the reference arm's non-zero ranks exiting without work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_work_counts():
    assert bench.CP_FLOPS == 2 * 128 * 64 * 252 * 252 * 72          # 74.91 GFLOP
    assert abs(bench.CP_FLOPS / 1e9 - 74.91) < 0.01
    assert bench.MP_BYTES == 4 * 32 * 64 * (512 * 512 + 511 * 511)  # 4.2866 GB
    # valid conv-transpose taps along one axis: 64 inputs x 4 taps minus the one
    # that falls at output row -1
    assert bench.CT_FLOPS == 2 * 128 * 64 * 128 * 255 * 255          # 136.37 GFLOP
    assert abs(bench.CT_FLOPS / 1e9 - 136.37) < 0.01


def test_sweep_covers_the_sweep_config():
    """The timed sweep is the conv+pool edge/size sweep's 36 shapes (each run there
    with seeds 0-2: 108 runs)."""
    assert len(bench.SWEEP) == 36 and len(set(bench.SWEEP)) == 36
    assert {s[0] for s in bench.SWEEP} == {1, 16, 128}
    assert {s[1] for s in bench.SWEEP} == {127, 255, 256}
    assert {s[2] for s in bench.SWEEP} == {16, 64}
    assert {s[3] for s in bench.SWEEP} == {2, 4}
    assert bench.cp_flops(N=2, ho=15) == 2 * 72 * 2 * 64 * 60 * 60  # the tiny config


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    vals = bench.reduce_max([10.0 + rank, 5.0 - rank, 2.5], ws)
    v = bench.weak_value(1e9, ws, vals[0])
    q.put((rank, vals, v))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, vals, v in res:
        assert vals == [11.0, 5.0, 2.5]
        assert v == pytest.approx(2 * 1e9 / 11e-3)


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    called = []
    monkeypatch.setattr(bench, "make_inputs", lambda *a, **k: called.append(1))
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert not called
