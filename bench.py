"""Benchmark of the fused sliding-window hot path on GB300.

One step = one pass of the whole path, each operator on its full workload:
  conv+pool : x [128,8,256,256] -> Conv2d(8->64,k3) -> tanh -> *2 -> +bias -> MaxPool2d(4) -> [128,64,63,63]
  maxpool   : x [32,64,512,512] -> MaxPool2d(k4,s1,p1,d1) -> [32,64,511,511]
  convT     : x [128,64,64,64] -> ConvTranspose2d(64->128,k4,s2,p1,op1) -> softmax(1) -> +bias -> *2
              -> sigmoid -> [128,128,129,129]
all three enqueued on one CUDA stream through the C ABI (ctypes binding).

`value` is the fused conv+pool throughput in TFLOP/s (algorithmic FLOPs: the
conv outputs the pool consumes, 2*72 FLOP each); the maxpool's HBM GB/s and the
conv-transpose's TFLOP/s are reported beside it, each with its roofline
fraction.  Inputs are larger than L2 (268 MB, 2.15 GB, 134 MB), so no flush is
needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun every rank runs the full per-GPU workload (weak scaling, no data
exchange); rank 0 prints one JSON line with the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused conv+pool TFLOP/s & maxpool2d HBM GB/s, % of GB300 roofline"
UNIT = "TFLOP/s"

# Workloads
CP = dict(N=128, Cin=8, H=256, W=256, Cout=64, k=3, pool=4, scale=2.0)
MP = dict(N=32, C=64, H=512, W=512, k=4, s=1, p=1, d=1)
CT = dict(N=128, Cin=64, H=64, W=64, Cout=128, k=4, s=2, p=1, op=1, scale=2.0)


def cp_flops(N=CP["N"], Cout=CP["Cout"], Cin=CP["Cin"], ho=63, pool=4, k=3):
    """Algorithmic FLOPs of conv+pool: the conv outputs the pool windows consume."""
    return 2.0 * N * Cout * (pool * ho) ** 2 * Cin * k * k


def mp_bytes(N=MP["N"], C=MP["C"], H=512, W=512, ho=511, wo=511):
    return 4.0 * N * C * (H * W + ho * wo)


def ct_flops(N=CT["N"], Cin=CT["Cin"], Cout=CT["Cout"], H=64, W=64, k=4, s=2, p=1, op=1):
    """Algorithmic FLOPs of the conv-transpose: valid taps only (2 FLOP per MAC)."""
    Ho = (H - 1) * s - 2 * p + k - 1 + op + 1

    def taps(n_in, n_out):
        t = 0
        for i in range(n_in):
            for kk in range(k):
                o = i * s - p + kk
                t += 0 <= o < n_out
        return t

    return 2.0 * N * Cin * Cout * taps(H, Ho) * taps(W, Ho)


CP_FLOPS, MP_BYTES, CT_FLOPS = cp_flops(), mp_bytes(), ct_flops()
CT_BYTES = 4.0 * (CT["N"] * CT["Cin"] * 64 * 64 + CT["N"] * CT["Cout"] * 129 * 129)
CP_BYTES = 4.0 * (CP["N"] * CP["Cin"] * 256 * 256 + CP["N"] * CP["Cout"] * 63 * 63)


# ---------------------------------------------------------------- helpers --

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# Nominal dense tensor-core ratio TF32 : BF16 on GB300 (1.1 : 2.25 PFLOP/s).
TF32_PER_BF16 = 1.1 / 2.25


def peaks():
    """Roofline denominators: measured HBM copy GB/s and measured bf16 tensor TFLOP/s
    (the TF32 peak is the bf16 one times the nominal TF32:BF16 ratio)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    src = "measured"
    try:
        mp = json.load(open(path))
        hbm = float(mp["hbm_gbs"])
        bf16 = float(mp["bf16_tflops"])
        sm_max = float(mp.get("sm_max_mhz", 2070.0))
    except Exception:  # noqa: BLE001
        hbm, bf16, sm_max, src = 6800.0, 1900.0, 2070.0, "fallback"
    return dict(hbm_gbs=hbm, hbm_src=src, sm_max_mhz=sm_max, tf32_tflops=bf16 * TF32_PER_BF16)


def fp32_peak_tflops(sm_count, mhz):
    # 128 FP32 FMA lanes per SM, 2 FLOP per FMA.
    return sm_count * 128 * 2 * mhz * 1e6 / 1e12


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:  # noqa: BLE001
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def traffic_for(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's source
    is unchanged since that capture (else None)."""
    try:
        t = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
        ent = t[kernel_key]
        src = os.path.join(ROOT, "pooling_sliding_window_gb300", "csrc", ent["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if h != ent["source_sha"]:
            return None
        return float(ent["dram_bytes_per_launch"])
    except Exception:  # noqa: BLE001
        return None


# ------------------------------------------------------------------ inputs --

def make_inputs(seed=0, only=None):
    from pooling_sliding_window_gb300 import synth
    want = lambda n: only is None or only == n
    cp = synth.convpool_inputs(CP["N"], CP["Cin"], CP["H"], CP["W"], CP["Cout"], seed=seed) if want("convpool") else {}
    mp = synth.maxpool_inputs(MP["N"], MP["C"], MP["H"], MP["W"], seed=seed) if want("maxpool") else {}
    ct = synth.convt_inputs(CT["N"], CT["Cin"], CT["H"], CT["W"], CT["Cout"], seed=seed) if want("convt") else {}
    return cp, mp, ct


def reduce_max(values, ws, device=None):
    """Element-wise max of a list of floats over all ranks (identity when ws == 1)."""
    if ws == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def weak_value(units_per_rank, ws, ms):
    """Whole-job throughput: every rank processed `units_per_rank`; `ms` is the max over ranks."""
    return ws * units_per_rank / (ms * 1e-3)


# -------------------------------------------------------------- CPU oracle --

def oracle_sample(cp, mp, ct, budget_s=12.0):
    """Time the oracle (single-threaded C) on bounded samples of each workload.
    Returns per-op throughputs in the benchmark's units."""
    from oracle import oracle as O
    res = {}
    # conv+pool: whole images until ~budget/2 seconds
    t0 = time.perf_counter()
    n = 0
    while n < CP["N"] and (n == 0 or time.perf_counter() - t0 < budget_s / 2):
        O.conv2d_tanh_scale_bias_maxpool(cp["x"][n:n + 1], cp["w"], cp["conv_b"], CP["scale"], cp["bias"], 4)
        n += 1
    dt = time.perf_counter() - t0
    res["convpool"] = dict(tflops=cp_flops(N=n) / dt / 1e12, images=n, seconds=dt)
    # maxpool: whole planes for ~budget/4 seconds
    t0 = time.perf_counter()
    planes = 0
    while planes < MP["N"] * MP["C"] and (planes == 0 or time.perf_counter() - t0 < budget_s / 4):
        nn, c = divmod(planes, MP["C"])
        O.maxpool2d(mp["x"][nn:nn + 1, c:c + 1], 4, 1, 1, 1)
        planes += 1
    dt = time.perf_counter() - t0
    res["maxpool"] = dict(gbs=mp_bytes(N=1, C=planes) / dt / 1e9, planes=planes, seconds=dt)
    # conv-transpose: whole images for ~budget/4 seconds
    t0 = time.perf_counter()
    n = 0
    while n < CT["N"] and (n == 0 or time.perf_counter() - t0 < budget_s / 4):
        O.convtranspose2d_softmax_bias_scale_sigmoid(ct["x"][n:n + 1], ct["w"], ct["conv_b"], ct["bias"],
                                                     CT["scale"])
        n += 1
    dt = time.perf_counter() - t0
    res["convt"] = dict(tflops=ct_flops(N=n) / dt / 1e12, images=n, seconds=dt)
    return res


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # not Linux
        return os.cpu_count() or 1


def oracle_full_openmp(cp, mp, ct):
    """Time the oracle's OpenMP build (the same C source compiled with -fopenmp, its
    pragmas spreading images / channels / planes over the host cores) once on each
    full workload."""
    os.environ.setdefault("OMP_NUM_THREADS", str(host_cores()))
    from oracle import oracle as O
    try:
        O.lib(openmp=True)
    except Exception as e:  # noqa: BLE001
        return {"unavailable": f"OpenMP build of the oracle failed: {e}"}
    res = {"cores": int(os.environ["OMP_NUM_THREADS"]), "kind": "oracle, -fopenmp build of the same source",
           "sample": "full workloads, one call each"}
    t0 = time.perf_counter()
    O.conv2d_tanh_scale_bias_maxpool(cp["x"], cp["w"], cp["conv_b"], CP["scale"], cp["bias"], 4, openmp=True)
    dt = time.perf_counter() - t0
    res["convpool"] = {"seconds": dt, "tflops": CP_FLOPS / dt / 1e12}
    t0 = time.perf_counter()
    O.maxpool2d(mp["x"], 4, 1, 1, 1, openmp=True)
    dt = time.perf_counter() - t0
    res["maxpool"] = {"seconds": dt, "gbs": MP_BYTES / dt / 1e9}
    t0 = time.perf_counter()
    O.convtranspose2d_softmax_bias_scale_sigmoid(ct["x"], ct["w"], ct["conv_b"], ct["bias"], CT["scale"],
                                                 openmp=True)
    dt = time.perf_counter() - t0
    res["convt"] = {"seconds": dt, "tflops": CT_FLOPS / dt / 1e12}
    return res


def cpu_baseline_obj(res):
    cp, mpr, ctr = res["convpool"], res["maxpool"], res["convt"]
    return {"value": cp["tflops"], "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"conv+pool on {cp['images']} of 128 images ({cp['seconds']:.1f} s); "
                       f"maxpool on {mpr['planes']} of 2048 planes ({mpr['gbs']:.3f} GB/s); "
                       f"convT on {ctr['images']} of 128 images ({ctr['tflops'] * 1e3:.3f} GFLOP/s); "
                       "single-threaded C, float64 sums")}


# ------------------------------------------------- the tiny and sweep configs --

SWEEP = [(N, H, Cout, pool) for N in (1, 16, 128) for H in (127, 255, 256) for Cout in (16, 64) for pool in (2, 4)]
L2_BYTES = 129 * 2 ** 20


def time_configs(FW, dev, stream, tf32_peak):
    """The tiny conv+pool (x [2,8,64,64], launch-bound) and the conv+pool size sweep
    (N in {1,16,128} x H=W in {127,255,256} x Cout in {16,64} x pool in {2,4}, seed 0:
    the timing does not depend on the seed), each through the default C-ABI call,
    outside the timed step.  Inputs smaller than L2 are also timed with L2 flushed
    before every call (a 256 MB buffer written between calls, outside the events)."""
    import torch
    from oracle import oracle as O
    from pooling_sliding_window_gb300 import synth
    flush = torch.empty(256 * 2 ** 20 // 4, device=dev)

    def per_call(fn, reps, flush_l2=False):
        """Median device time of one call: the GPU is kept busy (a spin kernel) while
        the call is enqueued, so the events bracket the kernels and not the host's
        launch overhead."""
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            if flush_l2:
                flush.fill_(1.0)
            torch.cuda._sleep(200_000)  # ~0.1 ms of GPU time
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    def back_to_back(fn, reps):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / reps

    def inputs(N, H, Cout, x=None):
        bound = 1.0 / np.sqrt(72.0)
        if x is None:
            x = synth.normal((N, 8, H, H), 0, synth.TID_X)
        return dict(x=x, w=synth.uniform((Cout, 8, 3, 3), -bound, bound, 0, synth.TID_W),
                    conv_b=synth.uniform((Cout,), -bound, bound, 0, synth.TID_CONV_B),
                    bias=synth.normal((Cout,), 0, synth.TID_BIAS))

    res = {}
    # A: the tiny conv+pool
    a = synth.convpool_inputs(2, 8, 64, 64, 64, seed=0)
    t = {k: torch.from_numpy(v).to(dev) for k, v in a.items()}
    out = torch.empty(2, 64, 15, 15, device=dev)
    fn = lambda: FW.fw_conv2d_tanh_scale_bias_maxpool(t["x"], t["w"], t["conv_b"], t["bias"], 2.0, 4, out=out)
    warm, flushed, b2b = per_call(fn, 100), per_call(fn, 50, True), back_to_back(fn, 500)
    t0 = time.perf_counter()
    O.conv2d_tanh_scale_bias_maxpool(a["x"], a["w"], a["conv_b"], 2.0, a["bias"], 4)
    o_s = time.perf_counter() - t0
    n_out = 2 * 64 * 15 * 15
    res["A_tiny_convpool"] = {
        "workload": "x[2,8,64,64] Conv2d(8->64,k3)+tanh+*2+bias+MaxPool2d(4)->[2,64,15,15]",
        "us_warm": warm * 1e3, "us_l2_flushed": flushed * 1e3, "us_back_to_back": b2b * 1e3,
        "outputs_per_s_warm": n_out / (warm * 1e-3), "outputs_per_s_back_to_back": n_out / (b2b * 1e-3),
        "tflops_warm": cp_flops(N=2, ho=15) / (warm * 1e-3) / 1e12,
        "oracle_single_thread_s": o_s, "oracle_outputs_per_s": n_out / o_s,
        "note": "us_warm / us_l2_flushed: median device time of one call (events around the call, enqueued "
                "behind a GPU spin so that host launch overhead is excluded); us_back_to_back: 500 calls "
                "through the Python binding enqueued back to back, per call (bound by the host's call rate)"}
    # E: the size sweep
    rows, xs = [], {}
    for N, H, Cout, pool in SWEEP:
        if (N, H) not in xs:
            xs = {(N, H): synth.normal((N, 8, H, H), 0, synth.TID_X)}
        d = inputs(N, H, Cout, xs[(N, H)])
        Ho, Wo = FW.fw_conv2d_pool_out_shape(H, H, 3, 3, pool, pool)
        t = {k: torch.from_numpy(v).to(dev) for k, v in d.items()}
        out = torch.empty(N, Cout, Ho, Wo, device=dev)
        fn = lambda: FW.fw_conv2d_tanh_scale_bias_maxpool(t["x"], t["w"], t["conv_b"], t["bias"], 2.0, pool,
                                                          out=out)
        ms = per_call(fn, 20 if N < 128 else 10)
        flops = 2.0 * 72 * N * Cout * (pool * Ho) * (pool * Wo)
        row = {"N": N, "H": H, "Cout": Cout, "pool": pool, "out": [N, Cout, Ho, Wo], "ms": ms,
               "tflops": flops / (ms * 1e-3) / 1e12, "tensor_frac": flops / (ms * 1e-3) / 1e12 / tf32_peak}
        if 4 * (d["x"].size + N * Cout * Ho * Wo) < L2_BYTES:
            row["us_l2_flushed"] = per_call(fn, 20, True) * 1e3
            row["us_warm"] = ms * 1e3
        rows.append(row)
        del t, out
    res["E_sweep"] = {"rows": rows, "shapes": len(rows),
                      "note": "per shape: median device time of one call (ms), algorithmic TFLOP/s (2*72 FLOP per "
                              "conv output the pool reads), fraction of dense TF32; inputs that fit in L2 also "
                              "with L2 flushed; seed 0 only (parity covers seeds 0-2)"}
    del flush
    return res


# ---------------------------------------------------------------- reference --

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    cp, mp, ct = make_inputs()
    for _ in range(args.warmup):
        oracle_sample(cp, mp, ct, budget_s=2.0)
    vals, steps = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = oracle_sample(cp, mp, ct, budget_s=8.0)
        steps.append(r)
        vals.append(r["convpool"]["tflops"])
    wall = time.perf_counter() - t0
    v = statistics.median(vals)
    cpu = cpu_baseline_obj(steps[-1])
    cpu["value"] = v
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall * 1e3 / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 sums, f32 stages",
            "data": "synthetic (seeded SplitMix64 / Box-Muller, the pages' shapes)",
            "config": config_obj(), "cpu_baseline": cpu,
            "maxpool_hbm_gbs": statistics.median(s["maxpool"]["gbs"] for s in steps),
            "convt_tflops": statistics.median(s["convt"]["tflops"] for s in steps),
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_obj():
    return {"workload": ("conv+pool x[128,8,256,256] Conv2d(8->64,k3)+tanh+*2+bias+MaxPool2d(4)->[128,64,63,63]; "
                         "maxpool x[32,64,512,512] MaxPool2d(k4,s1,p1,d1)->[32,64,511,511]; "
                         "convT x[128,64,64,64] ConvTranspose2d(64->128,k4,s2,p1,op1)+softmax(1)+bias+*2+sigmoid"
                         "->[128,128,129,129]"),
            "seed": 0, "l2": "inputs larger than L2 (268 MB, 2.15 GB, 134 MB); no flush",
            "precision": ("fp32 in/out; conv+pool on tensor cores with a 3xTF32 split (within 1e-5 of the "
                          "float64 oracle); convT on TF32 tensor cores (the TF32 path's 5e-3 bound; within 1e-5 "
                          "on this workload's near-flat softmax, a few 1e-4 on sharp logits); maxpool exact"),
            "parallelism": "weak scaling over GPUs, no collective"}


# ---------------------------------------------------------------- GPU arm --

def run_gpu(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl" if args.backend == "nccl" else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from pooling_sliding_window_gb300 import fusedwin as FW

    cp, mp, ct = make_inputs(seed=0, only=args.only)
    if args.batch:  # a smaller batch of every workload (profiling cases)
        cp = {k: (v[:args.batch] if k == "x" else v) for k, v in cp.items()}
        mp = {k: (v[:max(1, args.batch // 4)] if k == "x" else v) for k, v in mp.items()}
        ct = {k: (v[:args.batch] if k == "x" else v) for k, v in ct.items()}
    pinned = {(name, k): torch.from_numpy(np.ascontiguousarray(v)).pin_memory()
              for name, dct in (("cp", cp), ("mp", mp), ("ct", ct)) for k, v in dct.items()}
    d = {key: t.to(dev) for key, t in pinned.items()}
    stream = torch.cuda.current_stream(dev)

    specs = []  # (name, units per rank, device op, host op, out shape)
    if cp:
        n = cp["x"].shape[0]
        out_cp = torch.empty(n, CP["Cout"], 63, 63, device=dev)
        h_cp = torch.empty(tuple(out_cp.shape), pin_memory=True)

        cp_fn = (FW.fw_conv2d_tanh_scale_bias_maxpool_tf32 if args.convpool_precision == "tf32"
                 else FW.fw_conv2d_tanh_scale_bias_maxpool)  # tf32: profiling the plain-TF32 variant

        if args.convpool_layout == "nhwc":  # profiling the channels-last variant through the same step
            cp_x_nhwc = d[("cp", "x")].permute(0, 2, 3, 1).contiguous()
            cp_out_nhwc = torch.empty(n, 63, 63, CP["Cout"], device=dev)

        def op_cp(src, out):
            if args.convpool_layout == "nhwc" and src is d:
                FW.fw_conv2d_tanh_scale_bias_maxpool_nhwc(cp_x_nhwc, src[("cp", "w")], src[("cp", "conv_b")],
                                                          src[("cp", "bias")], CP["scale"], 4, out=cp_out_nhwc)
                return
            cp_fn(src[("cp", "x")], src[("cp", "w")], src[("cp", "conv_b")], src[("cp", "bias")], CP["scale"], 4,
                  out=out)
        hws_cp = torch.empty(FW.lib().fw_conv2d_tanh_scale_bias_maxpool_host_workspace_size(
            n, CP["Cin"], CP["H"], CP["W"], CP["Cout"], 3, 3, 4, 4) // 4 + 64, device=dev)

        def host_cp():  # C-ABI host-buffer call: pipelined H2D copies, kernels, D2H copies
            FW.fw_conv2d_tanh_scale_bias_maxpool_host(pinned[("cp", "x")], pinned[("cp", "w")],
                                                      pinned[("cp", "conv_b")], pinned[("cp", "bias")], CP["scale"],
                                                      4, out=h_cp, workspace=hws_cp)
        specs.append(dict(name="convpool", work=cp_flops(N=n), unit="TFLOP/s", scale=1e12, bound="tensor",
                          run=lambda: op_cp(d, out_cp), e2e=lambda: host_cp(), out=h_cp,
                          kernel=("convpool_tc_kernel<4,64,false,false> (tcgen05 kind::tf32, one TF32 product per "
                                  "MAC, kh taps stacked along N, two epilogue groups)" if args.convpool_precision == "tf32"
                                  else "convpool_tc_kernel<4,64,false,true> (tcgen05 kind::tf32, 3xTF32 split as two "
                                       "MMAs per tap, N = 128 [w_hi|w_lo] and N = 64: executed tensor FLOPs = 3 x "
                                       "algorithmic)"), source="convpool_tc.cu"))
    if mp:
        n = mp["x"].shape[0]
        out_mp = torch.empty(n, MP["C"], 511, 511, device=dev)
        h_mp = torch.empty(tuple(out_mp.shape), pin_memory=True)

        if args.maxpool_layout == "nhwc":  # profiling the channels-last variant through the same step
            mp_x_nhwc = d[("mp", "x")].permute(0, 2, 3, 1).contiguous()
            mp_out_nhwc = torch.empty(n, 511, 511, MP["C"], device=dev)

        def op_mp(src, out):
            if args.maxpool_layout == "nhwc" and src is d:
                FW.fw_maxpool2d_nhwc(mp_x_nhwc, 4, 1, 1, 1, out=mp_out_nhwc)
                return
            FW.fw_maxpool2d(src[("mp", "x")], 4, 1, 1, 1, out=out)
        hws_mp = torch.empty(FW.lib().fw_maxpool2d_host_workspace_size(n, MP["C"], MP["H"], MP["W"], 4, 1, 1, 1)
                             // 4 + 64, device=dev)

        def host_mp():
            FW.fw_maxpool2d_host(pinned[("mp", "x")], 4, 1, 1, 1, out=h_mp, workspace=hws_mp)
        specs.append(dict(name="maxpool", work=mp_bytes(N=n), unit="GB/s", scale=1e9, bound="hbm",
                          run=lambda: op_mp(d, out_mp), e2e=lambda: host_mp(), out=h_mp,
                          kernel="maxpool_s1_stream_kernel<4,1>", source="maxpool.cu"))
    if ct:
        n = ct["x"].shape[0]
        out_ct = torch.empty(n, CT["Cout"], 129, 129, device=dev)
        h_ct = torch.empty(tuple(out_ct.shape), pin_memory=True)
        wsz = FW.fw_convt_workspace_size(CT["Cin"], CT["Cout"], 4, 2, 1)
        wsp = torch.empty(max(1, wsz // 4), device=dev)

        if args.convt_layout == "nhwc":  # profiling the channels-last variant through the same step
            x_nhwc = d[("ct", "x")].permute(0, 2, 3, 1).contiguous()
            out_nhwc = torch.empty(n, 129, 129, CT["Cout"], device=dev)

        def op_ct(src, out):
            if args.convt_layout == "nhwc" and src is d:
                FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc(x_nhwc, src[("ct", "w")], src[("ct", "conv_b")],
                                                                      src[("ct", "bias")], CT["scale"], out=out_nhwc,
                                                                      workspace=wsp)
                return
            FW.fw_convtranspose2d_softmax_bias_scale_sigmoid(src[("ct", "x")], src[("ct", "w")],
                                                             src[("ct", "conv_b")], src[("ct", "bias")],
                                                             CT["scale"], out=out, workspace=wsp)
        hws_ct = torch.empty(FW.lib().fw_convtranspose2d_softmax_bias_scale_sigmoid_host_workspace_size(
            n, CT["Cin"], CT["H"], CT["W"], CT["Cout"], 4, 2, 1, 1) // 4 + 64, device=dev)

        def host_ct():
            FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_host(
                pinned[("ct", "x")], pinned[("ct", "w")], pinned[("ct", "conv_b")], pinned[("ct", "bias")],
                CT["scale"], out=h_ct, workspace=hws_ct)
        specs.append(dict(name="convt", work=ct_flops(N=n), unit="TFLOP/s", scale=1e12, bound="tensor",
                          run=lambda: op_ct(d, out_ct), e2e=lambda: host_ct(), out=h_ct,
                          kernel="convt_k4s2_pair_kernel<16> (CTA pairs, tcgen05.mma.cta_group::2 kind::tf32, both column phases per pair) + weight prepack",
                          source="convt_tc.cu"))

    def barrier():
        if ws > 1:
            dist.barrier()

    for _ in range(args.warmup):
        for sp in specs:
            sp["run"]()
    torch.cuda.synchronize()
    FW.fw_check_device_errors()

    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in specs]
          for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    launches0 = FW.fw_launch_count()
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        t_start.record(stream)
        for i in range(args.steps):
            for j, sp in enumerate(specs):
                ev[i][j][0].record(stream)
                sp["run"]()
                ev[i][j][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier()
    launches = FW.fw_launch_count() - launches0
    FW.fw_check_device_errors()
    local_ms = [t_start.elapsed_time(t_end)] + [
        statistics.mean(ev[i][j][0].elapsed_time(ev[i][j][1]) for i in range(args.steps)) for j in range(len(specs))]

    # End to end through the public API: pinned host tensors in, H2D + kernels + D2H per op.
    for sp in specs:
        sp["e2e"]()
    torch.cuda.synchronize()
    barrier()
    e2e_steps = max(3, min(args.steps, 7))
    e2e_local, e2e_range = [], {}
    for sp in specs:
        ts = []
        for _ in range(e2e_steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            sp["e2e"]()  # returns once the result is in host memory
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        e2e_local.append(statistics.median(ts))
        e2e_range[sp["name"]] = [min(ts), max(ts)]
    # What fusion saves: the same operators the pages' unfused way (conv output to memory,
    # then a second kernel), built from this library's kernels; outside the timed step.
    fusion = None
    if not args.no_fusion_compare and (cp or ct or mp):
        fusion = {}

        def med_ms(fn, reps=7):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            ts = []
            for _ in range(reps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                b.synchronize()
                ts.append(a.elapsed_time(b))
            return statistics.median(ts)

        if cp:
            n = cp["x"].shape[0]
            wsz = FW.fw_conv2d_pool_unfused_workspace_size(n, CP["H"], CP["W"], CP["Cout"], 3, 3, 4)
            wsp_cp = torch.empty(wsz // 4, device=dev)
            f_ms = med_ms(lambda: op_cp(d, out_cp))
            u_ms = med_ms(lambda: FW.fw_conv2d_tanh_scale_bias_maxpool_unfused(
                d[("cp", "x")], d[("cp", "w")], d[("cp", "conv_b")], d[("cp", "bias")], CP["scale"], 4,
                out=out_cp, workspace=wsp_cp))
            fusion["convpool"] = {"fused_ms": f_ms, "unfused_ms": u_ms, "unfused_over_fused": u_ms / f_ms,
                                  "intermediate_bytes": wsz,
                                  "unfused": "convpool_tc_kernel raw mode (conv + conv_b to memory) + "
                                             "pool_tanh_scale_bias_kernel"}
            del wsp_cp
            # plain-TF32 variant of the fused operator (one TF32 product per multiply-add, 5e-3 bound)
            out_tf = torch.empty_like(out_cp)
            tf_ms = med_ms(lambda: FW.fw_conv2d_tanh_scale_bias_maxpool_tf32(
                d[("cp", "x")], d[("cp", "w")], d[("cp", "conv_b")], d[("cp", "bias")], CP["scale"], 4, out=out_tf))
            fusion["convpool_tf32"] = {"ms": tf_ms, "x3_ms": f_ms, "work_per_launch": cp_flops(N=n),
                                       "kernel": "convpool_tc_kernel<4,64,false,false>: one TF32 product per MAC "
                                                 "(kh taps stacked along N: 21 MMAs of N = 64..192 per item), two "
                                                 "epilogue groups",
                                       "max_abs_diff_vs_x3": float((out_tf - out_cp).abs().max())}
            del out_tf
            # the same operator on the float32 FMA pipe only (no tensor cores)
            out_ff = torch.empty_like(out_cp)
            ff_ms = med_ms(lambda: FW.fw_conv2d_tanh_scale_bias_maxpool_ffma(
                d[("cp", "x")], d[("cp", "w")], d[("cp", "conv_b")], d[("cp", "bias")], CP["scale"], 4, out=out_ff))
            fusion["convpool_ffma"] = {"ms": ff_ms, "work_per_launch": cp_flops(N=n),
                                       "kernel": "convpool3x3_ffma_kernel<4>: persistent FP32-FMA implicit GEMM, "
                                                 "4x4 conv pixels x 4 channels per thread, cp.async staging",
                                       "max_abs_diff_vs_x3": float((out_ff - out_cp).abs().max())}
            del out_ff
            # channels-last variant (x [N,H,W,8] -> out [N,Ho,Wo,Cout]), the same 3xTF32 arithmetic
            xn = d[("cp", "x")].permute(0, 2, 3, 1).contiguous()
            on = torch.empty(n, out_cp.shape[2], out_cp.shape[3], CP["Cout"], device=dev)
            nhwc_ms = med_ms(lambda: FW.fw_conv2d_tanh_scale_bias_maxpool_nhwc(
                xn, d[("cp", "w")], d[("cp", "conv_b")], d[("cp", "bias")], CP["scale"], 4, out=on))
            fusion["convpool_channels_last"] = {
                "nchw_ms": f_ms, "nhwc_ms": nhwc_ms, "nhwc_tflops": cp_flops(N=n) / (nhwc_ms * 1e-3) / 1e12,
                "equal_to_nchw": bool(torch.equal(on, out_cp.permute(0, 2, 3, 1))),
                "kernel": "convpool_tc_kernel<4,64,false,true,true>: a position's 8 channels as two 16-byte "
                          "loads (core-matrix rows as they stand), 32 contiguous bytes per pooled pixel stored"}
            del xn, on
        if ct:
            n = ct["x"].shape[0]
            wsz = FW.fw_convt_unfused_workspace_size(n, CT["Cin"], CT["H"], CT["W"], CT["Cout"], 4, 2, 1, 1)
            wsp_ct = torch.empty(wsz // 4, device=dev)
            f_ms = med_ms(lambda: op_ct(d, out_ct))
            u_ms = med_ms(lambda: FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_unfused(
                d[("ct", "x")], d[("ct", "w")], d[("ct", "conv_b")], d[("ct", "bias")], CT["scale"],
                out=out_ct, workspace=wsp_ct))
            fusion["convt"] = {"fused_ms": f_ms, "unfused_ms": u_ms, "unfused_over_fused": u_ms / f_ms,
                               "intermediate_bytes": 4 * n * CT["Cout"] * 129 * 129,
                               "unfused": "convt_k4s2_tc_kernel raw mode (conv-transpose + conv_b to memory) + "
                                          "softmax_bias_scale_sigmoid_kernel (online max/sum pass, output pass)"}
            del wsp_ct
            # the same operator on the float32 FMA pipe only (no tensor cores)
            out_ff = torch.empty_like(out_ct)
            ff_ms = med_ms(lambda: FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_ffma(
                d[("ct", "x")], d[("ct", "w")], d[("ct", "conv_b")], d[("ct", "bias")], CT["scale"], out=out_ff,
                workspace=wsp))
            fusion["convt_ffma"] = {"ms": ff_ms, "work_per_launch": ct_flops(N=n),
                                    "kernel": "convt_k4s2_ffma_kernel: per phase, 8 x 16 phase pixels x 128 channels "
                                              "per CTA, 8 x 8 outputs per thread, shuffle softmax",
                                    "max_abs_diff_vs_tf32": float((out_ff - out_ct).abs().max())}
            del out_ff
            # channels-last variant of the same model (x [N,H,W,Cin] -> out [N,Ho,Wo,Cout])
            xn = d[("ct", "x")].permute(0, 2, 3, 1).contiguous()
            on = torch.empty(n, 129, 129, CT["Cout"], device=dev)
            nhwc_ms = med_ms(lambda: FW.fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc(
                xn, d[("ct", "w")], d[("ct", "conv_b")], d[("ct", "bias")], CT["scale"], out=on, workspace=wsp))
            fusion["convt_channels_last"] = {"nchw_ms": f_ms, "nhwc_ms": nhwc_ms,
                                             "kernel": "convt_k4s2_pair_kernel<16,true>: CTA pairs, 16-byte channel "
                                                       "gathers, 256-bit output stores"}
            del xn, on
        if mp:
            # channels-last maxpool of the same workload (x [N,H,W,C] -> out [N,Ho,Wo,C])
            n = mp["x"].shape[0]
            xn = d[("mp", "x")].permute(0, 2, 3, 1).contiguous()
            on = torch.empty(n, 511, 511, MP["C"], device=dev)
            f_ms = med_ms(lambda: op_mp(d, out_mp))
            nhwc_ms = med_ms(lambda: FW.fw_maxpool2d_nhwc(xn, 4, 1, 1, 1, out=on))
            fusion["maxpool_channels_last"] = {
                "nchw_ms": f_ms, "nhwc_ms": nhwc_ms, "nhwc_gbs": mp_bytes(N=n) / (nhwc_ms * 1e-3) / 1e9,
                "nhwc_frac_of_hbm": mp_bytes(N=n) / (nhwc_ms * 1e-3) / 1e9 / peaks()["hbm_gbs"],
                "kernel": "maxpool_nhwc_s1_kernel<4>: the block's input columns (all channels) stream into shared "
                          "memory by one bulk copy per row, ~24 KB stages; 4 channels of one output column per thread, "
                          "row maxima in a 4-deep register ring over a band of 64 output rows"}
            del xn, on
        FW.fw_check_device_errors()
    configs = None
    if not args.no_configs and args.only is None and not args.batch and rank == 0:
        configs = time_configs(FW, dev, stream, peaks()["tf32_tflops"])
    red = reduce_max(local_ms + e2e_local, ws, device=dev if args.backend == "nccl" else None)
    total_ms, op_ms, e2e_ms = red[0], red[1:1 + len(specs)], red[1 + len(specs):]
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = sum(sp["out"].numel() * 4 for sp in specs)

    if rank != 0:
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    pk = peaks()
    props = torch.cuda.get_device_properties(dev)
    fp32_peak = fp32_peak_tflops(props.multi_processor_count, pk["sm_max_mhz"])
    ops = {}
    for sp, ms in zip(specs, op_ms):
        ach = sp["work"] / (ms * 1e-3) / sp["scale"]
        peak = {"alu": fp32_peak, "tensor": pk["tf32_tflops"], "hbm": pk["hbm_gbs"]}[sp["bound"]]
        ops[sp["name"]] = dict(ms=ms, achieved=ach, unit=sp["unit"], bound=sp["bound"], peak=peak,
                               frac=ach / peak, work_per_launch=sp["work"], kernel=sp["kernel"])
    dom_i = max(range(len(specs)), key=lambda j: op_ms[j])
    dom = specs[dom_i]
    dv = ops[dom["name"]]
    roofline = {"bound": dv["bound"], "achieved": dv["achieved"], "peak": dv["peak"], "unit": dv["unit"],
                "frac": dv["frac"], "traffic": traffic_for(dom["name"]), "kernel": dv["kernel"],
                "peak_source": {
                    "alu": "FP32 FMA pipe: SMs x 128 lanes x 2 FLOP x max SM clock "
                           f"({props.multi_processor_count} x 128 x 2 x {pk['sm_max_mhz']:.0f} MHz)",
                    "tensor": f"dense TF32 = measured bf16 burst x {TF32_PER_BF16:.4f} (nominal 1.1/2.25), "
                              f"{pk['hbm_src']} (MEASURED_PEAKS.json)",
                    "hbm": f"HBM copy GB/s, {pk['hbm_src']} (MEASURED_PEAKS.json)"}[dv["bound"]]}
    by = {sp["name"]: (sp, ms, ems) for sp, ms, ems in zip(specs, op_ms, e2e_ms)}
    head = "convpool" if "convpool" in by else specs[0]["name"]
    hs, hms, hems = by[head]
    cpu = None
    if not args.no_cpu_baseline and args.only is None and not args.batch:
        cpu = cpu_baseline_obj(oracle_sample(cp, mp, ct, budget_s=args.cpu_budget))
        if not args.no_oracle_full:
            cpu["full_size_openmp"] = oracle_full_openmp(cp, mp, ct)
    line = {
        "metric": METRIC, "value": weak_value(hs["work"], ws, hms) / hs["scale"], "unit": hs["unit"],
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "tf32+f32",
        "data": "synthetic (seeded SplitMix64 / Box-Muller, the pages' shapes)", "config": config_obj(),
    }
    if "maxpool" in by:
        sp, ms, _ = by["maxpool"]
        line["maxpool_hbm_gbs"] = weak_value(sp["work"], ws, ms) / 1e9
        line["maxpool_hbm_frac"] = ops["maxpool"]["frac"]
    if "convpool" in by:
        line["convpool_tensor_frac"] = ops["convpool"]["frac"]
    if "convt" in by:
        sp, ms, _ = by["convt"]
        line["convt_tflops"] = weak_value(sp["work"], ws, ms) / 1e12
    line.update({
        "ops": ops, "roofline": roofline, "cpu_baseline": cpu,
        "e2e": {"value": weak_value(hs["work"], ws, hems) / hs["scale"], "unit": hs["unit"],
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ops_ms": {sp["name"]: e for sp, e in zip(specs, e2e_ms)},
                "ops_ms_range": e2e_range, "calls_per_op": e2e_steps,
                "note": "C-ABI host-buffer calls (fw_*_host) on pinned host tensors: per op, chunked H2D copies, "
                        "kernels and D2H copies pipelined on copy streams; timed until the result is in host memory; "
                        "median of the calls (ops_ms), with min and max (ops_ms_range), rank 0's range"},
        "gpu_launches": launches, "launches_per_step": launches / args.steps,
        "clocks": clk.summary(), "device": props.name,
    })
    if configs:
        line["configs"] = configs
    if fusion:
        if "convpool_tf32" in fusion:
            v = fusion["convpool_tf32"]
            v["tflops"] = v["work_per_launch"] / (v["ms"] * 1e-3) / 1e12
            v["frac_of_tf32_peak"] = v["tflops"] / pk["tf32_tflops"]
            line["convpool_tf32_tflops"] = v["tflops"]  # the plain-TF32 call, timed beside the step
            line["convpool_tf32_tensor_frac"] = v["frac_of_tf32_peak"]
        if "convpool_ffma" in fusion:
            v = fusion["convpool_ffma"]
            v["tflops"] = v["work_per_launch"] / (v["ms"] * 1e-3) / 1e12
            v["frac_of_fp32_peak"] = v["tflops"] / fp32_peak
            line["convpool_ffma_tflops"] = v["tflops"]  # the FP32-FMA call, timed beside the step
            line["convpool_ffma_fp32_frac"] = v["frac_of_fp32_peak"]
        if "convt_ffma" in fusion:
            v = fusion["convt_ffma"]
            v["tflops"] = v["work_per_launch"] / (v["ms"] * 1e-3) / 1e12
            v["frac_of_fp32_peak"] = v["tflops"] / fp32_peak
        line["fusion"] = fusion
    if (args.only or args.batch or args.convt_layout != "nchw" or args.convpool_precision != "x3" or
            args.convpool_layout != "nchw" or args.maxpool_layout != "nchw"):
        line["config"]["subset"] = {"only": args.only, "batch": args.batch, "convt_layout": args.convt_layout,
                                    "convpool_precision": args.convpool_precision,
                                    "convpool_layout": args.convpool_layout, "maxpool_layout": args.maxpool_layout}
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=16.0)
    ap.add_argument("--backend", default="nccl", choices=["nccl", "gloo"])
    ap.add_argument("--only", default=None, choices=["convpool", "maxpool", "convt"],
                    help="time one operator only (profiling)")
    ap.add_argument("--batch", type=int, default=0, help="smaller batch for every workload (profiling)")
    ap.add_argument("--convt-layout", default="nchw", choices=["nchw", "nhwc"],
                    help="layout of the conv-transpose in the timed step (nhwc: channels-last variant, profiling)")
    ap.add_argument("--maxpool-layout", default="nchw", choices=["nchw", "nhwc"],
                    help="layout of the maxpool in the timed step (nhwc: channels-last variant, profiling)")
    ap.add_argument("--convpool-layout", default="nchw", choices=["nchw", "nhwc"],
                    help="layout of the conv+pool in the timed step (nhwc: channels-last variant, profiling)")
    ap.add_argument("--convpool-precision", default="x3", choices=["x3", "tf32"],
                    help="conv+pool in the timed step: 3xTF32 split (x3) or plain TF32 (profiling)")
    ap.add_argument("--no-fusion-compare", action="store_true",
                    help="skip timing the unfused (conv output to memory) comparison path")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the tiny conv+pool and the conv+pool size sweep")
    ap.add_argument("--no-oracle-full", action="store_true",
                    help="skip timing the oracle's OpenMP build on the full workloads")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl != "reference":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
