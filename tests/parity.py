"""Shared helpers of the GPU parity tests (CUDA path through the C ABI vs the oracle)."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from oracle import oracle as O
from pooling_sliding_window_gb300 import fusedwin as FW
from pooling_sliding_window_gb300 import synth

# Tolerance of the FP32-FMA conv paths against the oracle (max abs error).
TOL_FFMA = 1e-5
# Tolerance of the plain-TF32 conv path (one TF32 product per multiply-add).
TOL_TF32 = 5e-3

POOL = ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1)))  # oracle calls release the GIL


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def bits_equal(a, b):
    """Bit-exact float32 equality, treating any two NaNs as equal."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    nan = np.isnan(a) & np.isnan(b)
    same = a.view(np.uint32) == b.view(np.uint32)
    return bool(np.all(same | nan)), int(np.sum(~(same | nan)))


def assert_bits_equal(a, b, what=""):
    ok, bad = bits_equal(a, b)
    assert ok, f"{what}: {bad} elements differ bitwise"


def assert_close(got, want, tol, what=""):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape, (got.shape, want.shape)
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    m = float(err.max()) if err.size else 0.0
    assert m <= tol, f"{what}: max abs err {m:.3e} > {tol:.1e} at {np.unravel_index(err.argmax(), err.shape)}"
    return m


def tf32_round(a):
    """Round float32 values to TF32 (10 explicit mantissa bits), to nearest with ties
    away from zero: add half of the dropped 13-bit field to the magnitude and clear
    it (finite inputs; a carry into the exponent is the correct rounding)."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    return ((u + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


# Canary guards: an output allocated inside a larger buffer whose head and tail hold a
# NaN bit pattern no kernel produces; after the call both must be untouched, so a
# kernel that writes past either end of its output fails the test that ran it.
GUARD = 4096                 # 32-bit words on each side (16 KB: keeps 256-byte alignment)
SENTINEL = 0x7FBADBAD        # a quiet-NaN payload


class Guarded:
    """An output tensor with sentinel words on both sides; `lead` more words in front
    shift its start (lead = 1: 4-byte but not 8-byte aligned)."""

    def __init__(self, shape, dtype=torch.float32, lead=0):
        n = int(np.prod(shape))
        words = n * (2 if dtype == torch.int64 else 1)
        self.buf = torch.full((words + 2 * GUARD + lead,), SENTINEL, dtype=torch.int32, device="cuda")
        self.out = self.buf[GUARD + lead:GUARD + lead + words].view(dtype).view(shape)

    def check(self, what=""):
        torch.cuda.synchronize()
        head, tail = self.buf[:GUARD], self.buf[-GUARD:]
        bad = int((head != SENTINEL).sum()) + int((tail != SENTINEL).sum())
        assert bad == 0, f"{what}: {bad} guard words around the output were overwritten"


def guarded_call(fn, shape, *args, lead=0, **kw):
    """Run fn(*args, out=<guarded tensor of `shape`>, **kw); check the guards; return the output on the host."""
    g = Guarded(shape, lead=lead)
    fn(*args, out=g.out, **kw)
    g.check(getattr(fn, "__name__", "call"))
    return host(g.out)


def pmap(fn, items):
    return list(POOL.map(fn, items))


def sample_indices(shape, count, seed):
    rng = np.random.default_rng(seed)
    return [tuple(int(rng.integers(0, s)) for s in shape) for _ in range(count)]


__all__ = ["O", "FW", "synth", "TOL_FFMA", "TOL_TF32", "tf32_round", "dev", "host", "assert_bits_equal", "assert_close", "pmap",
           "sample_indices", "bits_equal", "Guarded", "guarded_call"]
