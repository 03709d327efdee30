"""Seeded synthetic inputs shared by the CUDA path's tests/bench and by the oracle.

This module only draws random numbers.  It holds none of the arithmetic of the
operators (no convolution, pooling, softmax ...), so both sides can take their
inputs from it without sharing any of the method.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style: element ``i`` of tensor
``tid`` under seed ``seed`` is ``mix(base(seed, tid) + (i + 1) * GAMMA)``.
Uniforms take the top 24 bits of a word; normals use the Box-Muller transform
in float64 and are rounded to float32.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

# Tensor ids: each named input of a problem gets its own stream.
TID_X, TID_W, TID_CONV_B, TID_BIAS = 1, 2, 3, 4


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _base(seed: int, tid: int) -> np.uint64:
    s = np.array([(seed * 0x100000001B3 + tid * 0xD1B54A32D192ED03 + 1) & 0xFFFFFFFFFFFFFFFF],
                 dtype=np.uint64)
    return _mix(s)[0]


def _words(base: np.uint64, start: int, count: int) -> np.ndarray:
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + idx * GAMMA)


def _parallel(n: int, fill) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    chunks = [(a, min(n, a + _CHUNK)) for a in range(0, n, _CHUNK)]
    if len(chunks) <= 2:
        for a, b in chunks:
            fill(out, a, b)
    else:
        workers = min(len(chunks), os.cpu_count() or 1, 32)
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(lambda ab: fill(out, *ab), chunks))
    return out


def uniform(shape, lo: float, hi: float, seed: int, tid: int) -> np.ndarray:
    """float32 array of ``shape`` drawn from U[lo, hi)."""
    n = int(np.prod(shape)) if len(shape) else 1
    base = _base(seed, tid)

    def fill(out, a, b):
        u = (_words(base, a, b - a) >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
        out[a:b] = (lo + (hi - lo) * u).astype(np.float32)

    return _parallel(n, fill).reshape(shape)


def normal(shape, seed: int, tid: int) -> np.ndarray:
    """float32 array of ``shape`` drawn from N(0, 1) (Box-Muller on word pairs)."""
    n = int(np.prod(shape)) if len(shape) else 1
    base = _base(seed, tid)

    def fill(out, a, b):
        # Chunk starts are even, so pairs never straddle two chunks.
        pa, pb = a // 2, (b + 1) // 2
        w = _words(base, 2 * pa, 2 * (pb - pa))
        u1 = ((w[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u2 = (w[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * np.pi * u2
        z = np.empty(2 * (pb - pa), dtype=np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        out[a:b] = z[: b - a].astype(np.float32)

    return _parallel(n, fill).reshape(shape)


# ---------------------------------------------------------------------------
# Problem recipes (shapes and distributions of the three workloads)
# ---------------------------------------------------------------------------

def convpool_inputs(N, Cin, H, W, Cout, k=3, seed=0):
    """Inputs of the fused conv3x3+tanh+scale+bias+maxpool problem.

    x ~ N(0,1); conv weight and conv bias ~ U(+-1/sqrt(Cin*k*k)) (the default
    nn.Conv2d initialisation bound); extra bias [Cout] ~ N(0,1).
    """
    bound = 1.0 / np.sqrt(Cin * k * k)
    return dict(
        x=normal((N, Cin, H, W), seed, TID_X),
        w=uniform((Cout, Cin, k, k), -bound, bound, seed, TID_W),
        conv_b=uniform((Cout,), -bound, bound, seed, TID_CONV_B),
        bias=normal((Cout,), seed, TID_BIAS),
    )


def maxpool_inputs(N, C, H, W, seed=0):
    """Input of the MaxPool2d problem: x ~ N(0,1)."""
    return dict(x=normal((N, C, H, W), seed, TID_X))


def convt_inputs(N, Cin, H, W, Cout, k=4, seed=0):
    """Inputs of the ConvTranspose2d+softmax+bias+scale+sigmoid problem.

    x ~ N(0,1); weight [Cin, Cout, k, k] and conv bias ~ U(+-1/sqrt(Cin*k*k))
    (for the 64->128, k=4 workload: +-1/sqrt(1024)); extra bias [Cout] ~ N(0,1).
    """
    bound = 1.0 / np.sqrt(Cin * k * k)
    return dict(
        x=normal((N, Cin, H, W), seed, TID_X),
        w=uniform((Cin, Cout, k, k), -bound, bound, seed, TID_W),
        conv_b=uniform((Cout,), -bound, bound, seed, TID_CONV_B),
        bias=normal((Cout,), seed, TID_BIAS),
    )
