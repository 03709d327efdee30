"""Pins of the oracle to facts fixed outside itself.

Each test ties an oracle function to something it does not compute itself:
sizes and tables printed on the pages (tests/golden), library routines that a
special case reduces to (torch.nn.functional in float64), closed forms, brute
force written another way, invariants, and the adjoint identity between the
two linear stages.  No test here needs a GPU.
"""
import math
import os
import re

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as O
from pooling_sliding_window_gb300 import synth

RNG = np.random.default_rng(1234)


def rnd(*shape, lo=-1.0, hi=1.0):
    return RNG.uniform(lo, hi, size=shape).astype(np.float32)


def t64(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


# --------------------------------------------------------------- golden ----

def _golden_sizes(golden_dir):
    rows = []
    for line in open(os.path.join(golden_dir, "output_sizes.txt")):
        line = line.split("|")[0].strip()
        if not line or line.startswith("#"):
            continue
        lhs, rhs = line.split("->")
        rows.append((lhs.split(), int(rhs)))
    return rows


def test_golden_output_sizes(golden_dir):
    rows = _golden_sizes(golden_dir)
    assert len(rows) == 7
    for args, want in rows:
        op, a = args[0], args[1:]
        if op == "conv2d":
            got = O.conv2d_out_size(*map(int, a))
        elif op == "maxpool":
            got = O.pool_out_size(*map(int, a))
        elif op == "convt":
            got = O.convt_out_size(*map(int, a))
        elif op == "count":
            name = a[0]
            if name == "conv_outputs_p82":
                hc = O.conv2d_out_size(256, 3)
                got = 128 * 64 * hc * hc
            elif name == "conv_flops_p82":
                hc = O.conv2d_out_size(256, 3)
                got = 2 * 128 * 64 * hc * hc * (8 * 3 * 3)
            elif name == "maxpool_outputs_p42":
                ho = O.pool_out_size(512, 4, 1, 1, 1)
                got = 32 * 64 * ho * ho
            else:
                raise AssertionError(name)
        else:
            raise AssertionError(op)
        assert got == want, (args, got, want)


def test_sweep_and_tiny_sizes():
    # fused conv3x3 + pool: H -> conv H-2 -> floor((H-2-k)/k)+1
    want = {(127, 2): 62, (127, 4): 31, (255, 2): 126, (255, 4): 63, (256, 2): 127,
            (256, 4): 63, (64, 4): 15}
    for (H, k), ho in want.items():
        assert O.pool_out_size(O.conv2d_out_size(H, 3), k, k) == ho


def test_sizes_match_torch():
    for H in (1, 2, 5, 17, 64):
        for k in (1, 2, 3, 4, 5):
            for s in (1, 2, 3):
                for d in (1, 2, 3):
                    for p in range(0, k // 2 + 1):
                        if (H + 2 * p - d * (k - 1) - 1) < 0:
                            continue
                        x = torch.zeros(1, 1, H, H)
                        ho = F.max_pool2d(x, k, s, p, d).shape[-1]
                        assert O.pool_out_size(H, k, s, p, d) == ho
                for p in range(0, 3):
                    if H + 2 * p - k < 0:
                        continue
                    ho = F.conv2d(torch.zeros(1, 1, H, H), torch.zeros(1, 1, k, k), stride=s,
                                  padding=p).shape[-1]
                    assert O.conv2d_out_size(H, k, s, p) == ho
                    for op in range(0, s):
                        if (H - 1) * s - 2 * p + k + op < 1:
                            continue
                        ho = F.conv_transpose2d(torch.zeros(1, 1, H, H), torch.zeros(1, 1, k, k),
                                                stride=s, padding=p, output_padding=op).shape[-1]
                        assert O.convt_out_size(H, k, s, p, op) == ho


# --------------------------------------------------------------- conv2d ----

@pytest.mark.parametrize("stride,pad", [(1, 0), (1, 1), (2, 0), (2, 1), (3, 2)])
def test_conv2d_matches_torch_float64(stride, pad):
    x, w, cb = rnd(2, 3, 9, 11), rnd(5, 3, 3, 2), rnd(5)
    y = O.conv2d(x, w, cb, stride, pad)
    ref = F.conv2d(t64(x), t64(w), t64(cb), stride=stride, padding=pad).numpy()
    assert y.shape == ref.shape
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


def test_conv2d_delta_kernel_is_shift():
    x = rnd(1, 2, 7, 8)
    for kh in range(3):
        for kw in range(3):
            w = np.zeros((2, 2, 3, 3), np.float32)
            w[0, 1, kh, kw] = 1.0  # out channel 0 copies in channel 1
            w[1, 0, kh, kw] = 1.0
            y = O.conv2d(x, w)
            np.testing.assert_array_equal(y[0, 0], x[0, 1, kh:kh + 5, kw:kw + 6])
            np.testing.assert_array_equal(y[0, 1], x[0, 0, kh:kh + 5, kw:kw + 6])


def test_conv2d_box_sum_prefix():
    x = rnd(1, 3, 10, 9)
    w = np.ones((1, 3, 3, 3), np.float32)
    y = O.conv2d(x, w)
    s = x.astype(np.float64).sum(axis=1)[0]
    P = np.zeros((11, 10))
    P[1:, 1:] = s.cumsum(0).cumsum(1)
    box = P[3:, 3:] - P[:-3, 3:] - P[3:, :-3] + P[:-3, :-3]
    np.testing.assert_allclose(y[0, 0], box, atol=1e-12)


def test_conv2d_linearity_and_bias():
    x1, x2, w, cb = rnd(1, 2, 6, 6), rnd(1, 2, 6, 6), rnd(3, 2, 3, 3), rnd(3)
    a = O.conv2d(x1, w) + O.conv2d(x2, w)
    b = O.conv2d((x1.astype(np.float64) + x2).astype(np.float32), w)
    # x1 + x2 rounded to float32 first: compare loosely
    np.testing.assert_allclose(a, b, atol=1e-6)
    yb = O.conv2d(x1, w, cb)
    np.testing.assert_allclose(yb - O.conv2d(x1, w), np.broadcast_to(cb[None, :, None, None], yb.shape),
                               atol=1e-15)


def test_conv2d_one_matches_full():
    x, w, cb = rnd(2, 3, 8, 7), rnd(4, 3, 3, 3), rnd(4)
    y = O.conv2d(x, w, cb, 2, 1)
    lib = O.lib()
    for (n, co, oh, ow) in [(0, 0, 0, 0), (1, 3, 3, 3), (1, 2, 2, 0), (0, 1, 1, 2)]:
        v = lib.oracle_conv2d_one(x, 3, 8, 7, w, O._ptr_or_null(cb), 3, 3, 2, 1, n, co, oh, ow)
        assert v == y[n, co, oh, ow]


# -------------------------------------------------------------- maxpool ----

def brute_maxpool(x, k, s, p, d):
    """Explicit -inf padding, then windows by slicing (a second coding)."""
    N, Cc, H, W = x.shape
    Ho = (H + 2 * p - d * (k - 1) - 1) // s + 1
    Wo = (W + 2 * p - d * (k - 1) - 1) // s + 1
    xp = np.full((N, Cc, H + 2 * p + d * k + s, W + 2 * p + d * k + s), -np.inf, np.float32)
    xp[:, :, p:p + H, p:p + W] = x
    out = np.full((N, Cc, Ho, Wo), -np.inf, np.float32)
    for kh in range(k):
        for kw in range(k):
            tap = xp[:, :, kh * d: kh * d + s * (Ho - 1) + 1: s, kw * d: kw * d + s * (Wo - 1) + 1: s]
            out = np.maximum(out, tap)
    return out


GRID = [(k, s, p, d) for k in range(1, 6) for s in range(1, 4) for d in range(1, 4)
        for p in range(0, k // 2 + 1)]


def test_maxpool_matches_torch_and_brute_force():
    x = RNG.standard_normal((2, 3, 13, 11)).astype(np.float32)
    for k, s, p, d in GRID:
        if 13 + 2 * p - d * (k - 1) - 1 < 0 or 11 + 2 * p - d * (k - 1) - 1 < 0:
            continue
        out = O.maxpool2d(x, k, s, p, d)
        ref = F.max_pool2d(torch.from_numpy(x), k, s, p, d).numpy()
        np.testing.assert_array_equal(out, ref, err_msg=str((k, s, p, d)))
        np.testing.assert_array_equal(out, brute_maxpool(x, k, s, p, d))


def test_maxpool_invariants_and_separable():
    x = RNG.standard_normal((1, 2, 20, 17)).astype(np.float32)
    k, s, p, d = 4, 1, 1, 1
    out = O.maxpool2d(x, k, s, p, d)
    # separable: max over kw first (row max), then over kh
    xp = np.full((1, 2, 22, 19), -np.inf, np.float32)
    xp[:, :, 1:21, 1:18] = x
    hmax = np.max(np.stack([xp[..., :, j:j + 16] for j in range(4)]), axis=0)
    vmax = np.max(np.stack([hmax[..., i:i + 19, :] for i in range(4)]), axis=0)
    np.testing.assert_array_equal(out, vmax)
    for oh in range(out.shape[2]):
        for ow in range(out.shape[3]):
            win = xp[0, 0, oh:oh + 4, ow:ow + 4]
            assert np.all(out[0, 0, oh, ow] >= win)
            assert np.any(out[0, 0, oh, ow] == win)


def test_maxpool_identity_and_all_pad():
    x = rnd(1, 1, 5, 4)
    np.testing.assert_array_equal(O.maxpool2d(x, 1, 1, 0, 1), x)
    # k=1, p=1: the border ring of windows sees only padding -> -inf exactly there
    out = O.maxpool2d(x, 1, 1, 1, 1)
    assert out.shape == (1, 1, 7, 6)
    inner = out[0, 0, 1:-1, 1:-1]
    np.testing.assert_array_equal(inner, x[0, 0])
    ring = np.ones((7, 6), bool)
    ring[1:-1, 1:-1] = False
    assert np.all(np.isneginf(out[0, 0][ring]))
    assert not np.any(np.isinf(inner))


def test_maxpool_at_matches_full():
    x = RNG.standard_normal((2, 2, 9, 10)).astype(np.float32)
    out = O.maxpool2d(x, 3, 2, 1, 2)
    for idx in [(0, 0, 0, 0), (1, 1, 3, 3), (0, 1, 2, 1)]:
        assert O.maxpool2d_at(x, 3, 2, 1, 2, *idx) == out[idx]


def test_maxpool_tie_and_nan_reading():
    # ties: +0 and -0 compare equal; the first tap in row-major order is kept
    x = np.array([[[[-0.0, 0.0], [0.0, -0.0]]]], np.float32)
    out = O.maxpool2d(x, 2, 1, 0, 1)
    assert out[0, 0, 0, 0] == 0 and math.copysign(1, out[0, 0, 0, 0]) < 0
    x[0, 0, 0, 0] = 0.0
    x[0, 0, 0, 1] = -0.0
    out = O.maxpool2d(x, 2, 1, 0, 1)
    assert math.copysign(1, out[0, 0, 0, 0]) > 0
    # NaN propagates
    y = np.array([[[[1.0, 2.0], [np.nan, 0.5]]]], np.float32)
    assert np.isnan(O.maxpool2d(y, 2, 1, 0, 1)[0, 0, 0, 0])
    ref = F.max_pool2d(torch.from_numpy(y), 2, 1).numpy()
    assert np.isnan(ref[0, 0, 0, 0])


# ---------------------------------------------- maxpool extensions (ceil mode, indices) --
# Not on the pages: PyTorch's documented MaxPool2d options, pinned against its CPU
# implementation on NaN-free inputs (torch keeps the last NaN, the reading here is
# the first) and by invariants.

CEIL_GRID = [(k, s, p, d) for k in (1, 2, 3, 4) for s in (1, 2, 3) for p in range(0, k // 2 + 1) for d in (1, 2)]


def test_ceil_sizes_match_torch():
    seen_drop = False
    for H in (1, 2, 3, 4, 5, 6, 7, 10, 13):
        for k, s, p, d in CEIL_GRID:
            try:
                ref = F.max_pool2d(torch.zeros(1, 1, H, H), k, s, p, d, ceil_mode=True).shape[-1]
            except RuntimeError:  # torch: output size too small
                assert O.pool_out_size_ceil(H, k, s, p, d) < 1, (H, k, s, p, d)
                continue
            assert O.pool_out_size_ceil(H, k, s, p, d) == ref, (H, k, s, p, d)
            span = H + 2 * p - d * (k - 1) - 1
            if -(-span // s) * s >= H + p:  # the last ceil window would start in the right padding
                seen_drop = True
    assert seen_drop  # the sweep exercises the dropped-window rule


@pytest.mark.parametrize("ceil_mode", [False, True])
def test_maxpool_indices_match_torch(ceil_mode):
    # small integers: many ties, so the first-max rule is exercised
    x = RNG.integers(-3, 4, size=(2, 2, 11, 9)).astype(np.float32)
    for k, s, p, d in CEIL_GRID:
        if 9 + 2 * p - d * (k - 1) - 1 < 0:
            continue
        out, idx = O.maxpool2d_ex(x, k, s, p, d, ceil_mode)
        ro, ri = F.max_pool2d(torch.from_numpy(x), k, s, p, d, ceil_mode=ceil_mode, return_indices=True)
        np.testing.assert_array_equal(out, ro.numpy(), err_msg=str((k, s, p, d)))
        np.testing.assert_array_equal(idx, ri.numpy(), err_msg=str((k, s, p, d)))
        if not ceil_mode:
            np.testing.assert_array_equal(out, O.maxpool2d(x, k, s, p, d))


def test_maxpool_indices_invariants_with_nan():
    x = RNG.standard_normal((1, 2, 12, 10)).astype(np.float32)
    x[0, 0, 3, 4] = x[0, 1, 7, 2] = x[0, 1, 7, 5] = np.nan
    x[0, 0, 5, 5] = x[0, 0, 5, 6] = 9.0  # a tie at the maximum
    k, s, p, d = 3, 2, 1, 1
    out, idx = O.maxpool2d_ex(x, k, s, p, d, True)
    for c in range(2):
        plane = x[0, c]
        for oh in range(out.shape[2]):
            for ow in range(out.shape[3]):
                taps = [(oh * s - p + i * d, ow * s - p + j * d) for i in range(k) for j in range(k)]
                taps = [(h, w) for h, w in taps if 0 <= h < 12 and 0 <= w < 10]
                v, at = out[0, c, oh, ow], idx[0, c, oh, ow]
                assert (at // 10, at % 10) in taps
                vals = [plane[h, w] for h, w in taps]
                pos = taps.index((at // 10, at % 10))
                if np.isnan(v):  # the first NaN of the window in row-major order
                    assert np.isnan(plane[at // 10, at % 10]) and not any(np.isnan(vals[:pos]))
                else:  # the first maximum; no NaN in the window
                    assert plane[at // 10, at % 10] == v and not any(np.isnan(vals))
                    assert all(u < v for u in vals[:pos]) and all(u <= v for u in vals)
    assert idx[0, 0, 3, 3] == 5 * 10 + 5  # window rows/cols 5-7: the tie keeps the first tap
    assert idx[0, 0, 2, 2] == 3 * 10 + 4  # window rows/cols 3-5 holds the NaN at (3, 4)


def test_maxpool_index_of_window_without_input_tap():
    x = rnd(1, 1, 3, 3)
    out, idx = O.maxpool2d_ex(x, 1, 1, 1, 1, False)  # k = 1, p = 1: the border windows see only padding
    assert idx[0, 0, 0, 0] == -1 and np.isneginf(out[0, 0, 0, 0])
    assert idx[0, 0, 1, 1] == 0 and out[0, 0, 1, 1] == x[0, 0, 0, 0]


# ------------------------------------------------------ fused conv+pool ----

def torch_model_p82(x, w, cb, scale, bias, pk, ps):
    """The page's PyTorch model, float64 throughout (library special case)."""
    y = F.conv2d(t64(x), t64(w), t64(cb))
    y = torch.tanh(y) * scale + t64(bias).view(1, -1, 1, 1)
    return F.max_pool2d(y, pk, ps).numpy()


@pytest.mark.parametrize("pk,ps", [(4, 4), (2, 2), (3, 2), (1, 1)])
def test_convpool_matches_torch_model(pk, ps):
    x, w, cb, b = rnd(2, 3, 17, 14, lo=-2, hi=2), rnd(6, 3, 3, 3), rnd(6), rnd(6, lo=-3, hi=3)
    out = O.conv2d_tanh_scale_bias_maxpool(x, w, cb, 2.0, b, pk, ps)
    ref = torch_model_p82(x, w, cb, 2.0, b, pk, ps)
    assert out.shape == ref.shape
    # per-stage float32 rounding: a few float32 ulps of |out| <= ~5
    np.testing.assert_allclose(out, ref, rtol=0, atol=2e-6)


def test_convpool_negative_and_zero_scale():
    x, w, cb, b = rnd(1, 2, 10, 10, lo=-2, hi=2), rnd(3, 2, 3, 3), rnd(3), rnd(3)
    for scale in (-1.5, 0.0, 0.5):
        out = O.conv2d_tanh_scale_bias_maxpool(x, w, cb, scale, b, 4)
        np.testing.assert_allclose(out, torch_model_p82(x, w, cb, scale, b, 4, 4), atol=2e-6)
    out0 = O.conv2d_tanh_scale_bias_maxpool(x, w, cb, 0.0, b, 4)
    np.testing.assert_array_equal(out0, np.broadcast_to(b[None, :, None, None], out0.shape))


def test_convpool_range_bound_and_pool1():
    d = synth.convpool_inputs(2, 8, 20, 20, 16, seed=3)
    out = O.conv2d_tanh_scale_bias_maxpool(d["x"], d["w"], d["conv_b"], 2.0, d["bias"], 4)
    b = d["bias"][None, :, None, None]
    assert np.all(out >= b - 2) and np.all(out <= b + 2)
    # pool 1x1 is conv followed by the elementwise chain
    o1 = O.conv2d_tanh_scale_bias_maxpool(d["x"], d["w"], d["conv_b"], 2.0, d["bias"], 1)
    y = O.conv2d(d["x"], d["w"], d["conv_b"]).astype(np.float32)
    np.testing.assert_allclose(o1, 2.0 * np.tanh(y.astype(np.float64)) + b, atol=2e-6)


def test_convpool_literal_equals_reordered():
    """max_win(s*tanh(y)+b) == s*tanh(max_win y)+b for s>0, exactly, because every
    stage (and its float32 rounding) is monotone non-decreasing."""
    d = synth.convpool_inputs(2, 8, 22, 19, 8, seed=1)
    out = O.conv2d_tanh_scale_bias_maxpool(d["x"], d["w"], d["conv_b"], 2.0, d["bias"], 4)
    y = O.conv2d(d["x"], d["w"], d["conv_b"]).astype(np.float32)
    Ho, Wo = out.shape[2:]
    m = y[:, :, :4 * Ho, :4 * Wo].reshape(2, 8, Ho, 4, Wo, 4).max(axis=(3, 5))
    t = np.tanh(m.astype(np.float64)).astype(np.float32)
    u = (t.astype(np.float64) * 2.0).astype(np.float32)
    v = (u.astype(np.float64) + d["bias"][None, :, None, None]).astype(np.float32)
    np.testing.assert_array_equal(out, v)


def test_convpool_ragged_rows_are_dropped():
    # H=W=19 -> conv 17 -> pool4 -> 4; conv rows/cols 16 (and input row/col 18) unused
    d = synth.convpool_inputs(1, 8, 19, 19, 4, seed=2)
    base = O.conv2d_tanh_scale_bias_maxpool(d["x"], d["w"], d["conv_b"], 2.0, d["bias"], 4)
    x2 = d["x"].copy()
    x2[:, :, 18, :] += 5.0
    x2[:, :, :, 18] -= 5.0
    np.testing.assert_array_equal(
        base, O.conv2d_tanh_scale_bias_maxpool(x2, d["w"], d["conv_b"], 2.0, d["bias"], 4))
    x3 = d["x"].copy()
    x3[:, :, 17, :] += 5.0  # row 17 feeds conv row 15, inside the last window
    assert not np.array_equal(
        base, O.conv2d_tanh_scale_bias_maxpool(x3, d["w"], d["conv_b"], 2.0, d["bias"], 4))


def test_convpool_at_matches_full():
    d = synth.convpool_inputs(2, 8, 30, 27, 16, seed=0)
    for pk, ps in ((4, 4), (3, 2)):
        out = O.conv2d_tanh_scale_bias_maxpool(d["x"], d["w"], d["conv_b"], 2.0, d["bias"], pk, ps)
        for idx in [(0, 0, 0, 0), (1, 15, 6, 5), (0, 7, 3, 2), (1, 3, 0, 5), (1, 9, 5, 0)]:
            v = O.convpool_at(d["x"], d["w"], d["conv_b"], 2.0, d["bias"], pk, ps, *idx)
            assert v == out[idx]


def test_convpool_unique_max_window():
    # one input pixel far above the rest: its conv response wins its windows
    x = np.zeros((1, 1, 10, 10), np.float32)
    x[0, 0, 5, 6] = 3.0
    w = np.zeros((1, 1, 3, 3), np.float32)
    w[0, 0, 1, 1] = 1.0  # y[i,j] = x[i+1,j+1]
    out = O.conv2d_tanh_scale_bias_maxpool(x, w, None, 2.0, np.array([0.25], np.float32), 4)
    assert out.shape == (1, 1, 2, 2)
    # y peak at (4,5) -> window (1,1)
    assert out[0, 0, 1, 1] == np.float32(np.float32(2.0 * np.float32(math.tanh(3.0))) + 0.25)
    assert out[0, 0, 0, 0] == np.float32(0.25)


# --------------------------------------------------------- conv-transpose ----

@pytest.mark.parametrize("K,s,p,op", [(4, 2, 1, 1), (4, 2, 1, 0), (3, 2, 0, 1), (3, 1, 1, 0),
                                      (5, 3, 2, 2), (2, 2, 0, 0)])
def test_convt_matches_torch_float64(K, s, p, op):
    x, w, cb = rnd(2, 3, 6, 5), rnd(3, 5, K, K), rnd(5)
    y = O.convt2d(x, w, cb, s, p, op)
    ref = F.conv_transpose2d(t64(x), t64(w), t64(cb), stride=s, padding=p,
                             output_padding=op).numpy()
    assert y.shape == ref.shape
    np.testing.assert_allclose(y, ref, atol=1e-12)


def test_convt_adjoint_identity():
    """<convT(x; W), y> == <x, conv2d(y; W, stride s, pad p)>: W [Cin,Cout,K,K]
    read as a conv weight [out=Cin, in=Cout, K, K]."""
    for (H, W, K, s, p, op) in [(6, 7, 4, 2, 1, 1), (5, 5, 3, 2, 1, 0), (4, 6, 5, 3, 2, 1)]:
        x, w = rnd(2, 4, H, W), rnd(4, 3, K, K)
        yt = O.convt2d(x, w, None, s, p, op)
        y = rnd(*yt.shape)
        lhs = float(np.sum(yt * y.astype(np.float64)))
        cy = O.conv2d(y, w, None, s, p)
        assert cy.shape == x.shape
        rhs = float(np.sum(x.astype(np.float64) * cy))
        assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def test_convt_delta_input():
    w = rnd(2, 3, 4, 4)
    for (ih, iw) in [(0, 0), (2, 3), (4, 4)]:
        x = np.zeros((1, 2, 5, 5), np.float32)
        x[0, 1, ih, iw] = 1.0
        y = O.convt2d(x, w, None, 2, 1, 1)
        exp = np.zeros_like(y)
        for kh in range(4):
            for kw in range(4):
                oh, ow = 2 * ih - 1 + kh, 2 * iw - 1 + kw
                if 0 <= oh < y.shape[2] and 0 <= ow < y.shape[3]:
                    exp[0, :, oh, ow] = w[1, :, kh, kw]
        np.testing.assert_array_equal(y, exp)


def _phase_table(golden_dir):
    rows, phases = {}, {}
    for line in open(os.path.join(golden_dir, "convt_phase_taps.txt")):
        line = line.strip()
        if line.startswith("rows"):
            py = int(re.search(r"py=(\d)", line).group(1))
            rows[py] = [tuple(int(v) for v in t.split(":")) for t in line.split("->")[1].split()]
        elif line.startswith("phase"):
            lhs, rhs = line.split("->")
            py, px = map(int, lhs.split()[1:])
            phases[(py, px)] = [tuple(map(int, t.strip("()").split(","))) for t in rhs.split()]
    return rows, phases


def test_convt_phase_decomposition(golden_dir):
    """Gather through the page's 4-phase table == the scatter oracle (k4 s2 p1)."""
    rows, phases = _phase_table(golden_dir)
    for (py, px), taps in phases.items():
        assert sorted(taps) == sorted((kh, kw) for kh, _ in rows[py] for kw, _ in rows[px])
    x, w, cb = rnd(1, 3, 5, 6), rnd(3, 4, 4, 4), rnd(4)
    y = O.convt2d(x, w, cb, 2, 1, 1)
    H, W = 5, 6
    g = np.zeros_like(y)
    for oh in range(y.shape[2]):
        for ow in range(y.shape[3]):
            m, py = divmod(oh, 2)
            n, px = divmod(ow, 2)
            acc = cb.astype(np.float64).copy()
            for kh, dy in rows[py]:
                for kw, dx in rows[px]:
                    ih, iw = m + dy, n + dx
                    if 0 <= ih < H and 0 <= iw < W:
                        acc += x[0, :, ih, iw].astype(np.float64) @ w[:, :, kh, kw].astype(np.float64)
            g[0, :, oh, ow] = acc
    np.testing.assert_allclose(g, y, atol=1e-12)


def test_convt_gather_one_matches_scatter():
    x, w, cb = rnd(2, 3, 5, 4), rnd(3, 6, 4, 4), rnd(6)
    y = O.convt2d(x, w, cb, 2, 1, 1)
    for idx in [(0, 0, 0, 0), (1, 5, 10, 8), (0, 3, 9, 1), (1, 2, 4, 7)]:
        v = O.convt2d_one(x, w, cb, 2, 1, *idx)
        assert abs(v - y[idx]) <= 1e-12


# ------------------------------------------------------ softmax epilogue ----

def test_softmax_sums_to_one_and_order():
    y = (RNG.standard_normal(128) * 3).astype(np.float32)
    p = O.softmax_channels(y)
    assert abs(float(np.sum(p.astype(np.float64))) - 1.0) < 128 * 2 ** -24
    assert np.all(p > 0)
    assert np.argmax(p) == np.argmax(y)
    ref = torch.softmax(t64(y), 0).numpy()
    np.testing.assert_allclose(p, ref, rtol=2 ** -23, atol=0)
    # shift invariance
    np.testing.assert_array_equal(O.softmax_channels(y), O.softmax_channels((y + 0.0).astype(np.float32)))


def test_equal_logits_closed_form():
    C = 128
    b = RNG.standard_normal(C).astype(np.float32)
    out = O.softmax_bias_scale_sigmoid_pixel(np.full(C, 0.7, np.float32), b, 2.0)
    exp = 1.0 / (1.0 + np.exp(-2.0 * (1.0 / C + b.astype(np.float64))))
    np.testing.assert_allclose(out, exp, atol=3e-7)


def torch_model_p91(x, w, cb, bias, scale, s=2, p=1, op=1):
    y = F.conv_transpose2d(t64(x), t64(w), t64(cb), stride=s, padding=p, output_padding=op)
    y = torch.softmax(y, dim=1)
    return torch.sigmoid((y + t64(bias).view(1, -1, 1, 1)) * scale).numpy()


def test_convt_model_matches_torch():
    d = synth.convt_inputs(2, 8, 5, 6, 16, seed=4)
    out = O.convtranspose2d_softmax_bias_scale_sigmoid(d["x"], d["w"], d["conv_b"], d["bias"], 2.0)
    ref = torch_model_p91(d["x"], d["w"], d["conv_b"], d["bias"], 2.0)
    assert out.shape == (2, 16, 11, 13)
    assert np.all((out > 0) & (out < 1))
    np.testing.assert_allclose(out, ref, atol=2e-7)


def test_convt_fused_pixel_matches_full():
    d = synth.convt_inputs(2, 8, 5, 4, 16, seed=5)
    out = O.convtranspose2d_softmax_bias_scale_sigmoid(d["x"], d["w"], d["conv_b"], d["bias"], 2.0)
    for (n, oh, ow) in [(0, 0, 0), (1, 10, 8), (0, 5, 3), (1, 9, 0)]:
        v = O.convt_fused_pixel(d["x"], d["w"], d["conv_b"], d["bias"], 2.0, 2, 1, n, oh, ow)
        np.testing.assert_allclose(v, out[n, :, oh, ow], atol=1e-7)
