"""Planted mistakes in the oracle must fail its pins.

Each case copies the oracle's C source, plants one plausible mistake (a dropped
term, a wrong sign or index, a transposed operand, a wrong padding value ...),
compiles the copy on the CPU and runs the pin suite against it; at least one
pin has to fail.  The oracle itself is never modified.
"""
import inspect
import os
import subprocess

import pytest

from oracle import oracle as O
import tests.test_oracle_pins as pins

SRC = open(os.path.join(os.path.dirname(O.__file__), "fusedwin_oracle.c")).read()

MUTANTS = {
    "conv_drops_bias": ("double acc = cb ? (double)cb[co] : 0.0;\n    for (long ci = 0; ci < Cin; ++ci)\n        for (long kh = 0; kh < KH; ++kh)",
                        "double acc = 0.0;\n    for (long ci = 0; ci < Cin; ++ci)\n        for (long kh = 0; kh < KH; ++kh)"),
    "conv_kernel_transposed": ("w[((co * Cin + ci) * KH + kh) * KW + kw]", "w[((co * Cin + ci) * KH + kw) * KW + kh]"),
    "conv_pad_sign": ("long ih = oh * s - p + kh, iw = ow * s - p + kw;", "long ih = oh * s + p + kh, iw = ow * s - p + kw;"),
    "conv_size_off_by_one": ("return floordiv(H + 2 * p - k, s) + 1;", "return floordiv(H + 2 * p - k, s);"),
    "pool_pad_zero": ("plane[ih * W + iw] : -INFINITY;", "plane[ih * W + iw] : 0.0f;"),
    "pool_ignores_dilation": ("long ih = oh * s - p + kh * d, iw = ow * s - p + kw * d;",
                              "long ih = oh * s - p + kh, iw = ow * s - p + kw * d;"),
    "pool_tie_keeps_last": ("if (isnan(v) || v > m) return v;", "if (isnan(v) || v >= m) return v;"),
    "pool_size_formula": ("return floordiv(H + 2 * p - d * (k - 1) - 1, s) + 1;", "return floordiv(H + 2 * p - d * (k - 1), s) + 1;"),
    "ceil_keeps_window_in_right_padding": ("if (o >= 1 && (o - 1) * s >= H + p) o -= 1;", "if (o >= 1 && (o - 1) * s > H + p) o -= 1;"),
    "index_tie_keeps_last": ("if (at < 0 || (!isnan(m) && (isnan(v) || v > m))) {", "if (at < 0 || (!isnan(m) && (isnan(v) || v >= m))) {"),
    "index_transposed": ("                at = ih * W + iw;\n            }", "                at = iw * H + ih;\n            }"),
    "epilogue_bias_sign": ("return (float)((double)u + (double)b);", "return (float)((double)u - (double)b);"),
    "epilogue_no_tanh": ("float t = (float)tanh((double)y);", "float t = y;"),
    "convpool_window_stride": ("long oh = i * ps + a, ow = j * ps + b;", "long oh = i * pk + a, ow = j * ps + b;"),
    "convt_index_sign": ("long oh = ih * s - p + kh, ow = iw * s - p + kw;", "long oh = ih * s + p - kh, ow = iw * s - p + kw;"),
    "convt_weight_transposed": ("double wv = w[((ci * Cout + co) * K + kh) * K + kw];",
                                "double wv = w[((co * Cin + ci) * K + kh) * K + kw];"),
    "convt_gather_no_divisibility": ("if (th < 0 || th % s != 0 || th / s >= H) continue;",
                                     "if (th < 0 || th / s >= H) continue;"),
    "convt_size_no_plus_one": ("return (H - 1) * s - 2 * p + (k - 1) + op + 1;", "return (H - 1) * s - 2 * p + (k - 1) + op;"),
    "softmax_bad_normaliser": ("p[c] = (float)(e_scratch[c] / sum);", "p[c] = (float)(e_scratch[c] / (sum + 1.0));"),
    "sigmoid_sign": ("out[c] = (float)(1.0 / (1.0 + exp(-(double)r)));", "out[c] = (float)(1.0 / (1.0 + exp((double)r)));"),
    "scale_before_bias": ("float q = (float)((double)out[c] + (double)bias[c]);\n        float r = (float)((double)q * (double)scale);",
                          "float q = (float)((double)out[c] * (double)scale);\n        float r = (float)((double)q + (double)bias[c]);"),
}


def _pin_tests():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argnames = [a.strip() for a in params[0].args[0].split(",")]
            for vals in params[0].args[1]:
                vals = vals if isinstance(vals, tuple) else (vals,)
                out.append((name, fn, dict(zip(argnames, vals))))
        else:
            out.append((name, fn, {}))
    return out


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(mutant, tmp_path, golden_dir):
    old, new = MUTANTS[mutant]
    assert SRC.count(old) == 1, f"mutation anchor for {mutant} not unique"
    src = tmp_path / "mutant.c"
    src.write_text(SRC.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(so),
                    str(src), "-lm"], check=True)
    saved = O._lib
    O._lib = O.load(str(so))
    caught = None
    try:
        for name, fn, kwargs in _pin_tests():
            if "golden_dir" in inspect.signature(fn).parameters:
                kwargs = dict(kwargs, golden_dir=golden_dir)
            try:
                fn(**kwargs)
            except Exception as e:  # noqa: BLE001 - any failure of a pin counts
                caught = (name, type(e).__name__)
                break
    finally:
        O._lib = saved
    assert caught is not None, f"no pin caught the planted mistake {mutant}"
