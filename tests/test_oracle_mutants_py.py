"""The pins of the oracle's Python routes have teeth too.

Each mutant is a one-token slip planted in a copy of one function of
oracle/__init__.py (im2col, the window-order buffer, the indirection buffer,
the window-buffer size), swapped into the oracle module for the duration of
the check.  The pins of tests/test_oracle_pins.py that cover the function must
reject every mutant and pass the unmodified function.  Geometries are the pins'
own (several strides, dilations, paddings and non-square kernels).
"""
import inspect
import textwrap

import pytest

import oracle
import test_oracle_pins as pins

# function -> {mutant: (original text, planted slip)}
MUTANTS = {
    "im2col": {
        "taps_transposed": ("h0, w0 = kh * dilation, kw * dilation",
                            "h0, w0 = kw * dilation, kh * dilation"),
        "width_stride_dropped": ("w0:w0 + stride * (W_out - 1) + 1:stride",
                                 "w0:w0 + W_out"),
        "pad_offset_dropped": ("xp[:, pad:pad + H, pad:pad + W, :] = x_f64",
                               "xp[:, :H, :W, :] = x_f64"),
    },
    "indirection_buffer": {
        "pad_sign": ("h = ho * stride + kh * dilation - pad",
                     "h = ho * stride + kh * dilation + pad"),
        "offset_transposed": ("buf[ho, wo, kh, kw] = (h * W + w) * C_in",
                              "buf[ho, wo, kh, kw] = (w * H + h) * C_in"),
        "stride_dilation_swapped": ("w = wo * stride + kw * dilation - pad",
                                    "w = wo * dilation + kw * stride - pad"),
    },
    "im2win": {
        "width_one_too_many": ("W_used = (W_out - 1) * stride + (KW - 1) * dilation + 1",
                               "W_used = (W_out - 1) * stride + (KW - 1) * dilation + 2"),
        "column_offset_sign": ("w = wc - pad", "w = wc + pad"),
        "row_dilation_dropped": ("h = ho * stride + kh * dilation - pad",
                                 "h = ho * stride + kh - pad"),
    },
    "im2win_elements": {
        "rows_dropped": ("return N * H_out * W_used * KH * C_in",
                         "return N * H_out * W_used * C_in"),
        "width_from_input": ("W_used = (W_out - 1) * stride + (KW - 1) * dilation + 1",
                             "W_used = W + 2 * pad"),
    },
}


def _each_geom(test):
    return lambda: [test(g) for g in pins.GEOMS]


# the pins that cover each function
PINS = {
    "im2col": [_each_geom(pins.test_im2col_matches_torch_unfold),
               _each_geom(pins.test_direct_matches_im2col_gemm)],
    "indirection_buffer": [_each_geom(pins.test_indirection_buffer_reproduces_unfold)],
    "im2win": [_each_geom(pins.test_im2win_windows_reproduce_unfold),
               _each_geom(pins.test_im2win_width_is_the_tightest_span_of_the_columns_read)],
    "im2win_elements": [_each_geom(pins.test_im2win_windows_reproduce_unfold),
                        _each_geom(pins.test_im2win_width_is_the_tightest_span_of_the_columns_read)],
}


def _mutant(fname, old, new):
    src = textwrap.dedent(inspect.getsource(getattr(oracle, fname)))
    assert src.count(old) == 1, (fname, old)
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant of oracle.%s>" % fname, "exec"), ns)
    return ns[fname]


def _pins_pass(fname):
    try:
        for pin in PINS[fname]:
            pin()
    except (AssertionError, IndexError, ValueError):
        return False
    return True


CASES = [(f, m) for f in MUTANTS for m in MUTANTS[f]]


@pytest.mark.parametrize("fname", sorted(MUTANTS))
def test_unmodified_functions_pass_their_pins(fname):
    assert _pins_pass(fname)


@pytest.mark.parametrize("fname,mutant", CASES, ids=["%s-%s" % c for c in CASES])
def test_pins_reject_planted_slips(monkeypatch, fname, mutant):
    old, new = MUTANTS[fname][mutant]
    monkeypatch.setattr(oracle, fname, _mutant(fname, old, new))
    assert not _pins_pass(fname), "pins accepted %s in oracle.%s" % (mutant, fname)
