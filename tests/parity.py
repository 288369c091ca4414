"""Tolerance rule for 16-bit outputs averaged from values of magnitude above one.

The stated bars (out max-abs 1e-2, mean-abs 1e-3) assume values of order one.
A 16-bit result cannot meet them once the values being averaged are larger:
with m stored mantissa bits (7 for bf16, 10 for fp16) the unit roundoff is
2^-(m+1), and the GPU path rounds P to the 16-bit type before P.V and rounds
the output itself.  For one output element, with weights p_j and values v_j,

    A = sum_j p_j |v_j| / sum_j p_j        (the weighted mean magnitude)

bounds both: rounding each p_j moves the output by at most 2^-(m+1) A, and
rounding the output (|out| <= A) by at most 2^-(m+1) A more; fp32
accumulation adds far less.  A is what the oracle computes when given |V| in
place of V.  Reading, with `large` the elements where 2^-m A > 1e-2 (bf16: A
above 1.28):

  * elsewhere: the stated bars, |out - ref| <= 1e-2 each and the mean of
    those errors <= 1e-3;
  * large elements: |out - ref| <= 2^-m A each, and the mean of
    |out - ref| / (2^-m A) over them <= 0.5 (half the bound on average: the
    output's own rounding alone averages a quarter).

Values of order one therefore keep exactly the stated bars; the bound only
widens in proportion to the magnitude of the values averaged.
"""
import numpy as np


def abs_values(bits):
    """16-bit bit patterns with the sign bit cleared: |v| exactly."""
    return (np.asarray(bits, np.uint16) & np.uint16(0x7FFF)).astype(np.uint16)


def bounds_16(abs_mean, dtype: str = "bf16"):
    """(per-element bound, mask of the large elements) for outputs whose
    weighted mean value magnitude is `abs_mean` (the oracle's output on |V|)."""
    m = 7 if dtype == "bf16" else 10
    rel = np.abs(np.asarray(abs_mean, np.float64)) * 2.0 ** -m
    large = rel > 1e-2
    return np.where(large, rel, 1e-2), large


def assert_close_16(out, lse, ref_out, ref_lse, abs_mean, dtype: str = "bf16", lse_tol: float = 1e-3):
    out = np.asarray(out, np.float64)
    ref_out = np.asarray(ref_out, np.float64)
    assert np.all(np.isfinite(out))
    err = np.abs(out - ref_out)
    bound, large = bounds_16(abs_mean, dtype)
    r = err / bound
    i = int(np.argmax(r))
    assert r.max() <= 1.0, (f"abs err {err.flat[i]:.3g} where |ref| = {abs(ref_out.flat[i]):.4g} and the values "
                            f"average {np.abs(np.asarray(abs_mean)).flat[i]:.4g} (bound {bound.flat[i]:.3g})")
    if (~large).any():
        assert err[~large].mean() <= 1e-3, f"mean abs err {err[~large].mean():.3g} (values of order one)"
    if large.any():
        assert r[large].mean() <= 0.5, f"mean error {r[large].mean():.3g} of the bound (large values)"
    neg = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), neg)
    if (~neg).any():
        le = np.abs(np.asarray(lse)[~neg] - np.asarray(ref_lse)[~neg])
        assert le.max() <= lse_tol, f"lse err {le.max():.3g}"


def scale_16_bits(bits, factor: float, dtype: str = "bf16"):
    """16-bit bit patterns times a power of two, exactly (only the exponent
    moves; the caller keeps the values inside the format's normal range)."""
    assert float(factor) == 2.0 ** round(np.log2(factor))
    if dtype == "bf16":
        f = (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32) * np.float32(factor)
        out = (f.view(np.uint32) >> 16).astype(np.uint16)
        assert np.array_equal((out.astype(np.uint32) << 16).view(np.float32), f)
        return out
    f = np.asarray(bits, np.uint16).view(np.float16).astype(np.float32) * np.float32(factor)
    out = f.astype(np.float16)
    assert np.array_equal(out.astype(np.float32), f)
    return out.view(np.uint16)
