"""The output bar of the parity tests: max-abs 1e-2 and mean-abs 1e-3 against the fp64 oracle.

The operator returns O in bf16 (8 significant bits).  Below |o| = 4 the nearest bf16 value is
within 0.0078 of any real value, so 1e-2 leaves the arithmetic a margin.  From 4 on, bf16 values
are 1/32 apart (1/16 from 8): the nearest one can be 0.0156 away, and no bf16 output, however it
is computed, meets 1e-2 there.  For those elements the bar is that the output be one of the two
bf16 values around the exact one (faithful rounding): |o - exact| below the bf16 spacing at |o|.
The mean-abs bar and the LSE bar (fp32 output) are unchanged.
"""
import numpy as np

MAX_ABS, MEAN_ABS = 1e-2, 1e-3


def o_bar(ref):
    """Per-element bound on |output - oracle| for a bf16 output of exact value `ref`."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    wide = a >= 4.0
    spacing = np.exp2(np.floor(np.log2(np.where(wide, a, 1.0))) - 7)  # 2^(e - 7), e = exponent
    return np.where(wide, spacing, MAX_ABS)


def o_within_bar(got, ref):
    """True when every element of a bf16 output meets o_bar and the mean error is within
    MEAN_ABS; also returns the max error and the number of elements under the wider bar."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    ok = bool((err <= o_bar(ref)).all()) and err.mean() <= MEAN_ABS
    return ok, float(err.max()), int((np.abs(ref) >= 4.0).sum())
