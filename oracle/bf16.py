"""Round-to-nearest-even onto the bfloat16 grid, written from the format's
definition (8 significant bits, fp32 exponent range).  Used by the oracle to
place the same storage roundings as a bf16 program; the arithmetic between
those points stays fp64.  Test infrastructure only."""
import numpy as np


def round_bf16(x):
    """Nearest bf16 value of each fp64 element, ties to even.

    bf16 keeps 8 significant bits (1 implicit + 7 stored).  With
    x = m * 2**e, 0.5 <= |m| < 1, the grid spacing at x is 2**(e-8); rounding
    m * 2**8 to the nearest integer (half to even) and scaling back is exact
    in fp64.  Values below the smallest normal are not produced by any
    workload here and are rounded on the same formula.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    return np.where(np.isfinite(x), r, x)
