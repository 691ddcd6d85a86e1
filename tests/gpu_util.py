"""Helpers shared by the GPU parity tests."""
import numpy as np

# Tolerances. fp32 per-vertex: 1e-5 relative with an absolute floor of 1e-9;
# |sum - 1| <= 1e-5; iteration counts within +-1.
# fp64: 1e-11 relative (floor 1e-15), |sum - 1| <= 1e-12. Where that comes
# from: every fp64 operation rounds at 2^-53 ~ 1.1e-16; a row sum of up to
# 1e5 terms added in tree order gains at most log2(1e5) ulps ~ 2e-15
# relative; the update contracts earlier errors by d = 0.85, so the error
# settles below 1/(1 - d) ~ 6.7 times the per-update error, ~1.3e-14, plus a
# few ulps for the state round trip x = s * outdeg. 1e-11 leaves three
# orders of magnitude of headroom over that bound.
F32 = dict(rel=1e-5, abs=1e-9, sum=1e-5)
F64 = dict(rel=1e-11, abs=1e-15, sum=1e-12)


def assert_ranks_close(x, ref, tol, what=""):
    x = np.asarray(x, dtype=np.float64)
    err = np.abs(x - ref)
    bound = np.maximum(tol["rel"] * np.abs(ref), tol["abs"])
    bad = np.nonzero(err > bound)[0]
    if bad.size:
        w = bad[np.argmax(err[bad] / bound[bad])]
        raise AssertionError(f"{what}: {bad.size} of {x.size} vertices out of tolerance; worst v={w} "
                             f"gpu={x[w]!r} oracle={ref[w]!r} rel={err[w] / max(abs(ref[w]), 1e-300):.3e}")
