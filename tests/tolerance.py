"""Acceptance rules used by the parity tests.

bf16 attention output (vLLM PR 60684, Validation): all but a 1e-4 fraction
of the elements lie within atol = rtol = 0.05 of the reference, read as the
allclose form |got - ref| <= 0.05 + 0.05 * |ref|, and every element lies
within 0.25 absolute.  The page gives the reason: the probabilities are
rounded to E4M3 before the PV product.

FP32 quantities (the lse output, the combine of given fp32 partials): max
absolute difference to the FP64 oracle <= 1e-2.
"""
from __future__ import annotations

import math

import numpy as np

ATOL = 0.05
RTOL = 0.05
OUTLIER_FRACTION = 1e-4
HARD_BOUND = 0.25
FP32_PATH_TOL = 1e-2


def acceptance(got, ref):
    """Returns a dict of error statistics and whether the rule holds."""
    g = np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    err = np.abs(g - r)
    outside = err > ATOL + RTOL * np.abs(r)
    n = err.size
    allowed = math.floor(OUTLIER_FRACTION * n)
    stats = {
        "n": int(n),
        "outside": int(outside.sum()),
        "allowed": int(allowed),
        "max_abs": float(err.max(initial=0.0)),
        "mean_abs": float(err.mean()) if n else 0.0,
        "nonfinite": int((~np.isfinite(g)).sum()),
    }
    stats["ok"] = (stats["nonfinite"] == 0 and stats["outside"] <= allowed
                   and stats["max_abs"] <= HARD_BOUND)
    return stats


def assert_acceptance(got, ref, what=""):
    s = acceptance(got, ref)
    assert s["ok"], "%s: acceptance rule failed: %s" % (what, s)
    return s


def assert_lse(got, ref, what="", tol=FP32_PATH_TOL):
    g = np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    fin = np.isfinite(r)
    assert np.array_equal(np.isneginf(g), np.isneginf(r)), \
        "%s: -inf pattern of lse differs" % what
    err = np.abs(g[fin] - r[fin]).max(initial=0.0)
    assert err <= tol, "%s: lse max abs error %g > %g" % (what, err, tol)
    return float(err)
