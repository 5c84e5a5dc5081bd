"""The decode-attention tolerance of the GPU tests, and a record of the errors they observe.

The contract bounds the decode output by a maximum relative error of 2e-3 and a maximum
absolute error of 1e-3 against the fp64 oracle over the same dequantized values. Reading:
an output element passes when |gpu - oracle| <= max(1e-3, 2e-3 |oracle|), so the absolute
bound governs where |oracle| < 0.5 (a relative bound means nothing near zero) and the
relative one above.

Every check records, per case name, the largest absolute error, the largest relative error
among the elements where the relative bound governs, and the largest ratio of error to bound;
the session prints them at the end and, when KVQ_PARITY_REPORT names a file, writes them there
as JSON.
"""

import json
import os

import numpy as np

ATOL, RTOL = 1e-3, 2e-3

OBSERVED = {}


def bound(ref, atol=ATOL, rtol=RTOL):
    return np.maximum(atol, rtol * np.abs(ref))


def check(name, got, ref, atol=ATOL, rtol=RTOL, where=""):
    """Asserts |got - ref| <= max(atol, rtol |ref|) elementwise and records the error maxima
    under `name`. Returns the largest error / bound ratio of this call."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    b = bound(ref, atol, rtol)
    ratio = float(np.max(err / b)) if err.size else 0.0
    rel_zone = np.abs(ref) >= atol / rtol
    rec = OBSERVED.setdefault(name, {"max_abs": 0.0, "max_rel": 0.0, "worst_ratio": 0.0, "elements": 0,
                                     "atol": atol, "rtol": rtol})
    rec["max_abs"] = max(rec["max_abs"], float(err.max()) if err.size else 0.0)
    if rel_zone.any():
        rec["max_rel"] = max(rec["max_rel"], float(np.max(err[rel_zone] / np.abs(ref[rel_zone]))))
    rec["worst_ratio"] = max(rec["worst_ratio"], ratio)
    rec["elements"] += int(err.size)
    if not np.all(np.isfinite(got)):
        raise AssertionError(f"{name} {where}: non-finite outputs")
    if ratio > 1.0:
        i = int(np.argmax(err / b))
        raise AssertionError(f"{name} {where}: |gpu - oracle| {err.flat[i]:.3g} exceeds max({atol:g}, {rtol:g} |ref|)"
                             f" = {b.flat[i]:.3g} at element {i} (ref {ref.flat[i]:.4g})")
    return ratio


def report_lines():
    if not OBSERVED:
        return []
    lines = [f"{'case':44s} {'max |err|':>10s} {'max rel':>10s} {'err/bound':>9s} {'elements':>9s}"]
    for k in sorted(OBSERVED):
        r = OBSERVED[k]
        lines.append(f"{k:44s} {r['max_abs']:10.3e} {r['max_rel']:10.3e} {r['worst_ratio']:9.3f} {r['elements']:9d}")
    return lines


def write_report():
    path = os.environ.get("KVQ_PARITY_REPORT")
    if path and OBSERVED:
        with open(path, "w") as f:
            json.dump(OBSERVED, f, indent=1, sort_keys=True)
