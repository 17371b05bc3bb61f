"""Largest errors of the GPU parity tests, printed in pytest's closing summary.

Each parity test records, per output, the max-abs error against the fp64 oracle,
the tolerance it is held to, and the rounding floor: half a unit in the last
place of the reference in the output's dtype (the error a correctly rounded
result would still have), so the margin of every case is visible in the run's
log even with -q.
"""
ROWS = []


def record(case, errs, tols, floors=None):
    ROWS.append((case, dict(errs), dict(tols), dict(floors or {})))


def lines():
    out = []
    for case, errs, tols, floors in ROWS:
        parts = []
        for k, e in errs.items():
            fl = f", floor {floors[k]:.1e}" if k in floors else ""
            parts.append(f"{k} {e:.2e} (tol {tols[k]:.0e}{fl})")
        out.append(f"{case}: " + "; ".join(parts))
    return out
