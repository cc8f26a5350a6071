"""Analytic stalled-update model for a low-precision second moment
(TEST INFRASTRUCTURE ONLY; see oracle/__init__.py).

Follows "When Small Updates Disappear" (Topollai), sec. 1.1-3.2.  The page's
display equations were lost in extraction; the formulas below are the
reading that reproduces every percentage the page prints (94.6 % BF16 nearest
in sec. 2.3; 82.5 / 98.9 / 99.4 % stochastic in sec. 3.2):

* the stored value moves by Delta = (1 - b2) (g^2 - v)            (sec. 1.1)
* the grid spacing near v = m 2^e is u = 2^(e-p) = v / (m 2^p)     (sec. 2.1)
* nearest rounding stalls when |Delta| < u/2                       (sec. 2)
* with g/sigma ~ N(0,1), v ~ sigma^2, z = g^2/sigma^2 ~ chi^2_1 and the
  mantissa replaced by its typical value 1/ln 2, the ratio of update to grid
  depends on rho = eps ln2 / (2 (1 - b2)), eps = 2^-p            (sec. 2.3)
* nearest: P = Pr(|z - 1| < rho)                                   (sec. 2.3)
* stochastic: stall probability 1 - |Delta|/u when |Delta| < u, so
  P = E[max(0, 1 - |z - 1| / (2 rho))]                             (sec. 3.2)
"""
from __future__ import annotations

import math

from scipy import integrate, stats

# fraction bits p of each state format (sec. 2.1)
FRACTION_BITS = {"bf16": 7, "e4m3": 3, "e2m2": 2}


def rho(beta2: float, p: int) -> float:
    return (2.0 ** -p) * math.log(2.0) / (2.0 * (1.0 - beta2))


def stall_nearest(beta2: float, p: int) -> float:
    r = rho(beta2, p)
    lo, hi = max(0.0, 1.0 - r), 1.0 + r
    return float(stats.chi2.cdf(hi, 1) - stats.chi2.cdf(lo, 1))


def stall_stochastic(beta2: float, p: int) -> float:
    r = rho(beta2, p)
    lo, hi = max(0.0, 1.0 - 2.0 * r), 1.0 + 2.0 * r

    def integrand(z):
        return max(0.0, 1.0 - abs(z - 1.0) / (2.0 * r)) * stats.chi2.pdf(z, 1)

    # the chi^2_1 density has an integrable singularity at 0 and the tent a
    # kink at 1: split there
    pts = sorted({lo, 1.0, hi})
    total = 0.0
    for a, b in zip(pts[:-1], pts[1:]):
        val, _ = integrate.quad(integrand, a, b, limit=200)
        total += val
    return total
