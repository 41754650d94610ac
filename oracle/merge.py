"""The online-softmax log-sum-exp merge, Eq. 2.

Source: "Online Draft Co-Training ..." — rainbus page, "核心方法" (core
method), Eq. 2: l = log(e^l_m + e^l_b) and
O = (e^(l_m - l) O_m + e^(l_b - l) O_b) / (e^(l_m - l) + e^(l_b - l));
ai.info summary, Key Contributions 1 (the two attention results are merged
with the standard online-softmax reduction).

Reading: an empty part (no visible keys) has l = -inf and O = 0 and merges as
the identity; when both parts are empty the result is O = 0, l = -inf.  The
log of the sum is taken shifted by max(l_m, l_b) so that it does not
overflow; the denominator is evaluated as printed (it equals 1 up to
rounding).
"""

from __future__ import annotations

import numpy as np


def lse_merge(o_m: np.ndarray, l_m: np.ndarray, o_b: np.ndarray, l_b: np.ndarray):
    """Eq. 2 over rows.  o_*: [..., d]; l_*: [...]  ->  (o, l)."""
    o_m = np.asarray(o_m, dtype=np.float64)
    o_b = np.asarray(o_b, dtype=np.float64)
    l_m = np.asarray(l_m, dtype=np.float64)
    l_b = np.asarray(l_b, dtype=np.float64)
    top = np.maximum(l_m, l_b)
    both_empty = np.isneginf(top)
    shift = np.where(both_empty, 0.0, top)
    with np.errstate(invalid="ignore", divide="ignore"):
        l = shift + np.log(np.exp(l_m - shift) + np.exp(l_b - shift))
        l = np.where(both_empty, -np.inf, l)
        safe_l = np.where(both_empty, 0.0, l)
        w_m = np.where(np.isneginf(l_m), 0.0, np.exp(l_m - safe_l))
        w_b = np.where(np.isneginf(l_b), 0.0, np.exp(l_b - safe_l))
        den = w_m + w_b
        o = (w_m[..., None] * o_m + w_b[..., None] * o_b) / np.where(den == 0, 1.0, den)[..., None]
    o = np.where(both_empty[..., None], 0.0, o)
    return o, l
