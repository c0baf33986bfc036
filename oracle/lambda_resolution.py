"""Oracle for the threshold resolution (test infrastructure only).

Skip-Softmax design doc, "From configuration to the kernel threshold": the kernel
takes a threshold_scale_factor and divides it by the call's KV length,
lambda = factor / max_kv_len.  The factor comes from one of two mutually exclusive
controls:

    threshold = t          factor = t * max_kv_len          lambda = t
    target_sparsity = s    factor = a * exp(b * s)          lambda = a*exp(b*s)/max_kv_len

(BLASST talk notes, "threshold calibration": the fitted law lambda*L = a*exp(b*S),
Eq. 3's inverse-length form lambda = a/L.)  A request for target_sparsity without
calibration coefficients is an error that points to `threshold` (design doc,
"Skip-Softmax calibration config").
"""
from __future__ import annotations

import math

ACCEPTED_FORMULA = "a * exp(b * target_sparsity)"


class NoCalibration(ValueError):
    pass


def factor_from_threshold(threshold: float, max_kv_len: int) -> float:
    return float(threshold) * float(max_kv_len)


def factor_from_curve(a: float, b: float, target_sparsity: float) -> float:
    if a is None or b is None or not (math.isfinite(a) and math.isfinite(b)):
        raise NoCalibration("target_sparsity needs calibration coefficients a, b; "
                            "use threshold for a calibration-free setting")
    return float(a) * math.exp(float(b) * float(target_sparsity))


def lam(factor: float, max_kv_len: int) -> float:
    return float(factor) / float(max_kv_len)


def lambda_threshold(threshold: float, max_kv_len: int) -> float:
    return lam(factor_from_threshold(threshold, max_kv_len), max_kv_len)


def lambda_curve(a: float, b: float, target_sparsity: float, max_kv_len: int) -> float:
    return lam(factor_from_curve(a, b, target_sparsity), max_kv_len)
