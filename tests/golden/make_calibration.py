"""Choose the synthetic workloads' noise scales and record the achieved alpha.

Run from the repository root:  python tests/golden/make_calibration.py
It writes tests/golden/calibration.json.  The values it prints are then the
constants in workloads/synth.py (SPECS); tests/test_workloads.py checks that
the two agree and that the achieved mean acceptance is near its target.

The mean acceptance alpha = mean over rows of sum_x min(p, q) is computed with
the CPU oracle only.  Each parameter is found by bisection on a seeded
calibration batch (seed 123, a few sequences), over the parameter that
controls the target/draft agreement:
  * target = 0.9 * draft + N(0, s^2): bisect s (alpha falls as s grows);
  * target = rho * draft + sqrt(1 - rho^2) * N(0, sigma^2): bisect rho.
"""

from __future__ import annotations

import json
import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle.verify import acceptance_rate, row_to_float64  # noqa: E402
from workloads.synth import SPECS, make, with_sizes  # noqa: E402

CAL_SEED = 123


def chain_alpha(spec, n_seq=3):
    w = make(with_sizes(spec, B=n_seq), seed=CAL_SEED)
    vals = [acceptance_rate(row_to_float64(w["target"][b, i], spec.dtype),
                            row_to_float64(w["draft"][b, i], spec.dtype),
                            spec.temperature)
            for b in range(n_seq) for i in range(spec.gamma)]
    return float(np.mean(vals))


def tree_alpha(spec, n_seq=1):
    w = make(with_sizes(spec, B=n_seq), seed=CAL_SEED)
    N = w["target"].shape[1]
    vals = [acceptance_rate(row_to_float64(w["target"][b, i], spec.dtype),
                            row_to_float64(w["draft"][b, i], spec.dtype),
                            spec.temperature)
            for b in range(n_seq) for i in range(0, N, 4)]
    return float(np.mean(vals))


def cascade_alphas(spec, n_seq=2):
    w = make(with_sizes(spec, B=n_seq), seed=CAL_SEED)
    a01, a12 = [], []
    for b in range(n_seq):
        for j in range(spec.gamma1):
            a01.append(acceptance_rate(row_to_float64(w["l1"][b, j], spec.dtype),
                                       row_to_float64(w["l0"][b, j], spec.dtype),
                                       spec.temperature))
        for j in range(spec.gamma2):
            a12.append(acceptance_rate(row_to_float64(w["l2"][b, j], spec.dtype),
                                       row_to_float64(w["l1"][b, j], spec.dtype),
                                       spec.temperature))
    return float(np.mean(a01)), float(np.mean(a12))


def bisect(f, lo, hi, target, increasing, iters=18):
    """Find x in [lo, hi] with f(x) ~ target for a monotone f."""
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if (f(mid) < target) == increasing:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def main():
    out = {}
    # 0.9 * draft + noise: alpha decreases with s
    for name in ("sampling_chain_b32_g8_v32000_bf16",):
        spec = SPECS[name]
        s = bisect(lambda s: chain_alpha(with_sizes(spec, s=s)), 0.05, 4.0,
                   spec.alpha_target, increasing=False)
        s = round(s, 3)
        out[name] = dict(a=spec.a, s=s, alpha=chain_alpha(with_sizes(spec, s=s)))
    # correlation sweep at sigma = 2: alpha increases with rho
    for name in [k for k in SPECS if k.startswith("sampling_chain_b64")]:
        spec = SPECS[name]
        sig = spec.sigma_q

        def at(rho):
            return chain_alpha(with_sizes(spec, a=rho, s=sig * math.sqrt(max(0.0, 1 - rho * rho))))
        rho = round(bisect(at, 0.0, 0.999, spec.alpha_target, increasing=True), 4)
        s = round(sig * math.sqrt(1 - rho * rho), 4)
        out[name] = dict(a=rho, s=s, alpha=at(rho), alpha_at_rho0=at(0.0))
    for name in ("tree_b16_n64_v50257_bf16",):
        spec = SPECS[name]
        s = round(bisect(lambda s: tree_alpha(with_sizes(spec, s=s)), 0.05, 4.0,
                         spec.alpha_target, increasing=False), 3)
        out[name] = dict(a=spec.a, s=s, alpha=tree_alpha(with_sizes(spec, s=s)))
    for name in ("cascade_b128_g8_g4_v128256_bf16",):
        spec = SPECS[name]
        s01 = round(bisect(lambda s: cascade_alphas(with_sizes(spec, s01=s))[0],
                           0.05, 4.0, spec.alpha01_target, increasing=False), 3)
        s12 = round(bisect(lambda s: cascade_alphas(with_sizes(spec, s01=s01, s12=s))[1],
                           0.05, 4.0, spec.alpha12_target, increasing=False), 3)
        a01, a12 = cascade_alphas(with_sizes(spec, s01=s01, s12=s12))
        out[name] = dict(a01=spec.a01, s01=s01, a12=spec.a12, s12=s12,
                         alpha01=a01, alpha12=a12)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "calibration.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1, sort_keys=True)
        fh.write("\n")
    print(json.dumps(out, indent=1, sort_keys=True))


if __name__ == "__main__":
    main()
