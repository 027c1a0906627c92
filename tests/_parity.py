"""Parity bars of the GPU tests, and a record of the worst error each test measured.

Bars: max-abs error <= 2e-3 for the bf16 and fp8 paths and for verify, <= 5e-3 for the int8-QK path,
against the oracle (double accumulation), after discounting the rounding of the kernel's bf16
output and nothing else. That rounding is at most half a bf16 ulp of the value: bf16 keeps 8
significant bits, so a value x with 2^e <= |x| < 2^(e+1) is stored with an error up to 2^(e-8),
which is between 2^-9 |x| and 2^-8 |x|. Even an exact kernel misses 2e-3 by that much once |o| >= 1,
so the discount is that bound, computed for each element (for the larger of the two magnitudes, as
the kernel's unrounded value may sit in the binade above the oracle's).

The fp32 outputs of the verify partials carry no output rounding and are held to the bar raw.

Every comparison records its raw max-abs error and its excess over the discount under the running
test's id; when PKV_PARITY_LOG names a file, the session writes the records there as JSON.
"""
from __future__ import annotations

import json
import os

import numpy as np

import workloads as W

TOL_BF16 = 2e-3
TOL_INT8 = 5e-3

RECORDS: dict = {}


def _test_id() -> str:
    cur = os.environ.get("PYTEST_CURRENT_TEST", "?")
    return cur.rsplit(" (", 1)[0]


def record(raw: float, excess: float, tol: float, what: str = "") -> None:
    key = _test_id() + (f" [{what}]" if what else "")
    r = RECORDS.setdefault(key, {"max_abs": 0.0, "excess": -1.0, "tol": tol})
    r["max_abs"] = max(r["max_abs"], float(raw))
    r["excess"] = max(r["excess"], float(excess))


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp of |x|: 2^(e - 8) for 2^e <= |x| < 2^(e+1); 0 for x = 0."""
    m = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(m)  # m = f 2^e with 0.5 <= f < 1, so 2^(e-1) <= m < 2^e
    return np.where(m > 0, np.ldexp(1.0, e - 9), 0.0)


def close(gpu_bf16_u16, ref, tol: float, what: str = "") -> float:
    """Asserts max over elements of |gpu - ref| - half_ulp(max(|gpu|, |ref|)) <= tol; returns it."""
    g = W.bf16_bits_to_f32(gpu_bf16_u16).astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert not np.isnan(g).any(), f"NaN in GPU output at {np.argwhere(np.isnan(g))[:4].tolist()}"
    diff = np.abs(g - ref)
    err = diff - half_ulp_bf16(np.maximum(np.abs(g), np.abs(ref)))
    i = np.unravel_index(int(np.argmax(err)), err.shape)
    worst = float(err[i])
    record(float(diff.max()), worst, tol, what)
    assert worst <= tol, (f"error beyond the output rounding {worst:.3e} > {tol} at {tuple(int(x) for x in i)}: "
                          f"gpu {g[i]:.6f} oracle {ref[i]:.6f}; max |diff| {diff.max():.3e}, "
                          f"mean |diff| {diff.mean():.3e}")
    return worst


def close_raw(a, b, tol: float, what: str = "") -> float:
    """fp32 values (no output rounding): asserts max |a - b| <= tol; returns it."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    assert not np.isnan(a).any() and not np.isnan(b).any(), "NaN in comparison"
    d = float(np.abs(a - b).max()) if a.size else 0.0
    record(d, d, tol, what)
    assert d <= tol, f"max |diff| {d:.3e} > {tol}"
    return d


def dump(path: str) -> None:
    with open(path, "w") as f:
        json.dump(dict(sorted(RECORDS.items())), f, indent=1)
