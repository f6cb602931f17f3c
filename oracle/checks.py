"""Test-side helpers built on the oracle -- TEST INFRASTRUCTURE ONLY.

* routing margins: redraw input rows until every token's top-(k+1) router
  logits are separated by a margin, so that fp32 logits on the device (a
  different summation order) select the same experts in the same order;
* the layer-output comparison that allows for ambiguous int8 rounding
  decisions: where an intermediate SwiGLU activation lies within `delta` (in
  units of its quantisation step) of a rounding boundary, both neighbouring
  codes are correct results of the fp32 rule, and the expected output may be
  the oracle's with any set of those codes moved to the other neighbour.
"""
from __future__ import annotations

import numpy as np

from . import router_logits, weight_column


def small_gap_tokens(L: np.ndarray, k: int, margin: float) -> np.ndarray:
    E = L.shape[1]
    m = min(k + 1, E)
    top = -np.sort(-L, axis=1)[:, :m]
    gaps = top[:, :-1] - top[:, 1:]
    return np.nonzero((gaps < margin).any(axis=1))[0]


def margin_inputs(x, Wr, bias, k, seed, margin=1e-3, redraw=None, max_rounds=100):
    """x with every token's routing decided by at least `margin` in fp64."""
    import synth

    redraw = redraw or synth.redraw_rows
    for attempt in range(max_rounds):
        L = router_logits(x.numpy() if hasattr(x, "numpy") else x, Wr, bias)
        bad = small_gap_tokens(L, k, margin)
        if bad.size == 0:
            return x
        x = redraw(x, bad, seed, attempt)
    raise RuntimeError("could not reach the routing margin")


def compare_layer_output(y_dev, ref, down_codes, down_scales, bits, tol=2e-3, delta=1e-3, rms=None):
    """Check y_dev [n, H] against oracle.layer(..., detail=True) output `ref`.

    Returns (max_err_over_rms, n_tokens_needing_alternative_codes, n_alternative_codes).
    Raises AssertionError when a row cannot be matched within tol * RMS.
    """
    y_ref = ref["y"].astype(np.float64)
    y_dev = np.asarray(y_dev, np.float64)
    if rms is None:
        rms = float(np.sqrt(np.mean(y_ref**2)))
    bound = tol * rms
    err = np.abs(y_dev - y_ref)
    rows = np.nonzero(err.max(axis=1) > bound)[0]
    n_alt = 0
    H = y_ref.shape[1]
    for r in rows:
        resid = y_dev[r] - y_ref[r]
        cands = []
        for j in range(ref["idx"].shape[1]):
            e = int(ref["idx"][r, j])
            for i in np.nonzero(ref["hdist"][r, j] < delta)[0]:
                s = float(ref["sh"][r, j, i // 32])
                ratio = float(ref["h"][r, j, i]) / s
                step = 1.0 if ratio > ref["qh"][r, j, i] else -1.0
                col = weight_column(down_codes[e], down_scales[e], bits, H, int(i))
                cands.append(float(ref["w"][r, j]) * step * s * col)
        used = set()
        while np.abs(resid).max() > bound:
            best, best_norm = None, float(np.dot(resid, resid))
            for c_i, c in enumerate(cands):
                if c_i in used:
                    continue
                d = resid - c
                nn = float(np.dot(d, d))
                if nn < best_norm:
                    best, best_norm = c_i, nn
            if best is None:
                break
            used.add(best)
            resid = resid - cands[best]
        assert np.abs(resid).max() <= bound, (
            f"row {r}: max |y - oracle| = {np.abs(resid).max():.3e} > {bound:.3e} "
            f"after {len(used)} alternative roundings ({len(cands)} candidates)")
        err[r] = np.abs(resid)
        n_alt += len(used)
    return float(err.max() / rms), int(rows.size), n_alt
