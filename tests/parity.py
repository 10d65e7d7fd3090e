"""Parity rule between the CUDA path and the oracle, and test-input shaping that needs the
oracle (near-tie injection).  Test infrastructure only.

Tolerances (from the method's acceptance rule for this layer tail):
  - the residual is bit-exact (one bf16 rounding of one fp32/fp64 add: identical);
  - the selected expert set equals the oracle's in every row whose fp32 k-th minus
    (k+1)-th logit margin exceeds 1e-3 (rows at or below that margin may pick either of
    the near-tied experts and are excluded from the output check when they differ);
  - per row: cosine(out, oracle out) >= 0.9999 and max |out - oracle| <= 2e-2 * RMS(oracle
    row), where "oracle" is the oracle's exact fp64 output before its bf16 rounding and each
    element may also carry the half-ulp rounding of its own bf16 storage (a fp32 sum and a
    fp64 sum that straddle a rounding boundary land on different bf16 neighbours, which at
    a large element is more than 2e-2 * RMS on its own).
"""
import numpy as np

import oracle
from helpers import bf16_decode

MARGIN = 1e-3
COSINE_MIN = 0.9999
MAXERR_REL_RMS = 2e-2


def fp32_margins(logits, k):
    """k-th minus (k+1)-th largest fp32 logit of each row (inf when k == E)."""
    l32 = np.asarray(logits, dtype=np.float32).astype(np.float64)
    out = np.full(l32.shape[0], np.inf)
    if k < l32.shape[1]:
        s = -np.sort(-l32, axis=1)
        out = s[:, k - 1] - s[:, k]
    return out


def _f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_step(bits):
    """The spacing of bf16 values at each element's magnitude (bf16 bits in, float64 out)."""
    v = np.abs((np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32))
    return np.ldexp(1.0, np.floor(np.log2(np.maximum(v, 1e-38))).astype(int) - 7)


def check_parity(got_out, got_res, got_ids, orc, k, rows=None, residual_tol=None):
    """Assert the parity rule; returns a dict of measured figures.  The residual is bit-exact
    unless residual_tol (per element, absolute) is given."""
    R = orc["out"].shape[0] if rows is None else rows
    if residual_tol is None:
        assert np.array_equal(got_res[:R], orc["residual"][:R]), "residual not bit-exact"
    else:
        dres = np.abs(_f64(got_res[:R]) - _f64(orc["residual"][:R]))
        assert (dres <= residual_tol[:R]).all(), "residual off by %g" % dres.max()
    margins = fp32_margins(orc["logits"][:R], k)
    skipped = 0
    worst_cos, worst_err = 1.0, 0.0
    for r in range(R):
        same = set(got_ids[r].tolist()) == set(orc["ids"][r].tolist())
        if margins[r] > MARGIN:
            assert same, "row %d: selection %s != oracle %s (margin %.3g)" % (
                r, sorted(got_ids[r]), sorted(orc["ids"][r]), margins[r])
        elif not same:
            skipped += 1
            continue
        a = bf16_decode(got_out[r])
        b = np.asarray(orc["out_exact"][r], dtype=np.float64)
        assert np.isfinite(a).all(), "row %d: non-finite output" % r
        cos = float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))
        rms = float(np.sqrt(np.mean(b * b)))
        half_ulp = np.ldexp(1.0, np.floor(np.log2(np.maximum(np.abs(a), 1e-38))).astype(int) - 8)
        excess = np.abs(a - b) - half_ulp
        err = float(np.max(np.abs(a - b)))
        worst_cos = min(worst_cos, cos)
        worst_err = max(worst_err, float(np.max(excess)) / max(rms, 1e-300))
        assert cos >= COSINE_MIN, "row %d: cosine %.7f" % (r, cos)
        assert np.max(excess) <= MAXERR_REL_RMS * rms, \
            "row %d: max err %.4g (beyond half an ulp) > 2e-2 * rms %.4g" % (r, err, rms)
    return {"worst_cosine": worst_cos, "worst_err_over_rms": worst_err, "skipped": skipped,
            "min_margin": float(np.min(margins))}


def _row_margin(x_row, res_row, gamma, w_r, eps, k):
    _, n, _ = oracle.add_rmsnorm(x_row[None], res_row[None], gamma, eps)
    l = oracle.router(n, w_r)[0]
    order = sorted(range(len(l)), key=lambda e: (-np.float32(l[e]), e))
    a, b = order[k - 1], order[k]
    return float(np.float32(l[a])) - float(np.float32(l[b])), a, b


def _nudge_once(xrow, m0, res_row, gamma, w_r, eps, k, g, target, tol, iters):
    """One bracket-and-bisect pass along gamma * (W_r[a] - W_r[b]) for the row's current
    k-th (a) and (k+1)-th (b) experts; returns the best row found and its margin."""
    from moe_layer_tail_gb300.inputs import to_bf16_bits
    _, a, b = _row_margin(xrow, res_row, gamma, w_r, eps, k)
    x0 = bf16_decode(xrow)
    v = g * (bf16_decode(w_r[a]) - bf16_decode(w_r[b]))
    v /= np.abs(v).max()

    def trial(alpha):
        xr = to_bf16_bits((x0 + alpha * v)[None])[0]
        return _row_margin(xr, res_row, gamma, w_r, eps, k)[0], xr

    best = (abs(m0 - target), xrow.copy(), m0)
    lo, hi = None, 0.0  # alpha with margin < target (lo) / > target (hi)
    if m0 < target:
        lo, hi = 0.0, None
    step = 1e-4  # the logit gap moves ~20x the step: start far below the target change
    for _ in range(40):  # bracket
        probe = step if m0 < target else -step
        m, xr = trial(probe)
        if abs(m - target) < best[0]:
            best = (abs(m - target), xr, m)
        if (m - target) * (m0 - target) <= 0:
            if m0 < target:
                hi = probe
            else:
                lo = probe
            break
        step *= 2
    if lo is not None and hi is not None:
        for _ in range(iters):
            mid = 0.5 * (lo + hi)
            m, xr = trial(mid)
            if abs(m - target) < best[0]:
                best = (abs(m - target), xr, m)
            if best[0] <= tol:
                break
            if m < target:
                lo = mid
            else:
                hi = mid
    return best[1], best[2]


def inject_near_ties(x, residual, gamma, w_r, eps, k, target=1e-2, tol=1e-4, iters=40):
    """Nudge each row of x (bf16 bits) so that the oracle's fp32 k-th/(k+1)-th logit margin
    is target +- tol.  The nudge is along gamma * (W_r[a] - W_r[b]) for the row's current
    k-th and (k+1)-th experts, sized by bisection (bf16 rounding makes the margin a fine
    staircase in the step size).  Returns the new x and the achieved margins."""
    x = np.array(x, dtype=np.uint16, copy=True)
    got = []
    g = bf16_decode(gamma)
    for r in range(x.shape[0]):
        cur = x[r].copy()
        m_cur = _row_margin(cur, residual[r], gamma, w_r, eps, k)[0]
        for _outer in range(6):  # re-aim at the current k-th/(k+1)-th pair until within tol
            if abs(m_cur - target) <= tol:
                break
            cur, m_cur = _nudge_once(cur, m_cur, residual[r], gamma, w_r, eps, k, g, target,
                                     tol, iters)
        x[r] = cur
        got.append(m_cur)
    return x, np.array(got)
