"""Parity contract between the CUDA path and the fp64 oracle.

Forward and decode, per row i of O (bf16/fp16 output, fp32 accumulation):
  * max_j |O_gpu[i, j] - O_ref[i, j]|   <= 1e-2 (+ half an output unit of O_ref[i, j], when
                                            the output type is given: the final rounding of O
                                            alone reaches 1e-2 once |O| >= 2 in bf16)
  * ||O_gpu[i] - O_ref[i]||_2           <= 2e-2 * ||O_ref[i]||_2
  * |LSE_gpu[i] - LSE_ref[i]|           <= 1e-3
Rows that see no key must be exactly O = 0 and LSE = -inf on both sides.

Backward (check_grad), for each of dQ, dK, dV, with the oracle's rounding scales for one unit
of the storage type (oracle.backward.GradScales):
  * per row:     ||dX_gpu[r] - dX_ref[r]||_2 <= 2 * e_row[r] + 1e-2 * ||dX_ref[r]||_2 + 1e-6
  * per element: |dX_gpu[r, c] - dX_ref[r, c]| <= 2 * e_elem[r, c] + unit * |dX_ref[r, c]|
                                                  + tiny + 1e-6
where unit and tiny are the storage type's ulp at 1 and subnormal spacing (the second term
covers the gradient's own final rounding) and 1e-6 is a floor for fp32 accumulation.
"""
import numpy as np

ATOL_O = 1e-2
RTOL_ROW = 2e-2
ATOL_LSE = 1e-3

GRAD_SCALE_FACTOR = 2.0
GRAD_RTOL_ROW = 1e-2
GRAD_FLOOR = 1e-6

# (ulp at 1, subnormal spacing) of the 16-bit output types
UNITS = {"bf16": (2.0 ** -7, 2.0 ** -133), "f16": (2.0 ** -10, 2.0 ** -24)}


def check_rows(o_gpu, lse_gpu, o_ref, lse_ref, what="", dtype=None):
    o_gpu = np.asarray(o_gpu, dtype=np.float64).reshape(len(lse_ref), -1)
    o_ref = np.asarray(o_ref, dtype=np.float64).reshape(len(lse_ref), -1)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64).reshape(-1)
    lse_ref = np.asarray(lse_ref, dtype=np.float64).reshape(-1)
    assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
    empty = ~np.isfinite(lse_ref)
    if empty.any():
        assert np.all(lse_gpu[empty] == -np.inf), f"{what}: rows without keys must have LSE=-inf"
        assert np.all(o_gpu[empty] == 0.0), f"{what}: rows without keys must have O=0"
    live = ~empty
    og, orf = o_gpu[live], o_ref[live]
    assert np.all(np.isfinite(og)), f"{what}: non-finite O"
    assert np.all(np.isfinite(lse_gpu[live])), f"{what}: non-finite LSE"
    err = np.abs(og - orf)
    if dtype is not None:
        unit, tiny = UNITS[dtype]
        err = np.maximum(err - (0.5 * unit * np.abs(orf) + 0.5 * tiny), 0.0)
    row_max = err.max(axis=1) if og.size else np.zeros(0)
    row_l2 = np.linalg.norm(og - orf, axis=1)
    ref_l2 = np.linalg.norm(orf, axis=1)
    lse_err = np.abs(lse_gpu[live] - lse_ref[live])
    idx = np.nonzero(live)[0]
    bad_abs = np.nonzero(row_max > ATOL_O)[0]
    bad_rel = np.nonzero(row_l2 > RTOL_ROW * ref_l2)[0]
    bad_lse = np.nonzero(lse_err > ATOL_LSE)[0]
    msg = []
    if len(bad_abs):
        w = bad_abs[np.argmax(row_max[bad_abs])]
        msg.append(f"max|dO| {row_max[w]:.3e} at row {idx[w]} ({len(bad_abs)} rows)")
    if len(bad_rel):
        w = bad_rel[np.argmax(row_l2[bad_rel] / np.maximum(ref_l2[bad_rel], 1e-300))]
        msg.append(f"row-L2 {row_l2[w]:.3e} vs {RTOL_ROW}*{ref_l2[w]:.3e} at row {idx[w]} ({len(bad_rel)} rows)")
    if len(bad_lse):
        w = bad_lse[np.argmax(lse_err[bad_lse])]
        msg.append(f"|dLSE| {lse_err[w]:.3e} at row {idx[w]} ({len(bad_lse)} rows)")
    assert not msg, f"{what}: " + "; ".join(msg)
    return {
        "rows": int(len(lse_ref)),
        "max_abs": float(row_max.max()) if row_max.size else 0.0,
        "max_rel_l2": float((row_l2 / np.maximum(ref_l2, 1e-300)).max()) if row_l2.size else 0.0,
        "max_lse": float(lse_err.max()) if lse_err.size else 0.0,
    }


def grad_violations(got, ref, e_row, e_elem, dtype):
    """(row ratio, element ratio): the largest error / allowed of the row and element checks of
    check_grad (a ratio above 1 fails), without raising."""
    d = ref.shape[-1]
    got = np.asarray(got, dtype=np.float64).reshape(-1, d)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1, d)
    e_row = np.asarray(e_row, dtype=np.float64).reshape(-1)
    e_elem = np.asarray(e_elem, dtype=np.float64).reshape(-1, d)
    unit, tiny = UNITS[dtype]
    diff = np.abs(got - ref)
    row_err = np.linalg.norm(got - ref, axis=1)
    row_ok = GRAD_SCALE_FACTOR * e_row + GRAD_RTOL_ROW * np.linalg.norm(ref, axis=1) + GRAD_FLOOR
    el_ok = GRAD_SCALE_FACTOR * e_elem + unit * np.abs(ref) + tiny + GRAD_FLOOR
    return row_err / row_ok, diff / el_ok


def check_grad(name, got, ref, e_row, e_elem, dtype, what=""):
    """Row and element checks of one gradient (see the module docstring); returns the larger
    of the two worst error / allowed ratios."""
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite {name}"
    r_row, r_el = grad_violations(got, ref, e_row, e_elem, dtype)
    if r_row.size and r_row.max() > 1.0:
        w = int(np.argmax(r_row))
        raise AssertionError(f"{what}: {name} row {w} error / allowed {r_row[w]:.3f} "
                             f"({int((r_row > 1).sum())} rows)")
    if r_el.size and r_el.max() > 1.0:
        w = np.unravel_index(int(np.argmax(r_el)), r_el.shape)
        raise AssertionError(f"{what}: {name} element {tuple(int(x) for x in w)} error / allowed "
                             f"{r_el[w]:.3f} ({int((r_el > 1).sum())} elements)")
    return max(float(r_row.max()) if r_row.size else 0.0, float(r_el.max()) if r_el.size else 0.0)
