"""Parity contract between the CUDA path and the fp64 oracle.

Per row i of O (bf16/fp16 output, fp32 accumulation):
  * max_j |O_gpu[i, j] - O_ref[i, j]|   <= 1e-2
  * ||O_gpu[i] - O_ref[i]||_2           <= 2e-2 * ||O_ref[i]||_2
  * |LSE_gpu[i] - LSE_ref[i]|           <= 1e-3
Rows that see no key must be exactly O = 0 and LSE = -inf on both sides.
"""
import numpy as np

ATOL_O = 1e-2
RTOL_ROW = 2e-2
ATOL_LSE = 1e-3


def check_rows(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
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
