"""Pins of the fp64 backward oracle (oracle/backward.py) against things other than itself:
finite differences of the pinned forward oracle, closed forms and invariants of the softmax
Jacobian ("FlashAttention Explained", section "Backward Pass: Recomputation Beats Storage")."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from oracle.backward import attention_backward

F16, BF16 = "f16", "bf16"


def _inputs(B, Hq, Hkv, Nq, Nkv, d, seed, dtype=F16, causal=False):
    cfg = syn.PrefillConfig("bwd", B, Hq, Hkv, Nq, Nkv, d, dtype, causal, seed)
    q, k, v = cfg.host_inputs()
    do = syn.host_normal_bits((B, Hq, Nq, d), seed + 7, dtype)
    return cfg, q, k, v, do


def _loss(q, k, v, dod, cfg):
    """sum(dO o O) with O from the C forward oracle (pinned separately)."""
    o, _ = oracle.attention(q, k, v, cfg.dtype, cfg.B, cfg.Hq, cfg.Hkv, cfg.N_q, cfg.N_kv, cfg.d,
                            cfg.causal, cfg.scale)
    return float((dod * o).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("G", [1, 2])
def test_gradients_match_finite_differences_of_the_forward(causal, G):
    """Central differences over one fp16 ulp of an input element (exactly representable
    neighbours), through the C forward oracle, against the analytic gradients."""
    cfg, q, k, v, do = _inputs(1, 2 * G, 2, 5, 7, 4, 40 + G, F16, causal)
    dq, dk, dv, _, _ = attention_backward(q, k, v, do, F16, 1, 2 * G, 2, 5, 7, 4, causal, cfg.scale,
                                          exact_o=True)
    dod = oracle.bits_to_double(do, F16)
    grads = {"q": dq, "k": dk, "v": dv}
    arrays = {"q": q, "k": k, "v": v}
    rng = np.random.default_rng(G + 10 * causal)
    for name in ("q", "k", "v"):
        arr = arrays[name]
        for _ in range(12):
            idx = tuple(rng.integers(0, s) for s in arr.shape)
            x0 = arr[idx]
            up, dn = arr.copy(), arr.copy()
            up[idx] = np.uint16(x0 + 1) if oracle.bits_to_double(np.uint16(x0), F16) >= 0 else np.uint16(x0 - 1)
            dn[idx] = np.uint16(x0 - 1) if oracle.bits_to_double(np.uint16(x0), F16) > 0 else np.uint16(x0 + 1)
            xu = float(oracle.bits_to_double(np.uint16(up[idx]), F16))
            xd = float(oracle.bits_to_double(np.uint16(dn[idx]), F16))
            args = {n: (up if n == name else arrays[n]) for n in arrays}
            lu = _loss(args["q"], args["k"], args["v"], dod, cfg)
            args = {n: (dn if n == name else arrays[n]) for n in arrays}
            ld = _loss(args["q"], args["k"], args["v"], dod, cfg)
            fd = (lu - ld) / (xu - xd)
            an = grads[name][idx]
            assert abs(fd - an) <= 2e-4 + 2e-3 * abs(an), (name, idx, fd, an)


def test_output_and_lse_agree_with_the_forward_oracle():
    cfg, q, k, v, do = _inputs(2, 4, 2, 33, 47, 16, 50, BF16, True)
    _, _, _, o, lse = attention_backward(q, k, v, do, BF16, 2, 4, 2, 33, 47, 16, True, cfg.scale)
    of, lf = oracle.attention(q, k, v, BF16, 2, 4, 2, 33, 47, 16, True, cfg.scale)
    np.testing.assert_allclose(o, of, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lf, rtol=0, atol=1e-12)


def test_equal_value_rows_give_zero_query_and_key_gradients():
    """If every value row is the same vector, O does not depend on Q or K."""
    cfg, q, k, v, do = _inputs(1, 2, 1, 20, 30, 8, 60, BF16)
    v[:] = v[:, :, :1, :]
    dq, dk, dv, _, _ = attention_backward(q, k, v, do, BF16, 1, 2, 1, 20, 30, 8, False, cfg.scale)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    assert np.abs(dv).max() > 0.1


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_jacobian_invariants(causal):
    """Rows of P sum to one: sum_j dV_j = sum of dO over rows with a visible key; each row of
    dS sums to zero: sum_j dK_j = 0, and with equal key rows dQ = 0."""
    cfg, q, k, v, do = _inputs(1, 2, 2, 40, 40, 16, 70 + causal, BF16, causal)
    dq, dk, dv, _, lse = attention_backward(q, k, v, do, BF16, 1, 2, 2, 40, 40, 16, causal,
                                            cfg.scale, exact_o=True)
    dod = oracle.bits_to_double(do, BF16).reshape(1, 2, 40, 16)
    live = np.isfinite(lse)[..., None]
    np.testing.assert_allclose(dv.sum(axis=2), (dod * live).sum(axis=2), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, rtol=0, atol=1e-11)
    k[:] = k[:, :, :1, :]
    dq, _, _, _, _ = attention_backward(q, k, v, do, BF16, 1, 2, 2, 40, 40, 16, causal, cfg.scale,
                                        exact_o=True)
    assert np.abs(dq).max() < 1e-12


def test_grouped_heads_sum_their_contributions():
    cfg, q, k, v, do = _inputs(1, 4, 1, 25, 25, 8, 80, BF16, True)
    _, dk, dv, _, _ = attention_backward(q, k, v, do, BF16, 1, 4, 1, 25, 25, 8, True, cfg.scale)
    parts = [attention_backward(q, k, v, do, BF16, 1, 4, 1, 25, 25, 8, True, cfg.scale, heads=[h])
             for h in range(4)]
    np.testing.assert_allclose(sum(p[1] for p in parts), dk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(sum(p[2] for p in parts), dv, rtol=0, atol=1e-12)


def test_one_row_problem_gives_that_rows_query_gradient():
    """dQ_i = scale * sum_j P_ij (dP_ij - D_i) K_j involves only row i's q, do, its O and L and
    the keys it sees, so one query against its visible keys without a mask gives the same row of
    dQ and the same rounding scales as the whole causal problem (the reduction the large-size
    GPU test samples rows with)."""
    B, Hq, Hkv, N, d, dt = 1, 4, 2, 300, 64, "bf16"
    cfg = syn.PrefillConfig("row", B, Hq, Hkv, N, N, d, dt, True, 5)
    q, k, v = cfg.host_inputs()
    do = syn.host_normal_bits((B, Hq, N, d), 12, dt)
    full = attention_backward(q, k, v, do, dt, B, Hq, Hkv, N, N, d, True, cfg.scale,
                              error_scales=True)
    G = Hq // Hkv
    for h in range(Hq):
        for i in (0, 1, 127, 128, 171, N - 1):
            r = attention_backward(q[:, h:h + 1, i:i + 1], k[:, h // G:h // G + 1, :i + 1],
                                   v[:, h // G:h // G + 1, :i + 1], do[:, h:h + 1, i:i + 1], dt,
                                   1, 1, 1, 1, i + 1, d, False, cfg.scale, error_scales=True)
            np.testing.assert_allclose(r[0][0, 0, 0], full[0][0, h, i], rtol=0, atol=1e-14)
            np.testing.assert_allclose(r[5].row[0][0, 0, 0], full[5].row[0][0, h, i], rtol=1e-12)
            np.testing.assert_allclose(r[5].elem[0][0, 0, 0], full[5].elem[0][0, h, i],
                                       rtol=1e-12, atol=1e-300)


def test_stored_output_changes_only_the_d_term():
    """D from O rounded to the storage type: dV is unchanged, and dQ, dK move only by the
    rounding of D (dS changes by -P * dD)."""
    cfg, q, k, v, do = _inputs(1, 2, 2, 30, 30, 16, 90, BF16, True)
    ex = attention_backward(q, k, v, do, BF16, 1, 2, 2, 30, 30, 16, True, cfg.scale, exact_o=True)
    st = attention_backward(q, k, v, do, BF16, 1, 2, 2, 30, 30, 16, True, cfg.scale)
    np.testing.assert_array_equal(ex[2], st[2])
    assert 0 < np.abs(ex[0] - st[0]).max() < 1e-2 * np.abs(ex[0]).max()
    # the rounded O the oracle uses is the storage rounding of its exact O
    o_bits = oracle.round_to_storage(ex[3], BF16)
    assert np.abs(oracle.bits_to_double(o_bits, BF16) - ex[3]).max() <= 2.0 ** -8 * np.abs(ex[3]).max()


def _head(dtype, causal, seed, Nq=300, Nkv=300, d=64):
    from oracle.backward import _head_backward, storage_unit

    cfg, q, k, v, do = _inputs(1, 1, 1, Nq, Nkv, d, seed, dtype, causal)
    qd, kd, vd, dod = (oracle.bits_to_double(x, dtype).reshape(-1, d) for x in (q, k, v, do))
    unit, tiny = storage_unit(dtype)
    res = _head_backward(qd, kd, vd, dod, causal, cfg.scale, stored_dtype=dtype, unit=unit,
                         tiny=tiny)
    return cfg, (qd, kd, vd, dod), res


def _rnd(x, dtype):
    x = np.ascontiguousarray(x, dtype=np.float64)
    return oracle.bits_to_double(oracle.round_to_storage(x, dtype), dtype)


def _kernel_like_gradients(qd, kd, vd, dod, causal, scale, dtype, given=None):
    """The pages' forward and backward with every rounding a 16-bit kernel makes, in fp64
    otherwise: P unnormalised and rounded before P V, O rounded, L = m + ln l (or O and L as
    given); then P from L, D from the stored O, P and dS rounded before their products, the
    gradients rounded."""
    Nq, Nkv = qd.shape[0], kd.shape[0]
    s = scale * (qd @ kd.T)
    if causal:
        s = np.where(np.arange(Nkv)[None, :] <= np.arange(Nq)[:, None] + (Nkv - Nq), s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    live = np.isfinite(m)
    if given is None:
        pt = np.where(live, np.exp(s - np.where(live, m, 0.0)), 0.0)
        lsum = pt.sum(axis=1, keepdims=True)
        o = _rnd(np.where(live, (_rnd(pt, dtype) @ vd) / np.where(live, lsum, 1.0), 0.0), dtype)
        L = np.where(live, m + np.log(np.where(live, lsum, 1.0)), -np.inf)
    else:
        o, L = given
        L = L.astype(np.float32).astype(np.float64)[:, None]
    p = np.where(live, np.exp(s - np.where(live, L, 0.0)), 0.0)
    ds = p * (dod @ vd.T - (dod * o).sum(axis=1, keepdims=True))
    dv = _rnd(_rnd(p, dtype).T @ dod, dtype)
    dsr = _rnd(ds, dtype)
    return _rnd(scale * (dsr @ kd), dtype), _rnd(scale * (dsr.T @ qd), dtype), dv


@pytest.mark.parametrize("given", [False, True], ids=["forward_o", "oracle_o"])
@pytest.mark.parametrize("dtype,causal", [(BF16, True), (F16, True), (BF16, False), (F16, False)])
def test_gradient_bounds_hold_for_a_kernel_with_the_pages_roundings(dtype, causal, given):
    """The row and element bounds of the GPU parity check contain the gradients of a model of
    the kernel's arithmetic (every rounding to 16 bits it makes, fp64 elsewhere), for D formed
    from a forward kernel's stored O and from the oracle's stored O handed over: the bounds are
    not tighter than the rounding they describe."""
    from parity import grad_violations

    cfg, (qd, kd, vd, dod), res = _head(dtype, causal, 97 + causal, 260, 300, 64)
    o_given = _rnd(res[3], dtype)
    got = _kernel_like_gradients(qd, kd, vd, dod, causal, cfg.scale, dtype,
                                 (o_given, res[4]) if given else None)
    sc = res[5]
    rows, elems = (sc.given_row, sc.given_elem) if given else (sc.row, sc.elem)
    for g, ref, er, ee in zip(got, res[:3], rows, elems):
        r_row, r_el = grad_violations(g, ref, er, ee, dtype)
        assert r_row.max() <= 1.0 and r_el.max() <= 1.0, (r_row.max(), r_el.max())
        assert r_el.max() > 1e-3            # the model does round: the errors are not zero


@pytest.mark.parametrize("given", [False, True], ids=["forward_o", "oracle_o"])
def test_element_bound_catches_what_the_row_bound_lets_through(given):
    """One corrupted element of dQ, and one corrupted channel of dQ, dK and dV across every
    row, each half as large as the row bound allows: the row check passes all of them, the
    element check fails them.  With D from a forward kernel's O the element bound of dK holds
    the worst case of the forward's P rounding, so it catches most corrupted rows, not all."""
    from parity import GRAD_FLOOR, GRAD_RTOL_ROW, GRAD_SCALE_FACTOR, grad_violations

    cfg, _, (dq, dk, dv, o, lse, sc) = _head(BF16, True, 95)
    rows, elems = (sc.given_row, sc.given_elem) if given else (sc.row, sc.elem)

    def row_allow(ref, e):
        return GRAD_SCALE_FACTOR * e + GRAD_RTOL_ROW * np.linalg.norm(ref, axis=1) + GRAD_FLOOR

    # one element
    bad = dq.copy()
    r, c = 217, 13
    bad[r, c] += 0.5 * row_allow(dq, rows[0])[r]
    r_row, r_el = grad_violations(bad, dq, rows[0], elems[0], BF16)
    assert r_row.max() <= 1.0 and r_el.max() > 1.0, (r_row.max(), r_el.max())
    # one channel of every row (key rows that no query sees have a zero gradient and bound)
    for which, g, c in ((0, dq, 3), (1, dk, 40), (2, dv, 5)):
        bad = g.copy()
        bad[:, c] -= 0.5 * row_allow(g, rows[which])
        r_row, r_el = grad_violations(bad, g, rows[which], elems[which], BF16)
        live = np.abs(g).sum(axis=1) > 0
        caught = (r_el[live, c] > 1.0).mean()
        assert r_row.max() <= 1.0 and caught >= (0.8 if which == 1 and not given else 1.0), \
            (which, r_row.max(), caught)


def test_gradient_tolerance_rejects_plausible_mistakes():
    """The bounds used by the GPU parity test (row and element checks, D from a forward
    kernel's O or from the oracle's) separate a correct gradient from one with a dropped D
    term, a missing scale, a transposed dS or a sign error, all planted here in a copy of the
    oracle's arithmetic."""
    from parity import grad_violations

    cfg, (qd, kd, vd, dod), (dq, dk, dv, o, lse, sc) = _head(BF16, True, 95)

    def passes(got, ref, which):
        for rows, elems in ((sc.row, sc.elem), (sc.given_row, sc.given_elem)):
            r_row, r_el = grad_violations(got, ref, rows[which], elems[which], BF16)
            if r_row.max() > 1.0 or r_el.max() > 1.0:
                return False
        return True

    assert passes(dq, dq, 0) and passes(dk, dk, 1) and passes(dv, dv, 2)
    # the same algebra with one planted mistake each
    s = cfg.scale * (qd @ kd.T)
    i = np.arange(300)[:, None]
    s = np.where(np.arange(300)[None, :] <= i, s, -np.inf)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    dp = dod @ vd.T
    D = (dod * o).sum(axis=1, keepdims=True)
    assert not passes(cfg.scale * ((p * dp) @ kd), dq, 0)                    # D dropped
    assert not passes((p * (dp - D)) @ kd, dq, 0)                             # scale missing
    assert not passes(cfg.scale * ((p * (D - dp)) @ kd), dq, 0)               # sign of dS
    assert not passes(cfg.scale * ((p * (dp - D)) @ qd), dk, 1)               # dS not transposed
    assert not passes(p @ dod, dv, 2)                                         # P instead of P^T
