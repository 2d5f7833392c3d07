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


def test_gradient_tolerance_rejects_plausible_mistakes():
    """The per-row bound used by the GPU parity test (2 x the rounding scales + 1% of the row
    norm) separates a correct gradient from one with a dropped D term, a missing scale, a
    transposed dS or a sign error, all planted here in a copy of the oracle's arithmetic."""
    from oracle.backward import _head_backward

    cfg, q, k, v, do = _inputs(1, 1, 1, 300, 300, 64, 95, BF16, True)
    qd, kd, vd, dod = (oracle.bits_to_double(x, BF16).reshape(300, 64) for x in (q, k, v, do))
    dq, dk, dv, o, lse, (eq, ek, ev) = _head_backward(qd, kd, vd, dod, True, cfg.scale,
                                                      stored_dtype=BF16, unit=2.0 ** -7)

    def passes(got, ref, scales):
        err = np.linalg.norm(got - ref, axis=1)
        return bool(np.all(err <= 2.0 * scales + 1e-2 * np.linalg.norm(ref, axis=1) + 1e-6))

    assert passes(dq, dq, eq) and passes(dk, dk, ek) and passes(dv, dv, ev)
    # the same algebra with one planted mistake each
    s = cfg.scale * (qd @ kd.T)
    i = np.arange(300)[:, None]
    s = np.where(np.arange(300)[None, :] <= i, s, -np.inf)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    dp = dod @ vd.T
    D = (dod * o).sum(axis=1, keepdims=True)
    assert not passes(cfg.scale * ((p * dp) @ kd), dq, eq)                    # D dropped
    assert not passes((p * (dp - D)) @ kd, dq, eq)                             # scale missing
    assert not passes(cfg.scale * ((p * (D - dp)) @ kd), dq, eq)               # sign of dS
    assert not passes(cfg.scale * ((p * (dp - D)) @ qd), dk, ek)               # dS not transposed
    assert not passes(p @ dod, dv, ev)                                         # P instead of P^T
