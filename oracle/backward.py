"""fp64 oracle of the attention backward pass (TEST INFRASTRUCTURE ONLY).

Only the test suite, the smoke check and the CPU-baseline leg of the benchmark use this
module; the CUDA library shares nothing with it.

The exact gradient of O = softmax(scale * Q K^T + mask) V for an incoming gradient dO, in the
order the pages state it ("FlashAttention Explained", section "Backward Pass: Recomputation
Beats Storage"):

    P  = softmax(S),  S = scale * Q K^T (masked entries -inf)      (the forward definition)
    dV = P^T dO
    dP = dO V^T
    dS = P o (dP - D),   D_i = rowsum(dO_i o O_i)
    dQ = scale * dS K
    dK = scale * dS^T Q

for each (batch, query head), with O = P V computed here in fp64.  D is formed either from
that exact O (the exact gradient) or, by default, from O as the forward stores it: rounded to
the storage type, since the backward of the pages consumes the saved output.  The two differ
only by that rounding, which matters where dP - D nearly cancels (rows that see few keys).  Grouped-query heads map query head h to key/value head h / (Hq / Hkv); the
gradients of one key/value head are the sums over its query heads.  Masks are those of the
forward oracle (causal bottom-right aligned; a row with no visible key has P = 0 and
contributes nothing).  numpy's matmul is the only library step.
"""
import numpy as np

from . import bits_to_double, round_to_storage


def _head_backward(q, k, v, do, causal, scale, window=None, stored_dtype=None, unit=None):
    """One head, fp64 arrays q [Nq, d], k/v [Nkv, d], do [Nq, d] -> (dq, dk, dv, o, lse).
    stored_dtype: round O to this storage type before forming D (None: exact O).
    unit: if given, also return per-row rounding scales (see below) for this unit roundoff."""
    Nq, Nkv = q.shape[0], k.shape[0]
    s = scale * (q @ k.T)
    if causal or window is not None:
        i = np.arange(Nq)[:, None] + (Nkv - Nq)
        j = np.arange(Nkv)[None, :]
        vis = j <= i
        if window is not None:
            vis &= (i - j) <= window
        s = np.where(vis, s, -np.inf)
    m = s.max(axis=1, keepdims=True) if Nkv else np.full((Nq, 1), -np.inf)
    live = np.isfinite(m[:, 0])
    e = np.where(live[:, None], np.exp(s - np.where(live[:, None], m, 0.0)), 0.0)
    l = e.sum(axis=1, keepdims=True)
    p = np.where(live[:, None], e / np.where(l > 0, l, 1.0), 0.0)
    o = p @ v
    lse = np.where(live, m[:, 0] + np.log(np.where(l[:, 0] > 0, l[:, 0], 1.0)), -np.inf)
    dv = p.T @ do
    dp = do @ v.T
    o_used = o if stored_dtype is None else bits_to_double(round_to_storage(o, stored_dtype),
                                                            stored_dtype)
    D = (do * o_used).sum(axis=1, keepdims=True)
    ds = p * (dp - D)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    if unit is None:
        return dq, dk, dv, o, lse
    # Rounding scales of a kernel that follows the pages' algorithm: P and dS rounded to the
    # storage type before their products (relative `unit` per term), and D formed from a stored O
    # that may differ from the exact one by one unit of the storage type in each element
    # (|dD_i| <= unit * sum_c |dO_ic O_ic|; dS moves by -P dD, i.e. dQ_i by -scale dD_i (P K)_i).
    nk = np.linalg.norm(k, axis=1)
    nq = np.linalg.norm(q, axis=1)
    ndo = np.linalg.norm(do, axis=1)
    dd = unit * np.abs(do * o).sum(axis=1)
    eq = scale * (unit * (np.abs(ds) @ nk) + dd * np.linalg.norm(p @ k, axis=1))
    ek = scale * (unit * (np.abs(ds).T @ nq) + p.T @ (dd * nq))
    ev = unit * (p.T @ ndo)
    return dq, dk, dv, o, lse, (eq, ek, ev)


def attention_backward(q, k, v, do, dtype, B, Hq, Hkv, Nq, Nkv, d, causal, scale,
                       window=None, heads=None, exact_o=False, error_scales=False):
    """Gradients of every (or the listed) query head.

    q, do: uint16 storage bits [B, Hq, Nq, d]; k, v: [B, Hkv, Nkv, d].
    heads: optional list of flat query heads b * Hq + h to compute (their key/value head's dK
    and dV then hold only those query heads' contributions).
    exact_o: form D from the exact fp64 O (the exact gradient) instead of O rounded to the
    storage type as the forward saves it.
    error_scales: also return (eq [B,Hq,Nq], ek, ev [B,Hkv,Nkv]), per-row rounding scales of a
    kernel that rounds P and dS to the storage type and forms D from a stored O that may differ
    from the exact one by a unit of the storage type (unit = one ulp at 1: 2^-7 bf16, 2^-10 f16).
    Returns dq [B, Hq, Nq, d], dk, dv [B, Hkv, Nkv, d], o [B, Hq, Nq, d], lse [B, Hq, Nq]
    (float64; entries of heads not computed are NaN for dq/o/lse).
    """
    qd = bits_to_double(np.asarray(q), dtype).reshape(B, Hq, Nq, d)
    kd = bits_to_double(np.asarray(k), dtype).reshape(B, Hkv, Nkv, d)
    vd = bits_to_double(np.asarray(v), dtype).reshape(B, Hkv, Nkv, d)
    dod = bits_to_double(np.asarray(do), dtype).reshape(B, Hq, Nq, d)
    G = Hq // Hkv
    dq = np.full((B, Hq, Nq, d), np.nan)
    o = np.full((B, Hq, Nq, d), np.nan)
    lse = np.full((B, Hq, Nq), np.nan)
    dk = np.zeros((B, Hkv, Nkv, d))
    dv = np.zeros((B, Hkv, Nkv, d))
    unit = (2.0 ** -7 if str(dtype).lower().startswith("b") else 2.0 ** -10) if error_scales else None
    eq = np.full((B, Hq, Nq), np.nan)
    ek = np.zeros((B, Hkv, Nkv))
    ev = np.zeros((B, Hkv, Nkv))
    todo = range(B * Hq) if heads is None else heads
    for bh in todo:
        b, h = divmod(int(bh), Hq)
        hk = h // G
        res = _head_backward(qd[b, h], kd[b, hk], vd[b, hk], dod[b, h], causal, scale, window,
                             None if exact_o else dtype, unit)
        gq, gk, gv, go, gl = res[:5]
        dq[b, h], o[b, h], lse[b, h] = gq, go, gl
        dk[b, hk] += gk
        dv[b, hk] += gv
        if error_scales:
            eq[b, h] = res[5][0]
            ek[b, hk] += res[5][1]
            ev[b, hk] += res[5][2]
    if error_scales:
        return dq, dk, dv, o, lse, (eq, ek, ev)
    return dq, dk, dv, o, lse
