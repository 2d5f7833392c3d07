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
from collections import namedtuple

import numpy as np

from . import bits_to_double, round_to_storage

GradScales = namedtuple("GradScales", ["row", "elem", "given_row", "given_elem"])
GradScales.__doc__ = """Rounding scales of the gradients for one unit of the storage type.
row: (eq [..,Nq], ek, ev [..,Nkv]), bounds on the L2 error of each gradient row, and
elem: (eq, ek, ev) with the gradients' own shapes, bounds on each element's error, for a
kernel that forms D from O as a forward kernel stored it; given_row, given_elem: the same
for a kernel handed the oracle's own stored O (and L), so that only fp32 sums separate the
two D's."""


def _head_backward(q, k, v, do, causal, scale, window=None, stored_dtype=None, unit=None,
                   tiny=0.0):
    """One head, fp64 arrays q [Nq, d], k/v [Nkv, d], do [Nq, d] -> (dq, dk, dv, o, lse).
    stored_dtype: round O to this storage type before forming D (None: exact O).
    unit: if given, also return the rounding scales described below for this unit roundoff
    (one ulp at 1 of the storage type); tiny is that type's subnormal spacing."""
    Nq, Nkv = q.shape[0], k.shape[0]
    s = scale * (q @ k.T)
    i = np.arange(Nq)[:, None] + (Nkv - Nq)
    j = np.arange(Nkv)[None, :]
    vis = np.ones((Nq, Nkv), dtype=bool)
    if causal or window is not None:
        vis = j <= i
        if window is not None:
            vis &= (i - j) <= window
        s = np.where(vis, s, -np.inf)
    m = s.max(axis=1, keepdims=True) if Nkv else np.full((Nq, 1), -np.inf)
    live = np.isfinite(m[:, 0])
    vis &= live[:, None]
    e = np.where(live[:, None], np.exp(s - np.where(live[:, None], m, 0.0)), 0.0)
    del s
    l = e.sum(axis=1, keepdims=True)
    p = np.where(live[:, None], e / np.where(l > 0, l, 1.0), 0.0)
    del e
    o = p @ v
    lse = np.where(live, m[:, 0] + np.log(np.where(l[:, 0] > 0, l[:, 0], 1.0)), -np.inf)
    dv = p.T @ do
    dp = do @ v.T
    o_used = o if stored_dtype is None else bits_to_double(round_to_storage(o, stored_dtype),
                                                            stored_dtype)
    D = (do * o_used).sum(axis=1, keepdims=True)
    ds = p * (dp - D)
    del dp
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    if unit is None:
        return dq, dk, dv, o, lse
    # Rounding scales of a kernel that follows the pages' algorithm: P and dS rounded to the
    # storage type before their products, each rounding bounded by `unit` times the rounded
    # value plus `tiny` (the subnormal spacing of fp16; negligible for bf16), and D formed from a
    # stored O that differs from the oracle's by dO_stored, which moves D_i by
    # dd_i = sum_c |dO_ic| |dO_stored_ic|.  A rounded dS_ij (or P_ij) moves each output element
    # by its own term: dQ_ic by scale |K_jc| (unit |dS_ij| + tiny), dK_jc by
    # scale |Q_ic| (unit |dS_ij| + tiny), dV_jc by |dO_ic| (unit P_ij + tiny).  The D error
    # moves the whole row of dS by -P_i dD_i: dQ_i by exactly -scale dD_i (P K)_i, and dK_j by
    # scale sum_i P_ij dD_i Q_i, whose terms' signs are unknown.  Per row the same terms are
    # taken with the L2 norms of the rows of K, Q and dO.
    ads = np.abs(ds)
    del ds
    aq, ak, av, ado = np.abs(q), np.abs(k), np.abs(v), np.abs(do)
    visf = vis.astype(np.float64)
    pk = p @ k
    nk = np.linalg.norm(k, axis=1)
    nq = np.linalg.norm(q, axis=1)
    ndo = np.linalg.norm(do, axis=1)
    row_q = scale * unit * (ads @ nk)
    row_k = scale * unit * (ads.T @ nq)
    ev = unit * (p.T @ ndo)
    w = unit * ads + tiny * visf                         # per-term rounding of dS
    del ads
    el_q = scale * (w @ ak)
    el_k = scale * (w.T @ aq)
    del w
    ev_e = (unit * p + tiny * visf).T @ ado

    def with_d_term(dd_row, dd_el):
        return ((row_q + scale * dd_row * np.linalg.norm(pk, axis=1),
                 row_k + scale * (p.T @ (dd_row * nq)), ev),
                (el_q + scale * dd_el[:, None] * np.abs(pk),
                 el_k + scale * (p.T @ (dd_el[:, None] * aq)), ev_e))

    # O stored by a forward kernel: one unit of its own rounding of O, one of the oracle's, and
    # the forward's rounding of P before P V (|dO_stored| <= unit |O| + unit (P|V|) +
    # tiny (vis|V|) + tiny per element).  The per-row scales keep the plain one-unit form.
    o_err = unit * (np.abs(o) + p @ av) + tiny * (visf @ av + 1.0)
    row, elem = with_d_term(unit * np.abs(do * o).sum(axis=1), (ado * o_err).sum(axis=1))
    # O handed to the kernel by the oracle (its own rounding of the exact O): D then differs by
    # the kernel's fp32 sum of d products only, allowed 2^-20 of sum_c |dO_ic O_ic|.
    dd_given = 2.0 ** -20 * np.abs(do * o_used).sum(axis=1)
    given_row, given_elem = with_d_term(dd_given, dd_given)
    return dq, dk, dv, o, lse, GradScales(row, elem, given_row, given_elem)


def attention_backward(q, k, v, do, dtype, B, Hq, Hkv, Nq, Nkv, d, causal, scale,
                       window=None, heads=None, exact_o=False, error_scales=False):
    """Gradients of every (or the listed) query head.

    q, do: uint16 storage bits [B, Hq, Nq, d]; k, v: [B, Hkv, Nkv, d].
    heads: optional list of flat query heads b * Hq + h to compute (their key/value head's dK
    and dV then hold only those query heads' contributions).
    exact_o: form D from the exact fp64 O (the exact gradient) instead of O rounded to the
    storage type as the forward saves it.
    error_scales: also return a GradScales: rounding scales of a kernel that rounds P and dS
    to the storage type (unit = one ulp at 1: 2^-7 bf16, 2^-10 f16; tiny = the subnormal
    spacing, 2^-24 f16), per row ([B,Hq,Nq] for dq, [B,Hkv,Nkv] for dk, dv) and per element
    (the gradients' shapes), for D formed from O as a forward kernel stored it (row, elem) and
    from the oracle's own stored O handed to the kernel (given_row, given_elem).
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
    unit, tiny = storage_unit(dtype) if error_scales else (None, 0.0)
    shapes = ((B, Hq, Nq), (B, Hkv, Nkv), (B, Hkv, Nkv))
    acc = {f: [np.full(sh, np.nan) if n == 0 else np.zeros(sh)
               for n, sh in enumerate(shapes if "row" in f else [x + (d,) for x in shapes])]
           for f in GradScales._fields}
    todo = range(B * Hq) if heads is None else heads
    for bh in todo:
        b, h = divmod(int(bh), Hq)
        hk = h // G
        res = _head_backward(qd[b, h], kd[b, hk], vd[b, hk], dod[b, h], causal, scale, window,
                             None if exact_o else dtype, unit, tiny)
        gq, gk, gv, go, gl = res[:5]
        dq[b, h], o[b, h], lse[b, h] = gq, go, gl
        dk[b, hk] += gk
        dv[b, hk] += gv
        if error_scales:
            for f, (sq, sk, sv) in zip(GradScales._fields, res[5]):
                acc[f][0][b, h] = sq
                acc[f][1][b, hk] += sk
                acc[f][2][b, hk] += sv
    if error_scales:
        return dq, dk, dv, o, lse, GradScales(*(tuple(acc[f]) for f in GradScales._fields))
    return dq, dk, dv, o, lse


def storage_unit(dtype):
    """(unit, tiny) of a 16-bit storage type: its ulp at 1 and its subnormal spacing."""
    if str(dtype).lower().startswith("b"):
        return 2.0 ** -7, 2.0 ** -133
    return 2.0 ** -10, 2.0 ** -24
