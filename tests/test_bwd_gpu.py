"""GPU parity of the backward pass (attn_bwd) against the fp64 backward oracle.

"FlashAttention Explained", section "Backward Pass: Recomputation Beats Storage".  The GPU
backward consumes the GPU forward's own O and L (as a training step does); the oracle is the
exact gradient of the pages' algorithm with D formed from O as the forward stores it.
Tolerance, derived from the arithmetic: P and dS are rounded to 16 bits before their MMAs, the
stored O may differ from the oracle's rounding of the exact O by one unit in an element (which
moves D and, through dS = P (dP - D), dQ and dK), and the outputs are rounded once more.  The
oracle returns, per row, the size of the first two effects for one unit of the storage type
(error_scales); each row of dQ, dK and dV must lie within twice that plus 1% of the reference
row's L2 norm.  Rows whose terms nearly cancel (a query that sees two keys) get a bound as wide
as their terms, not their sum.
"""
import numpy as np
import pytest

import synthetic as syn
from oracle.backward import attention_backward

pytestmark = pytest.mark.gpu

RTOL_ROW = 1e-2
SCALE_FACTOR = 2.0


@pytest.fixture(scope="module")
def attn():
    import exact_io_aware_09_gb300 as m

    return m


def check_grad(name, got, ref, scales, what):
    got = np.asarray(got, dtype=np.float64).reshape(-1, ref.shape[-1])
    ref = np.asarray(ref, dtype=np.float64).reshape(-1, ref.shape[-1])
    scales = np.asarray(scales, dtype=np.float64).reshape(-1)
    assert np.all(np.isfinite(got)), f"{what}: non-finite {name}"
    err = np.linalg.norm(got - ref, axis=1)
    allowed = SCALE_FACTOR * scales + RTOL_ROW * np.linalg.norm(ref, axis=1) + 1e-6
    worst = int(np.argmax(err / allowed)) if len(err) else 0
    assert np.all(err <= allowed), (
        f"{what}: {name} row {worst} error {err[worst]:.3e} > {allowed[worst]:.3e} "
        f"({int((err > allowed).sum())} rows)")
    return float((err / allowed).max()) if len(err) else 0.0


def run_case(attn, B, Hq, Hkv, Nq, Nkv, d, dt, causal, seed, heads=None):
    import torch

    cfg = syn.PrefillConfig("bwd", B, Hq, Hkv, Nq, Nkv, d, dt, causal, seed)
    q, k, v = cfg.host_inputs()
    do = syn.host_normal_bits((B, Hq, Nq, d), seed + 7, dt)
    dev = lambda x: syn.bits_to_tensor(x, dt, "cuda")
    qt, kt, vt, dot = dev(q), dev(k), dev(v), dev(do)
    o, lse = attn.attn_fwd(qt, kt, vt, causal=causal, scale=cfg.scale)
    nan = lambda t: torch.full_like(t, float("nan"))
    dq, dk, dv = attn.attn_bwd(qt, kt, vt, o, dot, lse, causal=causal, scale=cfg.scale,
                               dq=nan(qt), dk=nan(kt), dv=nan(vt))
    assert attn.attn_poll_status() == 0
    rq, rk, rv, _, _, sc = attention_backward(q, k, v, do, dt, B, Hq, Hkv, Nq, Nkv, d, causal,
                                              cfg.scale, heads=heads, error_scales=True)
    got = [x.float().cpu().numpy() for x in (dq, dk, dv)]
    return cfg, got, (rq, rk, rv), sc, (qt, kt, vt, o, dot, lse)


SHAPES = [
    # (B, Hq, Hkv, N_q, N_kv, d, dtype, causal)
    (1, 2, 2, 128, 128, 64, "bf16", False),
    (1, 2, 1, 300, 300, 128, "f16", True),
    (2, 4, 2, 200, 333, 64, "bf16", True),     # ragged both ways, bottom-right causal
    (2, 4, 2, 200, 333, 128, "bf16", False),
    (1, 2, 2, 400, 100, 64, "f16", True),      # N_kv < N_q: top rows see no key
    (1, 2, 2, 100, 400, 128, "bf16", True),    # N_kv > N_q
    (1, 3, 1, 517, 517, 128, "bf16", True),    # 3 query heads per key/value head
    (1, 8, 1, 384, 384, 64, "f16", True),      # 8 query heads per key/value head
    (1, 1, 1, 255, 1000, 128, "bf16", False),
    (2, 4, 4, 640, 640, 128, "bf16", False),
    (1, 16, 2, 1024, 1024, 128, "bf16", True),
    # more dK/dV blocks than SMs under the causal mask: the blocks run in the launcher's packed
    # order, and every key tile of every head must still be computed once
    (2, 16, 8, 1280, 1280, 64, "bf16", True),
    (1, 32, 16, 1280, 1280, 128, "f16", True),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_backward_small(attn, shape):
    B, Hq, Hkv, Nq, Nkv, d, dt, causal = shape
    cfg, got, ref, sc, _ = run_case(attn, B, Hq, Hkv, Nq, Nkv, d, dt, causal,
                                    400 + sum(shape[:6]))
    for name, g, r, e in zip(("dq", "dk", "dv"), got, ref, sc):
        check_grad(name, g, r, e, f"shape {shape}")


def test_backward_deterministic(attn):
    import torch

    cfg, got, ref, _, (qt, kt, vt, o, dot, lse) = run_case(attn, 1, 8, 2, 700, 700, 128, "bf16",
                                                           True, 91)
    a = attn.attn_bwd(qt, kt, vt, o, dot, lse, causal=True, scale=cfg.scale)
    b = attn.attn_bwd(qt, kt, vt, o, dot, lse, causal=True, scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_gqa_full_size(attn):
    """The 70B-class GQA causal workload (B=1, Hq=64, Hkv=8, N=8192, d=128): dQ of the eight
    query heads of key/value head 0 and that head's dK and dV, against the oracle."""
    cfg, got, ref, sc, _ = run_case(attn, 1, 64, 8, 8192, 8192, 128, "bf16", True, 4001,
                                    heads=list(range(8)))
    dq, dk, dv = got
    rq, rk, rv = ref
    eq, ek, ev = sc
    check_grad("dq", dq[0, :8], rq[0, :8], eq[0, :8], "GQA N=8192")
    check_grad("dk", dk[0, :1], rk[0, :1], ek[0, :1], "GQA N=8192")
    check_grad("dv", dv[0, :1], rv[0, :1], ev[0, :1], "GQA N=8192")
