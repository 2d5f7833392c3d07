"""GPU parity of the backward pass (attn_bwd) against the fp64 backward oracle.

"FlashAttention Explained", section "Backward Pass: Recomputation Beats Storage".  Every case
runs the GPU backward twice: on the GPU forward's own O and L (as a training step does), and on
the oracle's O (its rounding of the exact O to the storage type) and L (rounded to fp32).  The
oracle is the exact gradient of the pages' algorithm with D formed from O as stored.
Tolerance, derived from the arithmetic (tests/parity.py, check_grad): P and dS are rounded to
16 bits before their MMAs, a stored O from the forward kernel moves D and, through
dS = P (dP - D), dQ and dK, and the outputs are rounded once more.  The oracle returns, per row
and per element, the size of these effects for one unit of the storage type (error_scales);
each row of dQ, dK and dV must lie within twice its row scale plus 1% of the reference row's L2
norm, and each element within twice its element scale plus one unit of its own magnitude.
"""
import numpy as np
import pytest

import synthetic as syn
from oracle import round_to_storage
from oracle.backward import attention_backward
from parity import check_grad

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    import exact_io_aware_09_gb300 as m

    return m


def run_case(attn, B, Hq, Hkv, Nq, Nkv, d, dt, causal, seed, heads=None):
    """Backward on the GPU forward's O and L, and on the oracle's.  Returns the config, the
    two sets of GPU gradients, the oracle gradients, its scales and the device tensors."""
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
    rq, rk, rv, ro, rl, sc = attention_backward(q, k, v, do, dt, B, Hq, Hkv, Nq, Nkv, d, causal,
                                                cfg.scale, heads=heads, error_scales=True)
    # the oracle's stored O and L (heads the oracle did not compute keep the GPU forward's,
    # which only reach gradients this test does not check)
    done = np.isfinite(rl) | np.isneginf(rl)
    o_or = dev(round_to_storage(np.where(done[..., None], ro, 0.0), dt))
    l_or = torch.from_numpy(rl.astype(np.float32)).cuda()
    mask = torch.from_numpy(done).cuda()
    o_or = torch.where(mask[..., None], o_or, o)
    l_or = torch.where(mask, l_or, lse)
    gq, gk, gv = attn.attn_bwd(qt, kt, vt, o_or, dot, l_or, causal=causal, scale=cfg.scale,
                               dq=nan(qt), dk=nan(kt), dv=nan(vt))
    assert attn.attn_poll_status() == 0
    host = lambda xs: [x.float().cpu().numpy() for x in xs]
    return cfg, host((dq, dk, dv)), host((gq, gk, gv)), (rq, rk, rv), sc, (qt, kt, vt, o, dot, lse)


def check_both(got, got_given, ref, sc, dt, what, sel=lambda x, i: x):
    """Row and element checks of dq, dk, dv for both sources of O; sel(x, i) picks the
    checked part of gradient i."""
    worst = 0.0
    for i, name in enumerate(("dq", "dk", "dv")):
        worst = max(worst, check_grad(name, sel(got[i], i), sel(ref[i], i), sel(sc.row[i], i),
                                      sel(sc.elem[i], i), dt, f"{what} (forward's O)"))
        worst = max(worst, check_grad(name, sel(got_given[i], i), sel(ref[i], i),
                                      sel(sc.given_row[i], i), sel(sc.given_elem[i], i), dt,
                                      f"{what} (oracle's O)"))
    return worst


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
    cfg, got, got_given, ref, sc, _ = run_case(attn, B, Hq, Hkv, Nq, Nkv, d, dt, causal,
                                               400 + sum(shape[:6]))
    check_both(got, got_given, ref, sc, dt, f"shape {shape}")


@pytest.mark.parametrize("nq,nkv", [(0, 300), (300, 0)], ids=["no_queries", "no_keys"])
def test_backward_with_an_empty_side_is_zero(attn, nq, nkv):
    """No (query, key) pair: every gradient is exactly zero (outputs pre-filled with NaN)."""
    import torch

    dt = torch.bfloat16
    q = torch.randn((2, 4, nq, 128), device="cuda").to(dt)
    k = torch.randn((2, 2, nkv, 128), device="cuda").to(dt)
    v = torch.randn_like(k)
    o = torch.zeros_like(q)
    do = torch.randn_like(q)
    lse = torch.full((2, 4, nq), float("-inf"), device="cuda")
    nan = lambda t: torch.full_like(t, float("nan"))
    dq, dk, dv = attn.attn_bwd(q, k, v, o, do, lse, causal=True, scale=0.125, dq=nan(q),
                               dk=nan(k), dv=nan(v))
    assert attn.attn_poll_status() == 0
    for t in (dq, dk, dv):
        assert torch.equal(t, torch.zeros_like(t))


def test_backward_deterministic(attn):
    import torch

    cfg, got, _, ref, _, (qt, kt, vt, o, dot, lse) = run_case(attn, 1, 8, 2, 700, 700, 128,
                                                              "bf16", True, 91)
    a = attn.attn_bwd(qt, kt, vt, o, dot, lse, causal=True, scale=cfg.scale)
    b = attn.attn_bwd(qt, kt, vt, o, dot, lse, causal=True, scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_gqa_full_size(attn):
    """The 70B-class GQA causal workload (B=1, Hq=64, Hkv=8, N=8192, d=128): dQ of the eight
    query heads of key/value head 0 and that head's dK and dV, against the oracle."""
    cfg, got, got_given, ref, sc, _ = run_case(attn, 1, 64, 8, 8192, 8192, 128, "bf16", True,
                                               4001, heads=list(range(8)))
    check_both(got, got_given, ref, sc, "bf16", "GQA N=8192",
               sel=lambda x, i: x[0, :8] if i == 0 else x[0, :1])


def test_dq_past_2_31_elements_sampled(attn):
    """Q, dO, O and dQ of 2.29e9 elements (B=1, Hq=128, Hkv=8, N=140,000 with a ragged last
    tile, d=128, bf16, causal), so that element offsets pass 2^31 in the last heads.  A query
    row's gradient depends only on its own q, o, do, L and its visible keys, so each sampled row
    of dQ is checked against the oracle run on that row alone: one query against its visible
    keys, without a mask (the GPU backward runs on the GPU forward's O and L, and the check is
    check_grad's with the scales for that source of O)."""
    import torch

    cfg = syn.PrefillConfig("bigbwd", 1, 128, 8, 140000, 140000, 128, "bf16", True, 6101)
    assert cfg.B * cfg.Hq * cfg.N_q * cfg.d > 2 ** 31
    q, k, v = cfg.device_inputs("cuda")
    do = syn.device_normal(q.shape, cfg.seed + 7, cfg.dtype, "cuda")
    o, lse = attn.attn_fwd(q, k, v, causal=True, scale=cfg.scale)
    dq, dk, dv = attn.attn_bwd(q, k, v, o, do, lse, causal=True, scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    del dk, dv
    G = cfg.Hq // cfg.Hkv
    rng = np.random.default_rng(6102)
    bits = lambda t: syn.tensor_to_bits(t.contiguous())
    for h in (0, 61, cfg.Hq - 1):
        rows = sorted({0, 1, 127, 128, cfg.N_q - 1, *rng.integers(0, cfg.N_q, 3).tolist()})
        for i in rows:
            vis = i + 1  # N_q == N_kv: row i sees keys 0 .. i
            qr, dor = bits(q[0, h, i:i + 1]), bits(do[0, h, i:i + 1])
            kr, vr = bits(k[0, h // G, :vis]), bits(v[0, h // G, :vis])
            rq, _, _, _, _, sc = attention_backward(qr, kr, vr, dor, cfg.dtype, 1, 1, 1, 1, vis,
                                                    cfg.d, False, cfg.scale, error_scales=True)
            got = dq[0, h, i].float().cpu().numpy().reshape(1, 1, 1, cfg.d)
            check_grad("dq", got, rq, sc.row[0], sc.elem[0], cfg.dtype,
                       f"2^31+ elements, head {h} row {i}")
    del q, k, v, do, o, lse, dq
    torch.cuda.empty_cache()
