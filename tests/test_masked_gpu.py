"""GPU parity of the prefill variants that change the operator, against the fp64 oracle.

attn_fwd_window: the pages' sliding_causal mask ("FlashAttention Explained", FlexAttention
section) with bottom-right alignment.  attn_fwd_block_sparse: a pattern of (query tile, key tile)
blocks ("FlashAttention, annotated", section 3.3).  Shapes cover several tiles, ragged edges,
windows inside one tile and across tiles, rows with no visible key, grouped-query heads, both
head dimensions and both element types, and more work items than SMs; the sliding window of the
pages' example (W = 1024) and the measured block pattern run at the 8192-token GQA size, every
row.  Tolerances are those of tests/parity.py.
"""
import numpy as np
import pytest

import oracle
import synthetic as syn
from kernels import d64_kernel, d64_modes
from parity import check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    import exact_io_aware_09_gb300 as m

    return m


def _inputs(shape, seed):
    B, Hq, Hkv, Nq, Nkv, d, dt = shape
    cfg = syn.PrefillConfig("masked", B, Hq, Hkv, Nq, Nkv, d, dt, True, seed)
    return cfg, cfg.host_inputs()


def _gpu(cfg, q, k, v):
    import torch

    qt, kt, vt = (syn.bits_to_tensor(x, cfg.dtype, "cuda") for x in (q, k, v))
    o = torch.full_like(qt, float("nan"))
    lse = torch.full((cfg.B, cfg.Hq, cfg.N_q), float("nan"), device="cuda")
    return qt, kt, vt, o, lse


def _host(o, lse, d):
    return (o.float().cpu().numpy().astype(np.float64).reshape(-1, d),
            lse.cpu().numpy().astype(np.float64).reshape(-1))


WINDOW_CASES = [
    # (B, Hq, Hkv, N_q, N_kv, d, dtype), W
    ((1, 2, 2, 300, 300, 64, "bf16"), 0),
    ((1, 2, 1, 300, 300, 128, "f16"), 1),
    ((2, 4, 2, 200, 333, 64, "bf16"), 100),     # window inside one key tile
    ((1, 2, 2, 700, 700, 128, "bf16"), 128),
    ((1, 3, 1, 517, 517, 128, "f16"), 300),     # window across tiles, ragged end
    ((1, 2, 2, 400, 100, 64, "f16"), 50),       # N_kv < N_q: top rows see no key
    ((1, 2, 2, 100, 900, 128, "bf16"), 257),    # N_kv > N_q
    ((1, 2, 2, 1000, 1000, 128, "bf16"), 5000), # wider than the sequence: causal
    ((2, 96, 8, 520, 520, 128, "bf16"), 200),   # more items than SMs, GQA
    ((2, 6, 2, 520, 520, 64, "f16"), 200),      # d = 64, 3 query heads per key/value head
]


@pytest.mark.parametrize("shape,W", WINDOW_CASES, ids=lambda x: str(x))
def test_window(attn, shape, W):
    cfg, (q, k, v) = _inputs(shape, 300 + W + sum(shape[:6]))
    orf, lrf = oracle.attention_rows(q, k, v, cfg.dtype, cfg.B, cfg.Hq, cfg.Hkv, cfg.N_q,
                                     cfg.N_kv, cfg.d, True, cfg.scale, window=W)
    for mode in d64_modes(cfg.d):
        qt, kt, vt, o, lse = _gpu(cfg, q, k, v)
        with d64_kernel(attn, mode):
            o, lse = attn.attn_fwd_window(qt, kt, vt, W, o=o, lse=lse, scale=cfg.scale)
        assert attn.attn_poll_status() == 0
        og, lg = _host(o, lse, cfg.d)
        check_rows(og, lg, orf, lrf, f"window {W} {shape}, d = 64 kernel {mode}",
                   dtype=cfg.dtype)


@pytest.mark.parametrize("d", [128, 64])
def test_window_matches_causal_when_wide(attn, d):
    """W >= N_kv: the same result as attn_fwd's causal mask, bit for bit."""
    import torch

    cfg, (q, k, v) = _inputs((1, 4, 2, 600, 600, d, "bf16"), 77)
    for mode in d64_modes(d):
        qt, kt, vt, o1, l1 = _gpu(cfg, q, k, v)
        o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
        with d64_kernel(attn, mode):
            attn.attn_fwd(qt, kt, vt, o=o1, lse=l1, causal=True, scale=cfg.scale)
            attn.attn_fwd_window(qt, kt, vt, 600, o=o2, lse=l2, scale=cfg.scale)
        assert attn.attn_poll_status() == 0
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_window_pages_example_full_size(attn):
    """The pages' sliding_causal example (W = 1024, 8192 tokens) on the 70B-class GQA heads;
    every row against the oracle."""
    cfg = syn.PrefillConfig("w1024", 1, 64, 8, 8192, 8192, 128, "bf16", True, 4001)
    q, k, v = cfg.host_inputs()
    qt, kt, vt, o, lse = _gpu(cfg, q, k, v)
    o, lse = attn.attn_fwd_window(qt, kt, vt, 1024, o=o, lse=lse, scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    og, lg = _host(o, lse, cfg.d)
    orf, lrf = oracle.attention_rows(q, k, v, "bf16", 1, 64, 8, 8192, 8192, 128, True,
                                     cfg.scale, None, window=1024)
    check_rows(og, lg, orf, lrf, "window 1024 at 8192", dtype=cfg.dtype)


BLOCK_CASES = [
    # (B, Hq, Hkv, N_q, N_kv, d, dtype), causal, density
    ((1, 2, 2, 512, 512, 64, "bf16"), False, 0.5),
    ((1, 2, 1, 640, 640, 128, "f16"), True, 0.6),
    ((2, 4, 2, 300, 700, 128, "bf16"), False, 0.3),   # ragged both ways
    ((1, 2, 2, 700, 300, 64, "f16"), True, 0.7),      # N_kv < N_q
    ((2, 80, 16, 384, 384, 64, "bf16"), True, 0.5),   # more items than SMs
]


@pytest.mark.parametrize("shape,causal,density", BLOCK_CASES, ids=lambda x: str(x))
def test_block_sparse(attn, shape, causal, density):
    import torch

    cfg, (q, k, v) = _inputs(shape, 500 + int(100 * density) + sum(shape[:6]))
    nqt, nkt = -(-cfg.N_q // 128), -(-cfg.N_kv // 128)
    rng = np.random.default_rng(int(1000 * density) + nqt)
    mask = (rng.random((nqt, nkt)) < density).astype(np.uint8)
    mask[0, :] = 0          # a query tile with no block at all
    if nkt > 1:
        mask[-1, :] = 1     # and one with every block
    mt = torch.from_numpy(mask).cuda()
    orf, lrf = oracle.attention_rows(q, k, v, cfg.dtype, cfg.B, cfg.Hq, cfg.Hkv, cfg.N_q,
                                     cfg.N_kv, cfg.d, causal, cfg.scale, block_mask=mask,
                                     block=128)
    for mode in d64_modes(cfg.d):
        qt, kt, vt, o, lse = _gpu(cfg, q, k, v)
        with d64_kernel(attn, mode):
            o, lse = attn.attn_fwd_block_sparse(qt, kt, vt, mt, causal=causal, o=o, lse=lse,
                                                scale=cfg.scale)
        assert attn.attn_poll_status() == 0
        og, lg = _host(o, lse, cfg.d)
        check_rows(og, lg, orf, lrf, f"block-sparse {shape} causal={causal}, d = 64 kernel {mode}",
                   dtype=cfg.dtype)


@pytest.mark.parametrize("d", [128, 64])
def test_block_sparse_all_ones_is_dense(attn, d):
    import torch

    cfg, (q, k, v) = _inputs((1, 4, 2, 600, 700, d, "bf16"), 88)
    qt, kt, vt, o1, l1 = _gpu(cfg, q, k, v)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    ones = torch.ones((5, 6), dtype=torch.uint8, device="cuda")
    for mode in d64_modes(d):
        for causal in (False, True):
            with d64_kernel(attn, mode):
                attn.attn_fwd(qt, kt, vt, o=o1, lse=l1, causal=causal, scale=cfg.scale)
                attn.attn_fwd_block_sparse(qt, kt, vt, ones, causal=causal, o=o2, lse=l2,
                                           scale=cfg.scale)
            assert attn.attn_poll_status() == 0
            assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_block_sparse_measured_pattern_full_size(attn):
    """The block pattern the bench line times (causal blocks kept with probability 1/2, the
    diagonal and the first key block always) on the 70B-class GQA prefill (B=1, Hq=64, Hkv=8,
    N=8192, d=128, bf16), in the bench's launch configuration: every row of every head against
    the oracle."""
    import torch

    cfg = syn.CONFIG4
    q, k, v = cfg.host_inputs()
    pattern = syn.causal_block_pattern(cfg.N_q, cfg.N_kv)
    qt, kt, vt, o, lse = _gpu(cfg, q, k, v)
    o, lse = attn.attn_fwd_block_sparse(qt, kt, vt, torch.from_numpy(pattern).cuda(), causal=True,
                                        o=o, lse=lse, scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    og, lg = _host(o, lse, cfg.d)
    orf, lrf = oracle.attention_rows(q, k, v, cfg.dtype, cfg.B, cfg.Hq, cfg.Hkv, cfg.N_q,
                                     cfg.N_kv, cfg.d, True, cfg.scale, block_mask=pattern,
                                     block=128)
    check_rows(og, lg, orf, lrf, "measured block pattern at 8192", dtype=cfg.dtype)


def test_masked_argument_errors(attn):
    import torch

    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(attn.AttnError):
        attn.attn_fwd_window(q, q, q, -1)
    with pytest.raises(attn.AttnError):
        attn.attn_fwd_block_sparse(q, q, q, torch.ones((2, 1), dtype=torch.uint8, device="cuda"))
