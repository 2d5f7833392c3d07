"""GPU parity of the prefill kernel (attn_fwd through the C ABI) against the fp64 oracle.

Small shapes cover several tiles, ragged query and key tails, bottom-right causal alignment,
rows with no visible key, grouped-query heads, both head dimensions and both element types;
the benchmark workloads run at full size, every row of every head.  Tolerances are those of
tests/parity.py.
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


def run_gpu(attn, cfg, q, k, v, sentinel=True):
    import torch

    qt, kt, vt = (syn.bits_to_tensor(x, cfg.dtype, "cuda") for x in (q, k, v))
    o = torch.full_like(qt, float("nan")) if sentinel else None
    lse = torch.full((cfg.B, cfg.Hq, cfg.N_q), float("nan"), device="cuda") if sentinel else None
    o, lse = attn.attn_fwd(qt, kt, vt, o=o, lse=lse, causal=cfg.causal, scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    return (o.float().cpu().numpy().astype(np.float64).reshape(-1, cfg.d),
            lse.cpu().numpy().astype(np.float64).reshape(-1))


def oracle_rows(cfg, q, k, v, rows=None):
    return oracle.attention_rows(q, k, v, cfg.dtype, cfg.B, cfg.Hq, cfg.Hkv, cfg.N_q, cfg.N_kv,
                                 cfg.d, cfg.causal, cfg.scale, rows)


SMALL = [
    # (B, Hq, Hkv, N_q, N_kv, d, dtype, causal)
    (1, 1, 1, 128, 128, 64, "f16", False),     # exactly one tile
    (1, 1, 1, 256, 256, 64, "f16", False),     # the single-head workload
    (1, 2, 2, 1, 1, 64, "bf16", False),        # one row, one key
    (1, 2, 2, 1, 1, 128, "f16", True),
    (2, 4, 2, 200, 333, 64, "bf16", True),     # ragged both ways, bottom-right causal
    (2, 4, 2, 200, 333, 64, "bf16", False),
    (1, 2, 1, 300, 300, 128, "f16", True),
    (1, 4, 4, 129, 129, 128, "bf16", False),
    (1, 2, 2, 1, 1000, 128, "bf16", True),     # one query row sees every key
    (1, 2, 2, 400, 100, 64, "f16", True),      # N_kv < N_q: top rows see no key
    (1, 3, 1, 517, 517, 128, "bf16", True),    # 3 query heads per key/value head
    (1, 8, 1, 384, 384, 64, "f16", True),      # 8 query heads per key/value head
    (1, 6, 2, 300, 300, 64, "bf16", True),     # d = 64, 3 query heads per key/value head: one
                                               # head of each group without a partner
    (1, 2, 2, 300, 300, 64, "f16", False),     # d = 64, odd number of query tiles
    (2, 2, 2, 640, 640, 128, "f16", False),
    (1, 2, 2, 1000, 1000, 128, "bf16", True),
    (1, 1, 1, 255, 4000, 64, "bf16", False),   # long key side, short query side
    (1, 1, 1, 4000, 255, 128, "f16", True),
]

# More work items than SMs, so that every resident block runs several items back to back:
# mixed item lengths, items with no visible key between the others, one-tile items (no partial
# sum to hand over) and ragged query tiles.
MANY_ITEMS = [
    (2, 80, 16, 300, 100, 64, "bf16", True),   # a third of the items see no key
    (1, 96, 8, 700, 700, 128, "f16", True),    # 1 to 6 K/V tiles per item
    (4, 64, 64, 130, 130, 64, "bf16", False),  # two tiles each, every other item 2 rows
    (1, 48, 48, 840, 840, 64, "f16", True),    # d = 64, seven query tiles a head (odd tail)
    (2, 200, 50, 128, 64, 128, "bf16", False), # one tile each
    (1, 160, 160, 257, 1000, 128, "bf16", True),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(attn, shape):
    B, Hq, Hkv, Nq, Nkv, d, dt, causal = shape
    cfg = syn.PrefillConfig("small", B, Hq, Hkv, Nq, Nkv, d, dt, causal, 100 + sum(shape[:6]))
    q, k, v = cfg.host_inputs()
    orf, lrf = oracle_rows(cfg, q, k, v)
    for mode in d64_modes(d):
        with d64_kernel(attn, mode):
            og, lg = run_gpu(attn, cfg, q, k, v)
        check_rows(og, lg, orf, lrf, f"shape {shape}, d = 64 kernel {mode}", dtype=dt)


@pytest.mark.parametrize("shape", MANY_ITEMS, ids=lambda s: "x".join(map(str, s)))
def test_many_items(attn, shape):
    B, Hq, Hkv, Nq, Nkv, d, dt, causal = shape
    cfg = syn.PrefillConfig("items", B, Hq, Hkv, Nq, Nkv, d, dt, causal, 200 + sum(shape[:6]))
    q, k, v = cfg.host_inputs()
    orf, lrf = oracle_rows(cfg, q, k, v)
    for mode in d64_modes(d):
        with d64_kernel(attn, mode):
            og, lg = run_gpu(attn, cfg, q, k, v)
        check_rows(og, lg, orf, lrf, f"shape {shape}, d = 64 kernel {mode}", dtype=dt)


@pytest.mark.parametrize("shape", [(1, 96, 8, 700, 700, 128, "f16", True),
                                   (2, 80, 16, 300, 100, 64, "bf16", True),
                                   (4, 64, 64, 130, 130, 64, "bf16", False)],
                         ids=lambda s: "x".join(map(str, s)))
def test_repeated_calls_are_bit_identical(attn, shape):
    """More work items than SMs, so that the blocks take over one another's items in an order
    that changes from launch to launch: O and L must not depend on it (no atomics, a fixed
    order of the sums within an item)."""
    import torch

    B, Hq, Hkv, Nq, Nkv, d, dt, causal = shape
    cfg = syn.PrefillConfig("det", B, Hq, Hkv, Nq, Nkv, d, dt, causal, 300 + sum(shape[:6]))
    q, k, v = cfg.device_inputs("cuda")
    for mode in d64_modes(d):
        with d64_kernel(attn, mode):
            first = attn.attn_fwd(q, k, v, causal=causal, scale=cfg.scale)
            for _ in range(3):
                o, lse = attn.attn_fwd(q, k, v, causal=causal, scale=cfg.scale)
                assert torch.equal(o.view(torch.int16), first[0].view(torch.int16)), mode
                assert torch.equal(lse.view(torch.int32), first[1].view(torch.int32)), mode
        assert attn.attn_poll_status() == 0


def test_output_16_byte_aligned(attn):
    """O only 16-byte aligned (the API's minimum for every pointer)."""
    import torch

    cfg = syn.PrefillConfig("align", 1, 96, 8, 300, 300, 128, "bf16", True, 211)
    q, k, v = cfg.host_inputs()
    qt, kt, vt = (syn.bits_to_tensor(x, cfg.dtype, "cuda") for x in (q, k, v))
    backing = torch.full((qt.numel() + 8,), float("nan"), device="cuda", dtype=qt.dtype)
    o = backing[8:].view(qt.shape)
    assert o.data_ptr() % 32 == 16
    o, lse = attn.attn_fwd(qt, kt, vt, o=o, causal=True, scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    assert torch.isnan(backing[:8]).all()  # nothing written before O
    og = o.float().cpu().numpy().astype(np.float64).reshape(-1, cfg.d)
    lg = lse.cpu().numpy().astype(np.float64).reshape(-1)
    orf, lrf = oracle_rows(cfg, q, k, v)
    check_rows(og, lg, orf, lrf, "16-byte aligned O", dtype=cfg.dtype)


def test_large_logits_small(attn):
    cfg = syn.PrefillConfig("x8", 1, 2, 2, 300, 300, 128, "f16", True, 31, q_scale_pow2=3)
    q, k, v = cfg.host_inputs()
    og, lg = run_gpu(attn, cfg, q, k, v)
    orf, lrf = oracle_rows(cfg, q, k, v)
    check_rows(og, lg, orf, lrf, "x8 logits", dtype=cfg.dtype)


def test_no_keys_and_empty_inputs(attn):
    import torch

    q = torch.randn(1, 2, 70, 64, device="cuda").half()
    k = torch.empty(1, 2, 0, 64, device="cuda").half()
    o, lse = attn.attn_fwd(q, k, k.clone(), causal=False)
    assert attn.attn_poll_status() == 0
    assert torch.all(o == 0) and torch.all(lse == float("-inf"))
    q0 = torch.empty(1, 2, 0, 64, device="cuda").half()
    o0, l0 = attn.attn_fwd(q0, q0, q0)
    assert o0.numel() == 0 and l0.numel() == 0


def test_stream_argument_is_honoured(attn):
    import torch

    cfg = syn.PrefillConfig("stream", 1, 2, 2, 256, 256, 64, "bf16", True, 5)
    q, k, v = cfg.host_inputs()
    s = torch.cuda.Stream()
    qt, kt, vt = (syn.bits_to_tensor(x, cfg.dtype, "cuda") for x in (q, k, v))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        o, lse = attn.attn_fwd(qt, kt, vt, causal=True, scale=cfg.scale, stream=s)
    s.synchronize()
    orf, lrf = oracle_rows(cfg, q, k, v)
    check_rows(o.float().cpu().numpy().reshape(-1, 64), lse.cpu().numpy().reshape(-1), orf, lrf,
               "side stream")


@pytest.mark.parametrize("cfg", [syn.CONFIG1, syn.CONFIG2], ids=lambda c: c.name)
def test_workload_full(attn, cfg):
    q, k, v = cfg.host_inputs()
    og, lg = run_gpu(attn, cfg, q, k, v)
    orf, lrf = oracle_rows(cfg, q, k, v)
    check_rows(og, lg, orf, lrf, cfg.name, dtype=cfg.dtype)


@pytest.mark.parametrize("cfg", [syn.CONFIG3A, syn.CONFIG3B, syn.CONFIG3SA, syn.CONFIG3SB],
                         ids=lambda c: c.name)
def test_long_workload_full(attn, cfg):
    q, k, v = cfg.host_inputs()
    og, lg = run_gpu(attn, cfg, q, k, v)
    orf, lrf = oracle_rows(cfg, q, k, v)
    check_rows(og, lg, orf, lrf, cfg.name, dtype=cfg.dtype)


def test_more_than_2_31_elements_sampled(attn):
    """Q and O of 2.29e9 elements (B=1, Hq=128, Hkv=8, N=140,000 with a ragged last tile, d=128,
    bf16, causal), so that element offsets pass 2^31 in the last heads: sampled rows of the
    first, a middle and the last query head (first and last rows, the ragged tail and random
    rows) against the oracle, which gets those heads' Q, K and V copied back."""
    import torch

    cfg = syn.PrefillConfig("big", 1, 128, 8, 140000, 140000, 128, "bf16", True, 6001)
    assert cfg.B * cfg.Hq * cfg.N_q * cfg.d > 2 ** 31
    q, k, v = cfg.device_inputs("cuda")
    o, lse = attn.attn_fwd(q, k, v, causal=True, scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    rng = np.random.default_rng(6002)
    G = cfg.Hq // cfg.Hkv
    for h in (0, 61, cfg.Hq - 1):
        rows = np.unique(np.concatenate([[0, 1, 127, 128, cfg.N_q - 129, cfg.N_q - 1],
                                         np.arange(cfg.N_q - 96, cfg.N_q, 13),
                                         rng.integers(0, cfg.N_q, 40)])).astype(np.int64)
        qh = syn.tensor_to_bits(q[0, h].contiguous())
        kh = syn.tensor_to_bits(k[0, h // G].contiguous())
        vh = syn.tensor_to_bits(v[0, h // G].contiguous())
        orf, lrf = oracle.attention_rows(qh, kh, vh, cfg.dtype, 1, 1, 1, cfg.N_q, cfg.N_kv,
                                         cfg.d, True, cfg.scale, rows)
        idx = torch.from_numpy(rows).cuda()
        og = o[0, h].index_select(0, idx).float().cpu().numpy().astype(np.float64)
        lg = lse[0, h].index_select(0, idx).cpu().numpy().astype(np.float64)
        check_rows(og, lg, orf, lrf, f"2^31+ elements, head {h}", dtype=cfg.dtype)
    del q, k, v, o, lse
    torch.cuda.empty_cache()


def test_gqa_long_context_full(attn):
    """The 70B-class GQA causal prefill (B=1, Hq=64, Hkv=8, N=8192, d=128, bf16): every row of
    every head against the oracle."""
    cfg = syn.CONFIG4
    q, k, v = cfg.host_inputs()
    og, lg = run_gpu(attn, cfg, q, k, v)
    orf, lrf = oracle_rows(cfg, q, k, v)
    check_rows(og, lg, orf, lrf, cfg.name, dtype=cfg.dtype)
