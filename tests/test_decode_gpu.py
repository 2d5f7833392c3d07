"""GPU parity of the split-KV decode (attn_decode_splitkv through the C ABI) against the fp64
oracle: ragged lengths around the 64-token stage and the split boundaries, empty sequences,
1 to 16 query heads per key/value head, split sizes, garbage (NaN) in cache rows no sequence
owns, a length beyond the promised maximum, the full 64-sequence workload, and a cache of more
than 2^31 elements."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from parity import check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    import exact_io_aware_09_gb300 as m

    return m


def run_decode(attn, dt, q, kc, vc, cu, max_len, split=512, capacity=None, fill_nan_rows=None):
    import torch

    qt = syn.bits_to_tensor(q, dt, "cuda")
    T = kc.shape[0]
    cap = capacity or T
    Hkv, d = kc.shape[1], kc.shape[2]
    kt = torch.zeros((cap, Hkv, d), device="cuda", dtype=syn.torch_dtype(dt))
    vt = torch.zeros_like(kt)
    kt[:T] = syn.bits_to_tensor(kc, dt, "cuda")
    vt[:T] = syn.bits_to_tensor(vc, dt, "cuda")
    if fill_nan_rows is not None:
        kt[fill_nan_rows] = float("nan")
        vt[fill_nan_rows] = float("nan")
    cut = torch.from_numpy(np.asarray(cu, dtype=np.int32)).cuda()
    o = torch.full_like(qt, float("nan"))
    lse = torch.full(qt.shape[:2], float("nan"), device="cuda")
    o, lse = attn.attn_decode_splitkv(qt, kt, vt, cut, max_len, o=o, lse=lse, split_size=split,
                                      scale=1.0 / np.sqrt(d))
    status = attn.attn_poll_status()
    return (o.float().cpu().numpy().astype(np.float64).reshape(-1, d),
            lse.cpu().numpy().astype(np.float64).reshape(-1), status)


CASES = [
    # (lengths, Hq, Hkv, d, dtype, split)
    ((1, 7, 63, 64, 65, 511, 512, 513, 1000, 2053), 8, 2, 128, "bf16", 512),
    ((1, 7, 63, 64, 65, 511, 512, 513, 1000, 2053), 4, 4, 64, "f16", 512),
    ((300, 4100, 17), 32, 2, 128, "bf16", 512),       # 16 query heads per key/value head
    ((0, 5, 0, 700), 8, 8, 128, "f16", 512),          # empty sequences
    ((129, 1000, 3333), 8, 1, 64, "bf16", 64),        # smallest split
    ((129, 8000, 3333), 8, 2, 128, "bf16", 4096),     # large split
    ((5000,), 16, 2, 128, "bf16", 512),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{len(c[0])}_G{c[1] // c[2]}_d{c[3]}_{c[4]}_s{c[5]}")
def test_decode_cases(attn, case):
    lengths, Hq, Hkv, d, dt, split = case
    cfg = syn.DecodeConfig("dec", len(lengths), Hq, Hkv, d, dt, 50 + sum(lengths) % 97,
                           lengths_override=tuple(lengths))
    q, kc, vc = cfg.host_inputs()
    cu = syn.cu_seqlens(lengths)
    og, lg, st = run_decode(attn, dt, q, kc, vc, cu, max(lengths), split)
    assert st == 0
    orf, lrf = oracle.decode_rows(q, kc, vc, cu, dt, cfg.B, Hq, Hkv, d, cfg.scale)
    check_rows(og, lg, orf, lrf, f"decode {case}", dtype=dt)


def test_garbage_in_unowned_cache_rows(attn):
    lengths = (70, 1, 130)
    cfg = syn.DecodeConfig("nan", 3, 8, 2, 128, "bf16", 77, lengths_override=lengths)
    q, kc, vc = cfg.host_inputs()
    cu = syn.cu_seqlens(lengths)
    T = int(cu[-1])
    cap = T + 200
    og, lg, st = run_decode(attn, "bf16", q, kc, vc, cu, max(lengths), 512, capacity=cap,
                            fill_nan_rows=slice(T, cap))
    assert st == 0
    orf, lrf = oracle.decode_rows(q, kc, vc, cu, "bf16", 3, 8, 2, 128, cfg.scale)
    check_rows(og, lg, orf, lrf, "NaN past the last sequence")


def test_length_beyond_max_is_reported(attn):
    lengths = (100, 900, 50)
    cfg = syn.DecodeConfig("bad", 3, 8, 2, 64, "f16", 78, lengths_override=lengths)
    q, kc, vc = cfg.host_inputs()
    cu = syn.cu_seqlens(lengths)
    og, lg, st = run_decode(attn, "f16", q, kc, vc, cu, 512, 512)
    assert st == -8
    orf, lrf = oracle.decode_rows(q, kc, vc, cu, "f16", 3, 8, 2, 64, cfg.scale)
    ok = np.r_[0:8, 16:24]   # sequences 0 and 2 are within the promise and still computed
    check_rows(og[ok], lg[ok], orf[ok], lrf[ok], "sequences within max_seqlen_k")
    assert np.all(np.isnan(lg[8:16]))    # sequence 1 is not written


def test_splitkv_workload_full(attn):
    import torch

    cfg = syn.CONFIG5
    lengths = cfg.lengths()
    cu = syn.cu_seqlens(lengths)
    qd, kd, vd = cfg.device_inputs("cuda")
    cut = torch.from_numpy(cu).cuda()
    o, lse = attn.attn_decode_splitkv(qd, kd, vd, cut, int(lengths.max()), split_size=cfg.split,
                                      scale=cfg.scale)
    # a second call gives the same bits (the merge adds the splits in a fixed order)
    o2, lse2 = attn.attn_decode_splitkv(qd, kd, vd, cut, int(lengths.max()), split_size=cfg.split,
                                        scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    del o2, lse2
    og = o.float().cpu().numpy().astype(np.float64).reshape(-1, cfg.d)
    lg = lse.cpu().numpy().astype(np.float64).reshape(-1)
    q, kc, vc = (syn.tensor_to_bits(t) for t in (qd, kd, vd))
    del kd, vd
    orf, lrf = oracle.decode_rows(q, kc, vc, cu, cfg.dtype, cfg.B, cfg.Hq, cfg.Hkv, cfg.d, cfg.scale)
    check_rows(og, lg, orf, lrf, cfg.name, dtype=cfg.dtype)


def test_cache_past_2_31_elements(attn):
    """A packed cache of 2.25e9 elements per K and V (16 sequences of about 140,000 tokens,
    Hkv=8, d=128, bf16), so that the last sequences' element offsets pass 2^31: the last two
    sequences against the oracle, which gets their query rows and cache slices copied back."""
    import torch

    lengths = tuple([140000] * 14 + [139999, 150001])
    cfg = syn.DecodeConfig("bigcache", 16, 64, 8, 128, "bf16", 7001, lengths_override=lengths)
    lens = cfg.lengths()
    cu = syn.cu_seqlens(lens)
    assert int(cu[-2]) * cfg.Hkv * cfg.d > 2 ** 31
    qd, kd, vd = cfg.device_inputs("cuda")
    cut = torch.from_numpy(cu).cuda()
    o, lse = attn.attn_decode_splitkv(qd, kd, vd, cut, int(lens.max()), split_size=cfg.split,
                                      scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    b0 = cfg.B - 2
    t0, t1 = int(cu[b0]), int(cu[cfg.B])
    q = syn.tensor_to_bits(qd[b0:])
    kc = syn.tensor_to_bits(kd[t0:t1])
    vc = syn.tensor_to_bits(vd[t0:t1])
    cu2 = (cu[b0:] - cu[b0]).astype(cu.dtype)
    orf, lrf = oracle.decode_rows(q, kc, vc, cu2, cfg.dtype, 2, cfg.Hq, cfg.Hkv, cfg.d, cfg.scale)
    og = o[b0:].float().cpu().numpy().astype(np.float64).reshape(-1, cfg.d)
    lg = lse[b0:].cpu().numpy().astype(np.float64).reshape(-1)
    check_rows(og, lg, orf, lrf, "cache past 2^31 elements", dtype=cfg.dtype)
    del qd, kd, vd, o, lse
    torch.cuda.empty_cache()
