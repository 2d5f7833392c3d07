"""GPU parity of the split-KV decode over a paged KV cache (attn_decode_paged).

"FlashAttention Explained", section "Decoding, Paged and Split-KV Variants": the cache lives in
fixed-size non-contiguous pages reached through a block table.  The oracle is the packed decode
definition of the gathered cache.  Page sizes from 16 (several pages per 64-token stage) to
1024 (several stages per page), shuffled page pools whose unused rows hold garbage (or NaN),
ragged and empty sequences, both head dimensions and element types.  At the full decode
workload the paged step must equal the packed step bit for bit.
"""
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


LENGTHS = [0, 1, 15, 16, 17, 63, 64, 65, 511, 512, 513, 1000, 3000]


@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256, 1024])
@pytest.mark.parametrize("d,dtype,Hq,Hkv", [(128, "bf16", 64, 8), (64, "f16", 16, 4)])
def test_paged_decode_vs_oracle(attn, page_size, d, dtype, Hq, Hkv):
    import torch

    cfg = syn.DecodeConfig("paged", len(LENGTHS), Hq, Hkv, d, dtype, 71 + page_size,
                           lengths_override=tuple(LENGTHS))
    q, kc, vc = cfg.host_inputs()
    table, n_pages, pg, sl = syn.paged_layout(LENGTHS, page_size, seed=page_size)
    kp = syn.scatter_to_pages(kc, n_pages, page_size, pg, sl, fill=1)
    vp = syn.scatter_to_pages(vc, n_pages, page_size, pg, sl, fill=2)
    dev = lambda x: syn.bits_to_tensor(x, dtype, "cuda")
    seq = torch.tensor(LENGTHS, dtype=torch.int32, device="cuda")
    o = torch.full((cfg.B, Hq, d), float("nan"), dtype=dev(q).dtype, device="cuda")
    lse = torch.full((cfg.B, Hq), float("nan"), device="cuda")
    o, lse = attn.attn_decode_paged(dev(q), dev(kp), dev(vp), torch.from_numpy(table).cuda(), seq,
                                    max(LENGTHS), o=o, lse=lse, scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    og = o.float().cpu().numpy().astype(np.float64).reshape(-1, d)
    lg = lse.cpu().numpy().astype(np.float64).reshape(-1)
    orf, lrf = oracle.decode_rows_paged(q, kp, vp, table, LENGTHS, page_size, dtype, cfg.B, Hq,
                                        Hkv, d, cfg.scale)
    check_rows(og, lg, orf, lrf, f"paged decode page={page_size} d={d}", dtype=dtype)


def test_paged_full_workload_equals_packed(attn):
    """The 64-sequence decode workload (1.16 M cached tokens) in 16-token pages of a shuffled,
    NaN-padded pool: the same bits as the packed decode of the same cache."""
    import torch

    cfg = syn.CONFIG5
    lengths = cfg.lengths()
    q, kc, vc = cfg.device_inputs("cuda")
    cu = torch.from_numpy(syn.cu_seqlens(lengths)).cuda()
    max_len = int(lengths.max())
    o_ref, l_ref = attn.attn_decode_splitkv(q, kc, vc, cu, max_len, scale=cfg.scale)
    for page_size in (16, 128):
        table, n_pages, pg, sl = syn.paged_layout(lengths, page_size, seed=5 + page_size)
        kp = syn.scatter_to_pages(kc, n_pages, page_size, pg, sl)
        vp = syn.scatter_to_pages(vc, n_pages, page_size, pg, sl)
        seq = torch.from_numpy(lengths.astype(np.int32)).cuda()
        o, l = attn.attn_decode_paged(q, kp, vp, torch.from_numpy(table).cuda(), seq, max_len,
                                      scale=cfg.scale)
        assert attn.attn_poll_status() == 0
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref), page_size
        del kp, vp


def test_paged_pool_past_2_31_elements_equals_packed(attn):
    """A pool of 2.25e9 elements per K and V (16 sequences of 140,000 to 150,000 tokens, Hkv=8,
    d=128, bf16): the packed cache itself read as consecutive 16-token pages, in reverse page
    order per sequence so that the table is not the identity.  The same bits as the packed
    decode, whose offsets past 2^31 are checked against the oracle in the decode tests."""
    import torch

    lengths = np.array([140000] * 14 + [140000, 150000], dtype=np.int64)
    cfg = syn.DecodeConfig("bigpool", 16, 64, 8, 128, "bf16", 7101,
                           lengths_override=tuple(int(x) for x in lengths))
    cu = syn.cu_seqlens(lengths)
    assert int(cu[-1]) * cfg.Hkv * cfg.d > 2 ** 31
    q, kc, vc = cfg.device_inputs("cuda")
    max_len = int(lengths.max())
    o_ref, l_ref = attn.attn_decode_splitkv(q, kc, vc, torch.from_numpy(cu).cuda(), max_len,
                                            scale=cfg.scale)
    page = 16
    n_pages = int(cu[-1]) // page
    max_pages = max_len // page
    table = np.zeros((cfg.B, max_pages), dtype=np.int32)
    # store sequence b's pages in reverse: its token t sits in pool page p0 + n - 1 - t // 16
    perm = np.empty(int(cu[-1]) // page, dtype=np.int64)
    for b in range(cfg.B):
        p0, n = int(cu[b]) // page, int(lengths[b]) // page
        table[b, :n] = p0 + n - 1 - np.arange(n)
        perm[p0:p0 + n] = p0 + np.arange(n)[::-1]
    idx = torch.from_numpy(perm).cuda()
    kp = kc.view(n_pages, page, cfg.Hkv, cfg.d).index_select(0, idx)
    vp = vc.view(n_pages, page, cfg.Hkv, cfg.d).index_select(0, idx)
    del kc, vc
    seq = torch.from_numpy(lengths.astype(np.int32)).cuda()
    o, l = attn.attn_decode_paged(q, kp, vp, torch.from_numpy(table).cuda(), seq, max_len,
                                  scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)
    del kp, vp, q, o, l
    torch.cuda.empty_cache()


def test_paged_bad_block_table_is_reported(attn):
    """A block-table entry outside the pool is reported, never read."""
    import torch

    cfg = syn.DecodeConfig("bad", 2, 8, 1, 64, "bf16", 9, lengths_override=(100, 40))
    q, kc, vc = cfg.device_inputs("cuda")
    table, n_pages, pg, sl = syn.paged_layout([100, 40], 16, seed=1)
    kp = syn.scatter_to_pages(kc, n_pages, 16, pg, sl)
    vp = syn.scatter_to_pages(vc, n_pages, 16, pg, sl)
    table[1, 1] = n_pages + 7
    seq = torch.tensor([100, 40], dtype=torch.int32, device="cuda")
    attn.attn_decode_paged(q, kp, vp, torch.from_numpy(table).cuda(), seq, 100, scale=cfg.scale)
    assert attn.attn_poll_status() == -8   # ATTN_ERR_BAD_LENGTHS
    table[1, 1] = 0
    o, l = attn.attn_decode_paged(q, kp, vp, torch.from_numpy(table).cuda(), seq, 100,
                                  scale=cfg.scale)
    assert attn.attn_poll_status() == 0


def test_paged_argument_errors(attn):
    import torch

    q = torch.zeros((1, 8, 64), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((4, 24, 1, 64), dtype=torch.bfloat16, device="cuda")   # page size 24
    table = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    seq = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(attn.AttnError):
        attn.attn_decode_paged(q, pool, pool, table, seq, 1)
    pool = torch.zeros((4, 16, 1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(attn.AttnError):   # max_seqlen beyond the table's reach
        attn.attn_decode_paged(q, pool, pool, table, seq, 65)
