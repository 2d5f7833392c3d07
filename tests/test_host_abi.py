"""CPU-only checks of the C-ABI library: it loads, exports every declared symbol, refuses bad
arguments before any launch, and its host-side schedule helper reproduces the pages' causal
tile listing.  No compute call is made (there is no GPU here)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def attn():
    import __graft_entry__

    __graft_entry__._cuda_build_module().build()
    import exact_io_aware_09_gb300 as m

    return m


def _has_cuda():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


def declared_functions():
    txt = open(os.path.join(ROOT, "include", "attn.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(attn_[a-z0-9_]+)\s*\(",
                       txt, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("attn_fwd", "attn_decode_splitkv", "attn_decode_workspace_bytes",
                     "attn_poll_status", "attn_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(attn):
    lib = ctypes.CDLL(attn.library_path)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/attn.h but not exported"
    assert "sm_103a" in attn.attn_version()


def test_status_strings(attn):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        s = attn.attn_status_string(code)
        assert s and s != "unknown status"
    assert attn.attn_status_string(123) == "unknown status"


def test_d64_kernel_choice(attn):
    assert attn.attn_fwd_set_d64_kernel(attn.D64_PAIR) == attn.D64_AUTO
    assert attn.attn_fwd_set_d64_kernel(attn.D64_SINGLE) == attn.D64_PAIR
    with pytest.raises(attn.AttnError):
        attn.attn_fwd_set_d64_kernel(3)
    assert attn.attn_fwd_set_d64_kernel(attn.D64_AUTO) == attn.D64_SINGLE  # 3 changed nothing


def test_kv_tile_range_matches_page_exercise(golden, attn):
    g = golden("causal_tiles_ex4.json")
    # the page's tiles are 1-based with B_r = 128, B_c = 64
    n, fm = attn.attn_fwd_kv_tiles(g["query_tile"] - 1, g["Br"], g["Bc"], g["N"], g["N"], True)
    assert n == len(g["loaded"]) and n == g["loaded"][-1]
    assert fm == len(g["unmasked"])          # tiles 1..8 unmasked, 9 and 10 masked


@pytest.mark.parametrize("bm,bn", [(128, 64), (128, 128), (64, 128), (128, 32)])
@pytest.mark.parametrize("N", [1, 63, 128, 129, 500, 1024, 4096])
def test_kv_tile_range_matches_oracle_listing(attn, bm, bn, N):
    nq = -(-N // bm)
    for qt in range(nq):
        t = oracle.causal_tiles(qt + 1, bm, bn, N)
        n, fm = attn.attn_fwd_kv_tiles(qt, bm, bn, N, N, True)
        assert n == len(t["loaded"])
        # the kernel also masks the ragged last K/V tile (keys past N), which the page's
        # listing never meets because its N is a multiple of both tile sizes
        ragged_last = (-(-N // bn) - 1) if N % bn else n
        assert fm == min(len(t["unmasked"]), ragged_last)
        n, fm = attn.attn_fwd_kv_tiles(qt, bm, bn, N, N, False)
        assert n == -(-N // bn)
        assert fm == (n - 1 if N % bn else n)


def brute_tiles(qt, bm, bn, nq, nkv, causal):
    """Tiles holding at least one (row, key) pair the mask keeps, and the first tile where some
    row of the query tile loses a key to the mask or to the ragged end."""
    rows = range(qt * bm, min((qt + 1) * bm, nq))
    n_all = -(-nkv // bn)
    vis = lambda i, j: j < nkv and (not causal or j <= i + nkv - nq)
    loaded = [j for j in range(n_all) if any(vis(i, c) for i in rows for c in range(j * bn, (j + 1) * bn))]
    n = (loaded[-1] + 1) if loaded else 0
    first = n
    for j in range(n):
        if any(not vis(i, c) for i in rows for c in range(j * bn, (j + 1) * bn)):
            first = j
            break
    return n, first


@pytest.mark.parametrize("nq,nkv", [(5, 17), (17, 5), (64, 64), (70, 200), (200, 70), (1, 300),
                                    (300, 1), (130, 130)])
def test_kv_tile_range_bottom_right_brute_force(attn, nq, nkv):
    bm, bn = 32, 16
    for causal in (False, True):
        for qt in range(-(-nq // bm)):
            assert attn.attn_fwd_kv_tiles(qt, bm, bn, nq, nkv, causal) == brute_tiles(qt, bm, bn, nq, nkv, causal)


def test_workspace_bytes(attn):
    # (m, l) + o[d] fp32 per (sequence, head, split), o block padded to 256 bytes
    parts = 64 * 64 * 64
    assert attn.attn_decode_workspace_bytes(64, 64, 32768, 512, 128) == parts * 128 * 4 + parts * 8
    assert attn.attn_decode_workspace_bytes(0, 64, 32768, 512, 128) == 0
    assert attn.attn_decode_workspace_bytes(1, 1, 1, 512, 64) >= 66 * 4


def test_fp8_workspace_layout(attn):
    B, Hq, Hkv, Nq, Nkv, d = 2, 8, 2, 300, 1000, 128
    off = attn.attn_fwd_fp8_workspace_offsets(B, Hq, Hkv, Nq, Nkv, d)
    total = attn.attn_fwd_fp8_workspace_bytes(B, Hq, Hkv, Nq, Nkv, d)
    nqt, nkt = -(-Nq // 128), -(-Nkv // 128)
    sizes = [B * Hq * Nq * d, B * Hkv * Nkv * d, B * Hkv * d * nkt * 128, B * Hq * nqt * 4,
             B * Hkv * nkt * 4, B * Hkv * 4, B * Hkv * 4]
    assert off[0] == 0
    for i in range(7):
        assert off[i] % 256 == 0
        end = off[i] + sizes[i]
        assert end <= (off[i + 1] if i < 6 else total)
    assert total - (off[6] + sizes[6]) < 256
    assert attn.attn_fwd_fp8_workspace_bytes(0, Hq, Hkv, Nq, Nkv, d) == 0


def test_bad_arguments_are_refused_before_launch(attn):
    L = attn.lib
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below fails its checks
    odd = ctypes.c_void_p((1 << 20) + 8)
    nul = ctypes.c_void_p(0)
    s = 0.125
    assert L.attn_fwd(fake, fake, fake, fake, fake, 1, 6, 4, 8, 8, 64, 0, s, nul, 0) == -1  # Hq % Hkv
    assert L.attn_fwd(fake, fake, fake, fake, fake, 1, 4, 4, 8, 8, 96, 0, s, nul, 0) == -2  # d
    assert L.attn_fwd(fake, fake, fake, fake, fake, 1, 4, 4, 8, 8, 64, 0, -1.0, nul, 0) == -1
    assert L.attn_fwd(fake, fake, fake, fake, fake, 1, 4, 4, 8, 8, 64, 0, float("nan"), nul, 0) == -1
    assert L.attn_fwd(fake, fake, fake, fake, fake, 1, 4, 4, 8, 8, 64, 0, s, nul, 7) == -1  # dtype
    assert L.attn_fwd(nul, fake, fake, fake, fake, 1, 4, 4, 8, 8, 64, 0, s, nul, 0) == -1
    assert L.attn_fwd(odd, fake, fake, fake, fake, 1, 4, 4, 8, 8, 64, 0, s, nul, 0) == -3
    assert L.attn_fwd(fake, fake, fake, fake, fake, 0, 4, 4, 8, 8, 64, 0, s, nul, 0) == 0   # no-op
    assert L.attn_fwd(fake, fake, fake, fake, fake, 1, 4, 4, 0, 8, 64, 0, s, nul, 0) == 0
    # A valid request with fake pointers must never reach a device: only where there is none
    # is it checked that the call is refused (not computed some other way).
    no_device = not _has_cuda()
    if no_device:
        assert L.attn_fwd(fake, fake, fake, fake, fake, 1, 4, 4, 8, 8, 64, 0, s, nul, 0) == -7

    def dec(split=512, hq=64, hkv=8, d=128, ws_bytes=1 << 30, ws=fake, cu=fake):
        return L.attn_decode_splitkv(fake, fake, fake, cu, 1024, 1024, fake, fake, 2, hq, hkv, d,
                                     split, s, 1, ws, ws_bytes, nul)

    assert dec(split=500) == -2
    assert dec(split=32) == -2
    assert dec(hq=64, hkv=2) == -2            # 32 query heads per key/value head
    assert dec(hq=12, hkv=8) == -1
    assert dec(d=80) == -2
    assert dec(ws_bytes=16) == -4
    assert dec(ws=nul) == -4
    assert dec(cu=ctypes.c_void_p((1 << 20) + 2)) == -3
    # more sequences than a grid dimension holds: refused before any launch
    assert L.attn_decode_splitkv(fake, fake, fake, fake, 1024, 1024, fake, fake, 65536, 64, 8, 128,
                                 512, s, 1, fake, 1 << 40, nul) == -2
    assert L.attn_decode_splitkv_static(fake, fake, fake, fake, 1024, 1024, fake, fake, 65536, 64,
                                        8, 128, 512, s, 1, nul) == -2
    assert L.attn_decode_paged(fake, fake, fake, fake, fake, 64, 16, 64, 1024, fake, fake, 65536,
                               64, 8, 128, 512, s, 1, fake, 1 << 40, nul) == -2
    if no_device:
        assert dec() == -7
    def fp8(d=128, ws_bytes=1 << 30, ws=fake, signs=nul, B=1, nkv=300):
        return L.attn_fwd_fp8(fake, fake, fake, fake, fake, B, 4, 2, 200, nkv, d, 1, s, signs, ws,
                              ws_bytes, nul, 1)

    assert fp8(d=64) == -2
    assert fp8(ws_bytes=1024) == -4
    assert fp8(ws=nul) == -4
    assert fp8(ws=odd) == -3
    assert fp8(B=0) == 0
    if no_device:
        assert fp8() == -7
        assert fp8(signs=fake) == -7
    assert L.attn_selftest_timeout(0, nul) == -1
    assert L.attn_selftest_timeout(2_000_000, nul) == -1


@pytest.mark.parametrize("causal,window", [(True, -1), (False, -1), (True, 0), (True, 1),
                                           (True, 127), (True, 128), (True, 300), (False, 1000)])
def test_kv_span_covers_exactly_the_visible_keys(attn, causal, window):
    """The key-tile span of each query tile holds every visible key and no tile without one;
    the unmasked middle tiles are fully visible to every row."""
    bm = bn = 128
    for N_q, N_kv in [(1, 1), (300, 300), (200, 333), (333, 200), (129, 1000), (1000, 129)]:
        off = N_kv - N_q
        n_kvt = -(-N_kv // bn)
        for qt in range(-(-N_q // bm)):
            jb, je, lo, hi = attn.attn_fwd_kv_span(qt, bm, bn, N_q, N_kv, causal, window)
            rows = np.arange(qt * bm, min(N_q, qt * bm + bm))
            keys = np.arange(N_kv)
            vis = np.ones((len(rows), N_kv), dtype=bool)
            if causal or window >= 0:
                vis &= keys[None, :] <= rows[:, None] + off
            if window >= 0:
                vis &= rows[:, None] + off - keys[None, :] <= window
            for j in range(n_kvt):
                tile = vis[:, j * bn:(j + 1) * bn]
                if tile.any():
                    assert jb <= j < je, (N_q, N_kv, qt, j, jb, je)
                elif not (causal or window >= 0):
                    continue
                else:
                    assert not (jb <= j < je) or j == jb or j == je - 1, (qt, j, jb, je)
                if max(jb, lo) <= j < hi:
                    assert tile.shape[1] == bn and tile.all(), (N_q, N_kv, qt, j, lo, hi)


def _list_schedule(order, weights, n_sm):
    """Makespan of blocks taken in `order` by whichever of n_sm SMs frees up first."""
    import heapq

    free = [(0, i) for i in range(n_sm)]
    heapq.heapify(free)
    end = 0
    for j in order:
        t, i = heapq.heappop(free)
        t += weights[j]
        end = max(end, t)
        heapq.heappush(free, (t, i))
    return end


def test_bwd_kv_order_packs_the_causal_grid(attn):
    """The 8192-token GQA backward (B=1, Hq=64, Hkv=8) on 152 SMs: every job exactly once, and
    taken in that order by the SMs as they free up the blocks finish within 1% of the average
    load, against about 7% over it when started longest first."""
    B, Hq, Hkv, N, n_sm = 1, 64, 8, 8192, 152
    order = attn.attn_bwd_kv_order(B, Hq, Hkv, N, N, True, n_sm)
    n_planes, n_kt = B * Hkv, N // 128
    assert sorted(order) == list(range(n_planes * n_kt))
    # a job's 64-query steps under the causal mask, plus the block's fixed cost (4)
    weights = [2 * (Hq // Hkv) * (N // 128 - j // n_planes) + 4 for j in range(n_planes * n_kt)]
    avg = sum(weights) / n_sm
    packed = _list_schedule(order, weights, n_sm)
    longest_first = _list_schedule(range(n_planes * n_kt), weights, n_sm)
    assert packed <= 1.01 * avg, (packed, avg)
    assert longest_first > 1.05 * avg  # the tail the packing removes
    assert packed < longest_first


def test_bwd_kv_order_keeps_the_default_order(attn):
    # equal jobs (no causal mask), no more blocks than SMs, more blocks than the table holds
    assert attn.attn_bwd_kv_order(1, 64, 8, 8192, 8192, False, 152) == []
    assert attn.attn_bwd_kv_order(1, 16, 2, 1024, 1024, True, 152) == []
    assert attn.attn_bwd_kv_order(8, 64, 8, 8192, 8192, True, 152, cap=2048) == []
    with pytest.raises(attn.AttnError):
        attn.attn_bwd_kv_order(1, 6, 4, 128, 128, True, 152)  # Hq not a multiple of Hkv


def test_bwd_kv_order_bottom_right_alignment(attn):
    """N_kv > N_q (bottom-right causal alignment): still a permutation of the jobs."""
    B, Hq, Hkv, Nq, Nkv = 2, 16, 8, 3000, 9000
    order = attn.attn_bwd_kv_order(B, Hq, Hkv, Nq, Nkv, True, 152)
    assert sorted(order) == list(range(B * Hkv * (-(-Nkv // 128))))


def test_tensors_off_the_gpu_are_refused_before_any_call():
    """The binding checks that every tensor is a CUDA tensor on one device before it calls the
    library (no compute runs here)."""
    import torch

    import exact_io_aware_09_gb300 as attn

    q = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16)
    with pytest.raises(attn.AttnError):
        attn.attn_fwd(q, q, q)
    with pytest.raises(attn.AttnError):
        attn.attn_decode_splitkv(q[0], q[0], q[0], torch.zeros(2, dtype=torch.int32), 8)
