"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test ties one oracle function to something other than itself: a value the pages
print (tests/golden/, each with its citation), a closed form, an invariant, a special case
that reduces to a library routine, or brute force on tiny inputs with an independent
formula.  A plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a wrong head mapping, a wrong mask side) fails at least one of them.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
import synthetic as syn

F16, BF16 = "f16", "bf16"


def f16_bits(values):
    return np.array([oracle.double_to_f16(x) for x in np.ravel(values)], dtype=np.uint16).reshape(
        np.shape(values))


def rounded(x, decimals):
    return abs(x) <= 0.5 * 10 ** (-decimals) + 1e-12


def close_dp(got, printed, decimals):
    got = np.atleast_1d(np.asarray(got, dtype=np.float64))
    printed = np.atleast_1d(np.asarray(printed, dtype=np.float64))
    return np.all(np.abs(got - printed) <= 0.5 * 10 ** (-decimals) + 1e-9)


def scores_as_inputs(scores, values):
    """q = e_0 (d = dv columns), k_j = (s_j, 0, ...), so S = scores exactly at scale 1."""
    scores = np.asarray(scores, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    if values.ndim == 1:
        values = values[:, None]
    n, dv = values.shape
    d = max(dv, 1)
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, 1, n, d))
    k[0, 0, :, 0] = scores
    v = np.zeros((1, 1, n, d))
    v[0, 0, :, :dv] = values
    return f16_bits(q), f16_bits(k), f16_bits(v), n, d


# ------------------------------------------------------------------------------------
# pages' worked examples
# ------------------------------------------------------------------------------------
def test_four_scores_definition(golden):
    g = golden("online_softmax_four_scores.json")
    q, k, v, n, d = scores_as_inputs(g["scores"], g["values"])
    o, lse = oracle.attention(q, k, v, F16, 1, 1, 1, 1, n, d, False, 1.0)
    assert close_dp(o[0, 0, 0, 0], g["output"], 3)
    # the textbook (no max subtraction) sum and exponentials
    assert close_dp(math.exp(lse[0, 0, 0]), g["exp_sum"], 3)
    assert close_dp([math.exp(s) for s in g["scores"]], g["exp_scores"], 3)
    # probabilities: V = identity makes O the row of P
    q2, k2, v2, n2, d2 = scores_as_inputs(g["scores"], np.eye(4))
    p, _ = oracle.attention(q2, k2, v2, F16, 1, 1, 1, 1, n2, d2, False, 1.0)
    assert close_dp(p[0, 0, 0, :4], g["probabilities"], 3)


def test_four_scores_recurrence(golden):
    g = golden("online_softmax_four_scores.json")
    tr = oracle.online_trace(g["scores"], g["values"], g["block_ends"])
    assert tr["m"][0] == g["block1"]["m"] and tr["m"][1] == g["block2"]["m"]
    assert close_dp(tr["l"][0], g["block1"]["l"], 3)
    assert close_dp(tr["a"][0, 0], g["block1"]["a"], 3)
    assert close_dp(tr["alpha"][1], g["block2"]["alpha"], 3)
    assert close_dp(tr["alpha"][1] * tr["l"][0], g["block2"]["l_rescaled"], 3)
    assert close_dp(tr["l"][1] - tr["alpha"][1] * tr["l"][0], g["block2"]["l_block"], 3)
    assert close_dp(tr["l"][1], g["block2"]["l"], 3)
    assert close_dp(tr["alpha"][1] * tr["a"][0, 0], g["block2"]["a_rescaled"], 3)
    assert close_dp(tr["a"][1, 0] - tr["alpha"][1] * tr["a"][0, 0], g["block2"]["a_block"], 3)
    assert close_dp(tr["a"][1, 0], g["block2"]["a"], 3)
    assert close_dp(tr["o"][0], g["output"], 3)


def test_four_scores_4dp(golden):
    g = golden("online_softmax_four_scores_4dp.json")
    tr = oracle.online_trace(g["scores"], g["values"], g["block_ends"])
    assert close_dp(tr["l"][0], g["tileA"]["l"], 4)
    assert close_dp(tr["a"][0, 0], g["tileA"]["o"], 4)
    assert close_dp(tr["alpha"][1], g["tileB"]["alpha"], 4)
    assert close_dp(math.exp(-3.0), g["tileB"]["exp_min"], 4)
    assert close_dp(tr["l"][1], g["tileB"]["l"], 4)
    assert close_dp(tr["a"][1, 0], g["tileB"]["o"], 4)
    assert abs(tr["o"][0] - g["output"]) <= g["output_tolerance"]
    q, k, v, n, d = scores_as_inputs(g["scores"], g["values"])
    o, lse = oracle.attention(q, k, v, F16, 1, 1, 1, 1, n, d, False, 1.0)
    assert abs(o[0, 0, 0, 0] - g["output"]) <= g["output_tolerance"]
    # direct weights relative to the global max 3
    w = [math.exp(s - 3.0) for s in g["scores"]]
    assert close_dp(w, g["direct_weights"], 4)
    assert close_dp(math.exp(lse[0, 0, 0] - 3.0), g["direct_weight_sum"], 4)


def test_block_merge_both_orders(golden):
    g = golden("block_merge.json")
    s1 = oracle.block_summary(g["blocks"][0])
    s2 = oracle.block_summary(g["blocks"][1])
    assert s1[0] == g["summaries"][0]["m"] and close_dp(s1[1], g["summaries"][0]["l"], 3)
    assert s2[0] == g["summaries"][1]["m"] and close_dp(s2[1], g["summaries"][1]["l"], 3)
    for a, b in ((s1, s2), (s2, s1)):
        m, l, _ = oracle.merge_states((a[0], a[1], [0.0]), (b[0], b[1], [0.0]))
        assert m == g["merged"]["m"] and close_dp(l, g["merged"]["l"], 3)
    direct = oracle.block_summary(g["blocks"][0] + g["blocks"][1])
    assert close_dp(direct[1], g["direct_l"], 3)


def test_two_tile_trace(golden):
    g = golden("two_tile_trace.json")
    tr = oracle.online_trace(g["scores"], g["values"], g["block_ends"])
    assert tr["m"][0] == g["tile1"]["m"] and tr["m"][1] == g["tile2"]["m"]
    assert close_dp(tr["l"][0], g["tile1"]["l"], 4)
    assert close_dp(tr["a"][0], g["tile1"]["a"], 4)
    assert close_dp(tr["alpha"][1], g["tile2"]["alpha"], 4)
    assert close_dp(tr["l"][1], g["tile2"]["l"], 4)
    assert close_dp(tr["a"][1], g["tile2"]["a"], 4)
    assert close_dp(tr["o"], g["output"], 4)
    w1 = [math.exp(s - g["tile1"]["m"]) for s in g["scores"][:2]]
    w2 = [math.exp(s - g["tile2"]["m"]) for s in g["scores"][2:]]
    assert close_dp(w1, g["tile1"]["w"], 4) and close_dp(w2, g["tile2"]["w"], 4)
    q, k, v, n, d = scores_as_inputs(g["scores"], g["values"])
    o, _ = oracle.attention(q, k, v, F16, 1, 1, 1, 1, n, d, False, 1.0)
    assert close_dp(o[0, 0, 0, :2], g["output"], 4)
    q2, k2, v2, n2, d2 = scores_as_inputs(g["scores"], np.eye(4))
    p, _ = oracle.attention(q2, k2, v2, F16, 1, 1, 1, 1, n2, d2, False, 1.0)
    assert close_dp(p[0, 0, 0, :4], g["global_weights"], 4)


def test_causal_tile_listing(golden):
    g = golden("causal_tiles_ex4.json")
    t = oracle.causal_tiles(g["query_tile"], g["Br"], g["Bc"], g["N"])
    assert t["loaded"] == g["loaded"]
    assert t["unmasked"] == g["unmasked"]
    assert t["masked"] == g["masked"]
    lo, hi = g["tile10_empty_rows"]
    assert t["empty_rows"][10] == list(range(lo, hi + 1))
    # skip bound j <= 2i for B_r = 2 B_c, every query tile of the page's problem
    for i in range(1, g["N"] // g["Br"] + 1):
        assert oracle.causal_tiles(i, 128, 64, 4096)["loaded"] == list(range(1, 2 * i + 1))


def test_bytes_model(golden):
    g = golden("bytes_model.json")
    N, d, b = g["N"], g["d"], g["bytes_per_element"]
    MiB = 1 << 20
    r, w = oracle.naive_traffic(N, d, b)
    assert (r, w, r + w) == (g["naive_unmasked"]["reads"], g["naive_unmasked"]["writes"],
                             g["naive_unmasked"]["total"])
    r, w = oracle.flash_traffic(N, d, b, g["Br"], g["Bc"])
    assert r == g["flash_unmasked"]["reads_mib"] * MiB and w == g["flash_unmasked"]["writes_mib"] * MiB
    assert r + w == g["flash_unmasked"]["total"]
    r, w = oracle.naive_traffic(N, d, b, causal=True)
    assert r == g["naive_causal_idealised"]["reads_mib"] * MiB
    assert w == g["naive_causal_idealised"]["writes_mib"] * MiB
    assert r + w == g["naive_causal_idealised"]["total_mib"] * MiB
    r, w = oracle.flash_traffic(N, d, b, g["Br"], g["Bc"], causal=True)
    assert r == g["flash_causal"]["reads_mib"] * MiB and w == g["flash_causal"]["writes_mib"] * MiB
    assert r + w == g["flash_causal"]["total"]
    assert oracle.bytes_model(N, d, b, "naive") == 138412032
    assert 8192 * 8192 * 2 == g["score_matrix_n8192_fp16_bytes"]
    # the logsumexp write adds 4 bytes per query row (16 KiB here)
    assert oracle.bytes_model(N, d, b, "flash", lse=True) - oracle.bytes_model(N, d, b, "flash") == 16384


# ------------------------------------------------------------------------------------
# storage-type conversions
# ------------------------------------------------------------------------------------
def test_fp16_nonassociativity(golden):
    g = golden("fp16_nonassociativity.json")

    def r16(x):
        return oracle.f16_to_double(oracle.double_to_f16(x))

    a, p2 = r16(1000.0), r16(0.2)
    left = r16(r16(a + p2) + p2)
    right = r16(a + r16(p2 + p2))
    assert left == g["left_assoc"]["fp16_result"]
    assert right == g["right_assoc"]["fp16_result"]
    assert r16(1000.0 + 0.5) - 1000.0 == g["spacing_near_1000"]


def test_f16_conversion_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.bits_to_double(bits, F16)
    ref = bits.view(np.float16).astype(np.float64)  # numpy's binary16 as a library check
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    for b in bits[finite][::7]:
        assert oracle.double_to_f16(float(ours[b])) == b or ours[b] == 0.0
    # round-to-nearest-even at ties and overflow
    assert oracle.double_to_f16(1 + 2 ** -11) == 0x3C00
    assert oracle.double_to_f16(1 + 3 * 2 ** -11) == 0x3C02
    assert oracle.double_to_f16(65504.0) == 0x7BFF
    assert oracle.double_to_f16(65519.99) == 0x7BFF
    assert oracle.double_to_f16(65520.0) == 0x7C00
    assert oracle.double_to_f16(2 ** -25) == 0x0000       # tie between 0 and 2^-24 -> even
    assert oracle.double_to_f16(3 * 2 ** -25) == 0x0002


def test_bf16_conversion():
    torch = pytest.importorskip("torch")
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.bits_to_double(bits, BF16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    rng = np.random.default_rng(7)
    x = rng.standard_normal(4096).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 4096)
    tb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for xi, bi in zip(x, tb):
        assert oracle.double_to_bf16(float(xi)) == bi


# ------------------------------------------------------------------------------------
# the definition against independent formulas
# ------------------------------------------------------------------------------------
def direct_attention(qd, kd, vd, causal, scale, Hq, Hkv):
    """Independent formula with no max subtraction: O = sum e^s v / sum e^s (small |s| only)."""
    B, _, Nq, d = qd.shape
    Nkv = kd.shape[2]
    G = Hq // Hkv
    o = np.zeros((B, Hq, Nq, d))
    lse = np.full((B, Hq, Nq), -np.inf)
    for b in range(B):
        for h in range(Hq):
            for i in range(Nq):
                num = np.zeros(d)
                den = 0.0
                for j in range(Nkv):
                    if causal and j - (Nkv - Nq) > i:
                        continue
                    s = scale * float(np.dot(qd[b, h, i], kd[b, h // G, j]))
                    e = math.exp(s)
                    num += e * vd[b, h // G, j]
                    den += e
                if den > 0:
                    o[b, h, i] = num / den
                    lse[b, h, i] = math.log(den)
    return o, lse


@pytest.mark.parametrize("d", [1, 2, 4, 64])
@pytest.mark.parametrize("G", [1, 2, 4])
def test_brute_force_small(d, G):
    rng = np.random.default_rng(1000 * d + G)
    Hkv = 2 if G < 4 else 1
    Hq = Hkv * G
    sizes = range(1, 9) if d <= 4 else (1, 3, 8)
    for Nq, Nkv in itertools.product(sizes, sizes):
        for causal in (False, True):
            B = 2
            qd = rng.standard_normal((B, Hq, Nq, d)) * 0.7
            kd = rng.standard_normal((B, Hkv, Nkv, d)) * 0.7
            vd = rng.standard_normal((B, Hkv, Nkv, d))
            q, k, v = f16_bits(qd), f16_bits(kd), f16_bits(vd)
            qx, kx, vx = (oracle.bits_to_double(t, F16) for t in (q, k, v))
            scale = 1.0 / math.sqrt(d)
            o, lse = oracle.attention(q, k, v, F16, B, Hq, Hkv, Nq, Nkv, d, causal, scale)
            o_ref, lse_ref = direct_attention(qx, kx, vx, causal, scale, Hq, Hkv)
            np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
            fin = np.isfinite(lse_ref)
            assert np.array_equal(np.isfinite(lse), fin)
            np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=0, atol=1e-12)
            # rows with no visible key (only when N_kv < N_q under causal)
            assert np.all(o[~fin] == 0.0)


def test_uniform_scores_give_mean_of_visible_values():
    B, H, N, d = 1, 2, 37, 8
    rng = np.random.default_rng(3)
    q = np.zeros((B, H, N, d), dtype=np.uint16)                       # Q = 0 -> all S equal
    k = f16_bits(rng.standard_normal((B, H, N, d)))
    vd = rng.standard_normal((B, H, N, d))
    v = f16_bits(vd)
    vx = oracle.bits_to_double(v, F16)
    o, lse = oracle.attention(q, k, v, F16, B, H, H, N, N, d, False, 0.5)
    np.testing.assert_allclose(o, np.broadcast_to(vx.mean(axis=2, keepdims=True), o.shape),
                               atol=1e-13)
    np.testing.assert_allclose(lse, math.log(N), atol=1e-13)
    o, lse = oracle.attention(q, k, v, F16, B, H, H, N, N, d, True, 0.5)
    for i in range(N):
        np.testing.assert_allclose(o[:, :, i], vx[:, :, : i + 1].mean(axis=2), atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], math.log(i + 1), atol=1e-13)
    # one visible key: row 0 of a causal square problem is V row 0 exactly
    assert np.array_equal(o[:, :, 0], vx[:, :, 0])


def test_rows_of_p_sum_to_one_and_are_nonnegative():
    rng = np.random.default_rng(11)
    B, H, Nq, Nkv = 1, 3, 5, 8
    d = Nkv                                   # V = identity turns O into the row of P
    q = f16_bits(rng.standard_normal((B, H, Nq, d)) * 2)
    k = f16_bits(rng.standard_normal((B, H, Nkv, d)) * 2)
    v = f16_bits(np.broadcast_to(np.eye(Nkv), (B, H, Nkv, d)))
    for causal in (False, True):
        p, _ = oracle.attention(q, k, v, F16, B, H, H, Nq, Nkv, d, causal, 1.0)
        assert np.all(p >= 0)
        np.testing.assert_allclose(p.sum(axis=-1), 1.0, atol=1e-12)
        if causal:   # bottom-right alignment: row i sees keys 0 .. i + Nkv - Nq
            for i in range(Nq):
                assert np.all(p[:, :, i, i + Nkv - Nq + 1:] == 0)


def test_one_hot_and_large_logits():
    # a score gap of 64 makes the softmax one-hot to far below 1e-12
    n, d = 6, 4
    scores = np.array([0.0, 1.0, 65.0, 2.0, -3.0, 1.0])
    vals = np.arange(n * d, dtype=np.float64).reshape(n, d)
    q, k, v, n_, d_ = scores_as_inputs(scores, vals)
    o, lse = oracle.attention(q, k, v, F16, 1, 1, 1, 1, n, d_, False, 1.0)
    np.testing.assert_allclose(o[0, 0, 0, :d], vals[2], atol=1e-12)
    assert abs(lse[0, 0, 0] - 65.0) < 1e-12
    # x8 stress draws: max subtraction keeps everything finite
    cfg = syn.PrefillConfig("stress", 1, 2, 2, 64, 64, 64, F16, False, 3001, 3)
    qb, kb, vb = cfg.host_inputs()
    o, lse = oracle.attention(qb, kb, vb, F16, 1, 2, 2, 64, 64, 64, False, cfg.scale)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def test_mask_changes_the_answer():
    cfg = syn.PrefillConfig("t6", 1, 1, 1, 16, 16, 8, F16, False, 9)
    q, k, v = cfg.host_inputs()
    o0, _ = oracle.attention(q, k, v, F16, 1, 1, 1, 16, 16, 8, False, cfg.scale)
    o1, _ = oracle.attention(q, k, v, F16, 1, 1, 1, 16, 16, 8, True, cfg.scale)
    assert np.allclose(o0[..., -1, :], o1[..., -1, :], atol=1e-12)   # last row sees all keys
    assert np.max(np.abs(o0[..., :-1, :] - o1[..., :-1, :])) > 1e-3


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(2, 4, 2, 33, 33, 16), (1, 6, 3, 20, 45, 32), (1, 2, 2, 70, 9, 8)])
def test_against_torch_sdpa_fp64(dtype, causal, shape):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    B, Hq, Hkv, Nq, Nkv, d = shape
    cfg = syn.PrefillConfig("lib", B, Hq, Hkv, Nq, Nkv, d, dtype, causal, 77)
    q, k, v = cfg.host_inputs()
    o, lse = oracle.attention(q, k, v, dtype, B, Hq, Hkv, Nq, Nkv, d, causal, cfg.scale)
    qt, kt, vt = (torch.from_numpy(oracle.bits_to_double(t, dtype)) for t in (q, k, v))
    G = Hq // Hkv
    kt = kt.repeat_interleave(G, dim=1)
    vt = vt.repeat_interleave(G, dim=1)
    mask = None
    if causal:
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nkv)[None, :]
        mask = j <= i + (Nkv - Nq)
    fin = np.isfinite(lse)
    ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=cfg.scale).numpy()
    np.testing.assert_allclose(o[fin], ref[fin], atol=1e-12, rtol=0)
    s = torch.einsum("bhid,bhjd->bhij", qt, kt) * cfg.scale
    if mask is not None:
        s = s.masked_fill(~mask, float("-inf"))
    lse_ref = torch.logsumexp(s, dim=-1).numpy()
    np.testing.assert_allclose(lse[fin], lse_ref[fin], atol=1e-12, rtol=0)


def test_selected_rows_match_full():
    cfg = syn.PrefillConfig("rows", 2, 4, 2, 40, 56, 16, BF16, True, 5)
    q, k, v = cfg.host_inputs()
    o, lse = oracle.attention(q, k, v, BF16, 2, 4, 2, 40, 56, 16, True, cfg.scale)
    rows = np.array([0, 5, 39, 40, 77, 200, 319], dtype=np.int64)
    o2, lse2 = oracle.attention_rows(q, k, v, BF16, 2, 4, 2, 40, 56, 16, True, cfg.scale, rows)
    assert np.array_equal(o.reshape(-1, 16)[rows], o2)
    assert np.array_equal(lse.reshape(-1)[rows], lse2)


# ------------------------------------------------------------------------------------
# merges and the decode definition
# ------------------------------------------------------------------------------------
def test_merge_any_order_equals_direct():
    rng = np.random.default_rng(21)
    for trial in range(40):
        n = int(rng.integers(2, 60))
        dv = int(rng.integers(1, 6))
        s = rng.standard_normal(n) * (1 + 5 * rng.random())
        vals = rng.standard_normal((n, dv))
        direct = oracle.online_trace(s, vals, [n])
        w = np.exp(s - s.max())
        ref_o = (w[:, None] * vals).sum(0) / w.sum()
        np.testing.assert_allclose(direct["o"], ref_o, atol=1e-13)
        cuts = sorted(set(rng.integers(1, n, size=int(rng.integers(1, min(n, 6)))).tolist()))
        bounds = [0] + cuts + [n]
        states = []
        for a, b in zip(bounds[:-1], bounds[1:]):
            m, l = oracle.block_summary(s[a:b])
            o = oracle.online_trace(s[a:b], vals[a:b], [b - a])["o"]
            states.append((m, l, o))
        for perm in itertools.islice(itertools.permutations(range(len(states))), 24):
            acc = (-np.inf, 0.0, np.zeros(dv))
            for p in perm:
                acc = oracle.merge_states(acc, states[p])
            np.testing.assert_allclose(acc[2], ref_o, atol=1e-12)
            assert abs(acc[0] - s.max()) == 0.0
            np.testing.assert_allclose(acc[1], w.sum(), rtol=1e-13)
        # random binary tree
        pool = list(states)
        while len(pool) > 1:
            i, j = sorted(rng.choice(len(pool), size=2, replace=False))
            merged = oracle.merge_states(pool[i], pool[j])
            pool = [x for t, x in enumerate(pool) if t not in (i, j)] + [merged]
        np.testing.assert_allclose(pool[0][2], ref_o, atol=1e-12)
        # the multi-block recurrence gives the same output
        tr = oracle.online_trace(s, vals, bounds[1:])
        np.testing.assert_allclose(tr["o"], ref_o, atol=1e-12)


def test_recurrence_masked_blocks_give_zero_not_nan():
    s = np.array([-np.inf, -np.inf, 1.0, -np.inf, 0.5])
    vals = np.arange(5.0)
    tr = oracle.online_trace(s, vals, [2, 4, 5])
    assert tr["m"][0] == -np.inf and tr["l"][0] == 0.0 and np.all(np.isfinite(tr["a"][1:]))
    w = np.array([0, 0, math.exp(0.0), 0, math.exp(-0.5)])
    np.testing.assert_allclose(tr["o"][0], (w * vals).sum() / w.sum(), atol=1e-14)


def test_decode_definition_matches_prefill_and_direct():
    lengths = [1, 7, 300, 513, 64]
    cfg = syn.DecodeConfig("dec", len(lengths), 8, 2, 16, BF16, 99, lengths_override=tuple(lengths))
    q, kc, vc = cfg.host_inputs()
    cu = syn.cu_seqlens(lengths)
    o, lse = oracle.decode_rows(q, kc, vc, cu, BF16, cfg.B, 8, 2, 16, cfg.scale)
    qx = oracle.bits_to_double(q, BF16)
    kx = oracle.bits_to_double(kc, BF16)
    vx = oracle.bits_to_double(vc, BF16)
    for b, L in enumerate(lengths):
        t0 = int(cu[b])
        kb = np.ascontiguousarray(kc[t0:t0 + L].transpose(1, 0, 2))[None]   # [1, Hkv, L, d]
        vb = np.ascontiguousarray(vc[t0:t0 + L].transpose(1, 0, 2))[None]
        op, lp = oracle.attention(q[b][None, :, None, :], kb, vb, BF16, 1, 8, 2, 1, L, 16,
                                  False, cfg.scale)
        np.testing.assert_array_equal(o[b * 8:(b + 1) * 8], op.reshape(8, 16))
        np.testing.assert_array_equal(lse[b * 8:(b + 1) * 8], lp.reshape(8))
        if L <= 64:
            od, ld = direct_attention(qx[b][None, :, None, :], kx[t0:t0 + L].transpose(1, 0, 2)[None],
                                      vx[t0:t0 + L].transpose(1, 0, 2)[None], False, cfg.scale, 8, 2)
            np.testing.assert_allclose(o[b * 8:(b + 1) * 8], od.reshape(8, 16), atol=1e-12)
            np.testing.assert_allclose(lse[b * 8:(b + 1) * 8], ld.reshape(8), atol=1e-12)


# ------------------------------------------------------------------------------------
# the masks that change the operator: sliding window and block-sparse pattern
# ("FlashAttention Explained", FlexAttention section, sliding_causal; "FlashAttention,
# annotated", section 3.3)
# ------------------------------------------------------------------------------------
def _masked_inputs(B, Hq, Hkv, Nq, Nkv, d, seed, dtype=BF16):
    cfg = syn.PrefillConfig("m", B, Hq, Hkv, Nq, Nkv, d, dtype, True, seed)
    return cfg, cfg.host_inputs()


@pytest.mark.parametrize("Nq,Nkv", [(37, 37), (20, 45), (45, 20)])
def test_window_wider_than_the_sequence_is_causal(Nq, Nkv):
    cfg, (q, k, v) = _masked_inputs(1, 4, 2, Nq, Nkv, 16, 700 + Nq)
    oc, lc = oracle.attention_rows(q, k, v, BF16, 1, 4, 2, Nq, Nkv, 16, True, cfg.scale)
    for causal in (True, False):   # the window implies the causal bound either way
        ow, lw = oracle.attention_rows(q, k, v, BF16, 1, 4, 2, Nq, Nkv, 16, causal, cfg.scale,
                                       window=Nkv + Nq)
        np.testing.assert_array_equal(ow, oc)
        np.testing.assert_array_equal(lw, lc)


@pytest.mark.parametrize("Nq,Nkv", [(33, 33), (12, 40), (40, 12)])
def test_window_zero_sees_only_the_diagonal_key(Nq, Nkv):
    """W = 0: one visible key per row, so O is that key's value row and L its score."""
    cfg, (q, k, v) = _masked_inputs(1, 2, 1, Nq, Nkv, 8, 800 + Nq)
    o, lse = oracle.attention_rows(q, k, v, BF16, 1, 2, 1, Nq, Nkv, 8, True, cfg.scale, window=0)
    # bf16 -> fp32 by bit placement, independently of the oracle's conversion table
    as_f64 = lambda bits: (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    qx, kx, vx = as_f64(q), as_f64(k), as_f64(v)
    off = Nkv - Nq
    for h in range(2):
        for i in range(Nq):
            r = h * Nq + i
            j = i + off
            if j < 0:
                assert lse[r] == -np.inf and np.all(o[r] == 0.0)
                continue
            np.testing.assert_array_equal(o[r], vx[0, 0, j])
            assert abs(lse[r] - cfg.scale * float(np.dot(qx[0, h, i], kx[0, 0, j]))) < 1e-12


@pytest.mark.parametrize("W", [1, 5, 16])
def test_window_row_is_full_attention_over_its_keys(W):
    """Each windowed row equals unmasked attention over the keys [i + off - W, i + off]."""
    Nq, Nkv, d = 30, 41, 16
    cfg, (q, k, v) = _masked_inputs(1, 2, 2, Nq, Nkv, d, 900 + W)
    o, lse = oracle.attention_rows(q, k, v, BF16, 1, 2, 2, Nq, Nkv, d, True, cfg.scale, window=W)
    off = Nkv - Nq
    for h in range(2):
        for i in range(Nq):
            hi = i + off
            lo = max(0, hi - W)
            ks = np.ascontiguousarray(k[:, h:h + 1, lo:hi + 1])
            vs = np.ascontiguousarray(v[:, h:h + 1, lo:hi + 1])
            qs = np.ascontiguousarray(q[:, h:h + 1, i:i + 1])
            of, lf = oracle.attention_rows(qs, ks, vs, BF16, 1, 1, 1, 1, hi - lo + 1, d, False,
                                           cfg.scale)
            np.testing.assert_allclose(o[h * Nq + i], of[0], rtol=0, atol=1e-14)
            assert abs(lse[h * Nq + i] - lf[0]) < 1e-13


def test_block_mask_all_ones_and_all_zeros():
    Nq, Nkv, d, bs = 50, 70, 8, 16
    cfg, (q, k, v) = _masked_inputs(1, 2, 1, Nq, Nkv, d, 950)
    shape = (-(-Nq // bs), -(-Nkv // bs))
    for causal in (False, True):
        ref = oracle.attention_rows(q, k, v, BF16, 1, 2, 1, Nq, Nkv, d, causal, cfg.scale)
        ones = oracle.attention_rows(q, k, v, BF16, 1, 2, 1, Nq, Nkv, d, causal, cfg.scale,
                                     block_mask=np.ones(shape, np.uint8), block=bs)
        np.testing.assert_array_equal(ones[0], ref[0])
        np.testing.assert_array_equal(ones[1], ref[1])
    o, lse = oracle.attention_rows(q, k, v, BF16, 1, 2, 1, Nq, Nkv, d, False, cfg.scale,
                                   block_mask=np.zeros(shape, np.uint8), block=bs)
    assert np.all(o == 0.0) and np.all(lse == -np.inf)


@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_row_is_full_attention_over_listed_blocks(causal):
    Nq, Nkv, d, bs = 48, 64, 8, 8
    cfg, (q, k, v) = _masked_inputs(1, 1, 1, Nq, Nkv, d, 960 + causal)
    rng = np.random.default_rng(961)
    mask = (rng.random((Nq // bs, Nkv // bs)) < 0.4).astype(np.uint8)
    o, lse = oracle.attention_rows(q, k, v, BF16, 1, 1, 1, Nq, Nkv, d, causal, cfg.scale,
                                   block_mask=mask, block=bs)
    off = Nkv - Nq
    for i in range(Nq):
        keys = [j for j in range(Nkv) if mask[i // bs, j // bs] and (not causal or j <= i + off)]
        if not keys:
            assert lse[i] == -np.inf and np.all(o[i] == 0.0)
            continue
        ks = np.ascontiguousarray(k[:, :, keys])
        vs = np.ascontiguousarray(v[:, :, keys])
        qs = np.ascontiguousarray(q[:, :, i:i + 1])
        of, lf = oracle.attention_rows(qs, ks, vs, BF16, 1, 1, 1, 1, len(keys), d, False, cfg.scale)
        np.testing.assert_allclose(o[i], of[0], rtol=0, atol=1e-14)
        assert abs(lse[i] - lf[0]) < 1e-13


# ------------------------------------------------------------------------------------
# paged KV cache: an addressing scheme over the same definition
# ("FlashAttention Explained", section "Decoding, Paged and Split-KV Variants")
# ------------------------------------------------------------------------------------
@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_paged_decode_is_the_packed_definition(page_size):
    lengths = [0, 1, 37, 130, 64]
    Hq, Hkv, d = 8, 2, 16
    cfg = syn.DecodeConfig("pg", len(lengths), Hq, Hkv, d, BF16, 123, lengths_override=tuple(lengths))
    q, kc, vc = cfg.host_inputs()
    cu = syn.cu_seqlens(lengths)
    ref_o, ref_l = oracle.decode_rows(q, kc, vc, cu, BF16, cfg.B, Hq, Hkv, d, cfg.scale)
    # scatter the packed cache into shuffled pages, leaving unused pages full of garbage
    rng = np.random.default_rng(page_size)
    n_pages = [-(-L // page_size) for L in lengths]
    total = sum(n_pages) + 5
    perm = rng.permutation(total)
    kp = rng.integers(0, 65535, size=(total, page_size, Hkv, d)).astype(np.uint16)
    vp = rng.integers(0, 65535, size=(total, page_size, Hkv, d)).astype(np.uint16)
    table = np.full((len(lengths), max(n_pages)), -1, dtype=np.int32)
    used = 0
    for b, L in enumerate(lengths):
        for pg in range(n_pages[b]):
            phys = perm[used]
            used += 1
            table[b, pg] = phys
            t = np.arange(pg * page_size, min(L, (pg + 1) * page_size))
            kp[phys, t - pg * page_size] = kc[cu[b] + t]
            vp[phys, t - pg * page_size] = vc[cu[b] + t]
    o, lse = oracle.decode_rows_paged(q, kp, vp, table, lengths, page_size, BF16, cfg.B, Hq, Hkv, d,
                                      cfg.scale)
    np.testing.assert_array_equal(o, ref_o)
    np.testing.assert_array_equal(lse, ref_l)
    # the gather itself: every token of every sequence comes back in order
    np.testing.assert_array_equal(oracle.gather_pages(kp, table, lengths, page_size), kc)
