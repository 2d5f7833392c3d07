"""Pins of the FP8 oracle (oracle/fp8.py): the E4M3 codec against the format's definition and
an independent library conversion, the signed Hadamard rotation against a library Hadamard
matrix and orthogonality, and the fp64 attention against the pinned prefill oracle
("FlashAttention Explained", section "FP8 Attention and Incoherent Processing")."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from oracle import fp8


def test_e4m3_decode_fixed_points():
    dec = fp8.e4m3_decode
    assert dec(0x7E) == 448.0 and dec(0xFE) == -448.0      # largest finite
    assert dec(0x38) == 1.0 and dec(0x08) == 2.0 ** -6     # one, smallest normal
    assert dec(0x01) == 2.0 ** -9 and dec(0x07) == 7 * 2.0 ** -9   # subnormals
    assert dec(0x39) == 1.125 and dec(0x3F) == 1.875
    assert np.isnan(dec(0x7F)) and np.isnan(dec(0xFF))
    assert dec(0x00) == 0.0


def test_e4m3_encode_round_trips_every_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    np.testing.assert_array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes)), codes)


def test_e4m3_encode_ties_to_even_and_saturates():
    enc = fp8.e4m3_encode
    assert enc(1.0625) == 0x38       # halfway 1.0 / 1.125 -> even mantissa (1.0)
    assert enc(1.1875) == 0x3A       # halfway 1.125 / 1.25 -> 1.25
    assert enc(1.0626) == 0x39
    assert enc(2.0 ** -10) == 0x00   # halfway 0 / 2^-9 -> 0
    assert enc(3 * 2.0 ** -10) == 0x02
    assert enc(1000.0) == 0x7E and enc(-1e9) == 0xFE
    assert enc(464.0) == 0x7E


def test_e4m3_encode_matches_an_independent_conversion():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(20000) * 10.0 ** rng.uniform(-3, 2.5, 20000)).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(fp8.e4m3_encode(x), ref)


@pytest.mark.parametrize("d", [64, 128])
def test_rotation_is_the_signed_hadamard_matrix(d):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(d) / np.sqrt(d)
    signs = np.where(np.random.default_rng(d).random(d) < 0.5, -1.0, 1.0)
    eye = np.eye(d, dtype=np.float32)
    M = fp8.rotate_f32(eye, signs).astype(np.float64)   # row i = M applied to e_i
    np.testing.assert_allclose(M, (H @ np.diag(signs)).T, rtol=0, atol=2e-7)
    np.testing.assert_allclose(M @ M.T, np.eye(d), rtol=0, atol=1e-6)
    x = np.random.default_rng(1).standard_normal((5, d)).astype(np.float32)
    y = np.random.default_rng(2).standard_normal((7, d)).astype(np.float32)
    np.testing.assert_allclose(fp8.rotate_f32(x, signs) @ fp8.rotate_f32(y, signs).T, x @ y.T,
                               rtol=0, atol=5e-5)


def test_quantisation_error_is_at_most_half_a_step():
    x = np.random.default_rng(4).standard_normal((3, 300, 128)).astype(np.float32)
    x[0, 5, 7] = 60.0  # an outlier sets its tile's scale
    codes, scales = fp8.quantize_tiles(x)
    for t in range(3):
        blk = x[:, t * 128:(t + 1) * 128] / scales[:, t][:, None, None]
        deq = fp8.e4m3_decode(codes[:, t * 128:(t + 1) * 128])
        a = np.abs(blk).astype(np.float64)
        step = np.exp2(np.maximum(np.floor(np.log2(np.maximum(a, 1e-30))), -6) - 3)
        assert np.all(np.abs(deq - blk) <= step / 2 + 1e-12)
    # the tile holding the outlier, 60 = 240 * 2^-2, reaches the upper half of the E4M3 range
    assert scales[0, 0] == 0.25 and np.abs(fp8.e4m3_decode(codes[0, :128])).max() == 240.0


def test_block_scale_is_the_smallest_power_of_two_that_fits():
    """pow2_scale: 2^e with amax <= 448 * 2^e < 2 * amax, checked against the definition at the
    boundaries (448 itself, the next float up, powers of two, tiny and huge values)."""
    f32 = np.float32
    vals = np.array([448.0, np.nextafter(f32(448.0), f32(1e9)), 224.0, 1.0, 3.0, 60.0, 1e-30,
                     2.0 ** -120, 3e38, 1.0 / 3.0], dtype=np.float32)
    sc = fp8.pow2_scale(vals).astype(np.float64)
    for a, s_ in zip(vals.astype(np.float64), sc):
        m, e = np.frexp(s_)
        assert m == 0.5                              # a power of two
        if e - 1 > -126:
            assert a <= 448.0 * s_ < 2 * a + 1e-300  # and the smallest that fits
        else:
            assert a <= 448.0 * s_ and s_ == 2.0 ** -126
    assert list(sc[:4]) == [1.0, 2.0, 0.5, 2.0 ** -8]
    assert fp8.pow2_scale(np.float32(0.0)) == 1.0


def test_f64_attention_matches_the_prefill_oracle():
    cfg = syn.PrefillConfig("f8", 1, 4, 2, 70, 90, 32, "bf16", True, 55)
    q, k, v = cfg.host_inputs()
    qx, kx, vx = (oracle.bits_to_double(t, "bf16") for t in (q, k, v))
    o, lse = fp8.attention_f64(qx, kx, vx, True, cfg.scale)
    of, lf = oracle.attention(q, k, v, "bf16", 1, 4, 2, 70, 90, 32, True, cfg.scale)
    np.testing.assert_allclose(o, of, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lf, rtol=0, atol=1e-12)


def test_rotation_leaves_unquantised_scores_unchanged():
    """(Q M)(K M)^T = Q K^T: without quantisation the rotated problem is the same attention."""
    cfg = syn.PrefillConfig("f8", 1, 2, 1, 40, 40, 64, "bf16", False, 56)
    q, k, v = cfg.host_inputs()
    qx, kx, vx = (oracle.bits_to_double(t, "bf16") for t in (q, k, v))
    signs = np.where(np.random.default_rng(0).random(64) < 0.5, -1.0, 1.0)
    qr = fp8.rotate_f32(qx.astype(np.float32), signs).astype(np.float64)
    kr = fp8.rotate_f32(kx.astype(np.float32), signs).astype(np.float64)
    o1, l1 = fp8.attention_f64(qx, kx, vx, False, cfg.scale)
    o2, l2 = fp8.attention_f64(qr, kr, vx, False, cfg.scale)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-5)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-5)


def test_prepare_dequantises_to_the_rotated_inputs():
    """prepare + dequantized: each value is within half an E4M3 step (times its block's scale)
    of the rotated Q / K and the unrotated V; the scales are those of the right block (128
    rows of one (batch, head) plane for Q and K, the whole plane for V); planes are (batch,
    head) in that order.  Every scale is the smallest power of two 2^e with amax <= 448 * 2^e."""
    rng = np.random.default_rng(21)
    B, Hq, Hkv, Nq, Nkv, d = 2, 4, 2, 200, 150, 64
    q = rng.standard_normal((B, Hq, Nq, d)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, Nkv, d)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, Nkv, d)).astype(np.float32)
    q[1, 2, 130, 5] = 40.0   # an outlier in one tile of one plane
    v[0, 1, 7, 3] = -30.0    # and in one V plane
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    prep = fp8.prepare(q, k, v, signs)
    qd, kd, vd = fp8.dequantized(prep, B, Hq, Hkv, Nq, Nkv, d)
    H = np.asarray(__import__("scipy.linalg", fromlist=["hadamard"]).hadamard(d), np.float64)
    M = H @ np.diag(signs) / np.sqrt(d)          # x -> M x, rows as vectors: x M^T
    qr = q.astype(np.float64) @ M.T
    kr = k.astype(np.float64) @ M.T
    for got, ref, sc, rows in ((qd, qr, prep["sq"], 128), (kd, kr, prep["sk"], 128)):
        b_, h_, n_, _ = ref.shape
        for b in range(b_):
            for h in range(h_):
                for t in range(-(-n_ // rows)):
                    blk = ref[b, h, t * rows:(t + 1) * rows]
                    s = sc[b * h_ + h, t]
                    amax = float(np.abs(blk).max())
                    assert amax <= 448.0 * s * (1 + 1e-6) and 448.0 * s < 2 * amax * (1 + 1e-6)
                    err = np.abs(got[b, h, t * rows:(t + 1) * rows] - blk)
                    # half a step of E4M3 (2^-4 relative, 2^-10 absolute below 2^-6) plus the
                    # fp32 rotation's rounding
                    assert np.all(err <= s * np.maximum(np.abs(blk) / s * 2.0 ** -4, 2.0 ** -10)
                                  + 1e-5)
    for b in range(B):
        for h in range(Hkv):
            s = prep["sv"][b * Hkv + h]
            assert s == fp8.pow2_scale(np.abs(v[b, h]).max())
            err = np.abs(vd[b, h] - v[b, h])
            assert np.all(err <= s * np.maximum(np.abs(v[b, h]) / s * 2.0 ** -4, 2.0 ** -10))
    # the outlier's tile: the rotation spreads 40 over 64 channels (5 each), about twice the
    # tile's other maxima; unrotated V keeps it whole
    assert prep["sq"][1 * Hq + 2, 1] > 1.5 * prep["sq"][1 * Hq + 2, 0]
    assert prep["sv"][0 * Hkv + 1] > 5 * prep["sv"][0 * Hkv + 0]


def test_per_tensor_baseline_equals_block_scaling_when_every_block_shares_the_maximum():
    """With the same amax in every 128-row tile of every Q and K plane and in every V plane, one
    scale per tensor is the same as one per block: the baseline equals the unrotated block model
    exactly."""
    rng = np.random.default_rng(31)
    B, Hq, Hkv, N, d = 1, 4, 2, 256, 64
    q = rng.uniform(-1, 1, (B, Hq, N, d)).astype(np.float32)
    k = rng.uniform(-1, 1, (B, Hkv, N, d)).astype(np.float32)
    v = rng.uniform(-1, 1, (B, Hkv, N, d)).astype(np.float32)
    for x in (q, k):
        x[:, :, ::128, 0] = 2.0   # the first row of every tile holds the maximum
    v[:, :, 0, 0] = 2.0
    o_base, l_base = fp8.fp8_attention_per_tensor(q, k, v, True, d ** -0.5)
    o_blk, l_blk, _ = fp8.fp8_attention(q, k, v, None, True, d ** -0.5)
    np.testing.assert_array_equal(o_base, o_blk)
    np.testing.assert_array_equal(l_base, l_blk)


def test_per_tensor_baseline_lets_one_outlier_set_every_scale():
    """One very large Q entry in head 0 sets the baseline's one scale for the whole tensor, which
    pushes head 1's values (about 10^-5 of the outlier) into E4M3's subnormal range; the block
    model gives head 1 a scale of its own.  Head 1's output error grows only in the baseline."""
    rng = np.random.default_rng(32)
    B, Hq, Hkv, N, d = 1, 2, 1, 128, 64
    q = rng.standard_normal((B, Hq, N, d)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, N, d)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, N, d)).astype(np.float32)
    q[0, 0, 3, 5] = 1.0e5
    exact, _ = fp8.attention_f64(q.astype(np.float64), k.astype(np.float64),
                                 v.astype(np.float64), False, d ** -0.5)
    o_base, _ = fp8.fp8_attention_per_tensor(q, k, v, False, d ** -0.5)
    o_blk, _, _ = fp8.fp8_attention(q, k, v, None, False, d ** -0.5)
    err = lambda o: float(np.sqrt(np.mean((o[0, 1] - exact[0, 1]) ** 2)))
    assert err(o_base) > 2 * err(o_blk), (err(o_base), err(o_blk))


def test_fp32_rotation_codes_are_within_a_step_of_the_exact_rotation():
    """The codes of the fp32 butterfly rotation (the order the kernel uses) against E4M3 of the
    same rows rotated in fp64 by the explicit Sylvester-Hadamard matrix, with the same scales:
    every code within one E4M3 spacing of the exact value and nearly all identical."""
    rng = np.random.default_rng(41)
    d = 128
    x = rng.standard_normal((2, 300, d)).astype(np.float32)
    x[0, 3, 9] = 50.0
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    H = np.asarray(__import__("scipy.linalg", fromlist=["hadamard"]).hadamard(d), np.float64)
    np.testing.assert_array_equal(fp8.hadamard_sylvester(d), H)
    codes, scales = fp8.quantize_tiles(fp8.rotate_f32(x, signs))
    exact = fp8.rotate_exact(x, signs)
    sc = np.repeat(scales, 128, axis=1)[:, :300, None].astype(np.float64)
    y = exact / sc
    deq = fp8.e4m3_decode(codes)
    assert np.all(np.abs(deq - y) <= fp8.e4m3_spacing(y))
    assert (codes == fp8.e4m3_encode(y)).mean() > 0.99
