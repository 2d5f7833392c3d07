"""Oracle of the FP8 forward with incoherent processing (TEST INFRASTRUCTURE ONLY).

Only the test suite, the smoke check and the CPU-baseline leg of the benchmark use this
module; the CUDA library shares nothing with it.

"FlashAttention Explained", section "FP8 Attention and Incoherent Processing": Q and K are
multiplied by the same random orthogonal matrix M before quantisation, so that
(Q M)(K M)^T = Q K^T while outlier channels spread over all channels; M is a Hadamard transform
with random sign flips; the inputs are quantised to E4M3 with per-block scaling factors.

Steps, each written out here:
  1. M = H diag(s) / sqrt(d): x -> H (s o x) / sqrt(d), H the Sylvester Hadamard matrix applied
     by the fast Walsh-Hadamard butterflies (stage h = 1, 2, 4, ..., d/2: (a, b) -> (a + b,
     a - b) on elements j and j + h), in fp32 in that order, then one fp32 multiply by the fp32
     value of 1/sqrt(d).  The rotation decides integer codes below, so it is evaluated in the
     precision and order the kernel uses (fp32).
  2. Block quantisation: one scale per 128-row tile of a (batch, head) plane for Q and K
     and one per plane for V (not rotated).  A scale is a power of two, the smallest 2^e with
     amax <= 448 * 2^e (448 is the largest E4M3 value; e >= -126; 1 for an all-zero block);
     code = E4M3(x * 2^-e) rounded to nearest even, saturating at +-448.
  3. Attention in fp64 of the dequantised operands (code value * scale): the same definition as
     the prefill oracle, on these inputs.
Where the pages are silent the readings above are taken: the 128-row block shape, one scale per
plane for V, and power-of-two scales.
"""
import numpy as np

E4M3_MAX = 448.0


# ------------------------------------------------------------------------------------------
# E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is subnormal
# (m * 2^-9); exponent 15 with mantissa 7 is NaN (no infinities); largest finite 1.75 * 2^8.
# ------------------------------------------------------------------------------------------
def e4m3_decode(codes):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def e4m3_encode(x):
    """Nearest E4M3 code (ties to even), saturating to +-448; x float32/float64 (exact)."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x)
    a = np.abs(x)
    a = np.minimum(a, E4M3_MAX)  # saturating (finite inputs only)
    # exponent of the normal binade, clamped to the subnormal range
    _, ex = np.frexp(a)          # a = f * 2^ex, f in [0.5, 1)
    e_unb = np.maximum(ex - 1, -6)   # binade [2^e, 2^(e+1)); below 2^-6 the spacing is 2^-9
    step = np.exp2(e_unb.astype(np.float64) - 3)  # spacing of representable values
    q = a / step                      # exact (power-of-two scaling)
    r = np.floor(q)
    frac = q - r
    up = (frac > 0.5) | ((frac == 0.5) & (np.mod(r, 2) == 1))
    r = r + up
    v = r * step                      # rounded magnitude (may reach the next binade: still exact)
    v = np.minimum(v, E4M3_MAX)
    # back to bits
    _, ev = np.frexp(v)
    e_v = np.maximum(ev - 1, -6)
    is_sub = (v < 2.0 ** -6)
    m_sub = np.round(v / 2.0 ** -9).astype(np.int64)
    m_nrm = np.round((v / np.exp2(e_v.astype(np.float64)) - 1.0) * 8).astype(np.int64)
    e_field = np.where(is_sub, 0, e_v + 7)
    m_field = np.where(is_sub, m_sub, m_nrm)
    code = (e_field.astype(np.int64) << 3) | m_field
    code = np.where(v == 0, 0, code)
    return (code | np.where(sign, 0x80, 0)).astype(np.uint8)


# ------------------------------------------------------------------------------------------
# rotation and quantisation
# ------------------------------------------------------------------------------------------
def rotate_f32(x, signs):
    """Rows of x (float32 [..., d]) -> H (s o x) / sqrt(d) in fp32, butterflies in order."""
    y = np.asarray(x, dtype=np.float32) * np.asarray(signs, dtype=np.float32)
    d = y.shape[-1]
    y = y.copy()
    h = 1
    while h < d:
        y = y.reshape(y.shape[:-1] + (d // (2 * h), 2, h))
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(y.shape[:-3] + (d,))
        h *= 2
    return y * np.float32(1.0 / np.sqrt(np.float32(d)))


def pow2_scale(amax):
    """Block scales for the amax values (float32 array): the smallest power of two 2^e with
    amax <= 448 * 2^e, e >= -126; 1 where amax is 0.  With amax = f 2^k, f in [0.5, 1), and
    448 = 0.875 * 2^9: e = k - 9 when f <= 0.875, else k - 8."""
    a = np.asarray(amax, dtype=np.float64)
    f, k = np.frexp(a)
    e = np.maximum(np.where(f <= 0.875, k - 9, k - 8), -126)
    return np.where(a > 0, np.ldexp(1.0, e), 1.0).astype(np.float32)


def hadamard_sylvester(d):
    """The d x d Sylvester-Hadamard matrix (d a power of two): H_1 = [1],
    H_2k = [[H_k, H_k], [H_k, -H_k]]."""
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


def rotate_exact(x, signs):
    """Rows of x -> H (s o x) / sqrt(d) as one fp64 matrix product with the explicit matrix:
    independent of the butterfly order the fp32 rotation follows."""
    d = np.asarray(x).shape[-1]
    M = hadamard_sylvester(d) * np.asarray(signs, dtype=np.float64)[None, :] / np.sqrt(d)
    return np.asarray(x, dtype=np.float64) @ M.T


def e4m3_spacing(x):
    """Spacing of the E4M3 values around |x| (2^-9 in the subnormal range)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -30)))
    return np.exp2(np.maximum(e, -6) - 3)


def quantize_tiles(x, rows_per_tile=128):
    """x float32 [planes, N, d] -> (codes uint8 [planes, N, d], scales float32 [planes, tiles]).
    One power-of-two scale per 128-row tile (pow2_scale of the tile's amax); codes =
    E4M3(x / scale), an exact power-of-two scaling."""
    x = np.asarray(x, dtype=np.float32)
    P, N, d = x.shape
    nt = -(-N // rows_per_tile)
    codes = np.zeros((P, N, d), dtype=np.uint8)
    scales = np.ones((P, nt), dtype=np.float32)
    for t in range(nt):
        blk = x[:, t * rows_per_tile:(t + 1) * rows_per_tile]
        sc = pow2_scale(np.abs(blk).reshape(P, -1).max(axis=1))
        scales[:, t] = sc
        codes[:, t * rows_per_tile:(t + 1) * rows_per_tile] = e4m3_encode(
            blk.astype(np.float64) / sc[:, None, None].astype(np.float64))
    return codes, scales


def quantize_planes(x):
    """x float32 [planes, N, d] -> (codes, scales [planes]): one power-of-two scale per plane."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).reshape(x.shape[0], -1).max(axis=1) if x.size else np.zeros(x.shape[0])
    sc = pow2_scale(amax)
    return e4m3_encode(x.astype(np.float64) / sc[:, None, None].astype(np.float64)), sc


def prepare(q, k, v, signs):
    """float32 q [B, Hq, Nq, d], k/v [B, Hkv, Nkv, d] and signs [d] (None: no rotation) ->
    the quantised operands and their scales, as the kernel's preparation writes them."""
    B, Hq, Nq, d = q.shape
    _, Hkv, Nkv, _ = k.shape
    qr = rotate_f32(q, signs) if signs is not None else np.asarray(q, np.float32)
    kr = rotate_f32(k, signs) if signs is not None else np.asarray(k, np.float32)
    q8, sq = quantize_tiles(qr.reshape(B * Hq, Nq, d))
    k8, sk = quantize_tiles(kr.reshape(B * Hkv, Nkv, d))
    v8, sv = quantize_planes(np.asarray(v, np.float32).reshape(B * Hkv, Nkv, d))
    return dict(q8=q8, sq=sq, k8=k8, sk=sk, v8=v8, sv=sv)


def dequantized(prep, B, Hq, Hkv, Nq, Nkv, d):
    """fp64 values the FP8 kernel multiplies: code value times its block's scale."""
    qd = e4m3_decode(prep["q8"]) * np.repeat(prep["sq"], 128, axis=1)[:, :Nq, None]
    kd = e4m3_decode(prep["k8"]) * np.repeat(prep["sk"], 128, axis=1)[:, :Nkv, None]
    vd = e4m3_decode(prep["v8"]) * prep["sv"][:, None, None].astype(np.float64)
    return qd.reshape(B, Hq, Nq, d), kd.reshape(B, Hkv, Nkv, d), vd.reshape(B, Hkv, Nkv, d)


def attention_f64(q, k, v, causal, scale):
    """fp64 attention of arbitrary fp64 operands q [B,Hq,Nq,d], k/v [B,Hkv,Nkv,d] (numpy matmul
    per head; the same masking and empty-row rule as the prefill oracle) -> (o, lse)."""
    B, Hq, Nq, d = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    o = np.zeros((B, Hq, Nq, d))
    lse = np.full((B, Hq, Nq), -np.inf)
    for b in range(B):
        for h in range(Hq):
            s = scale * (q[b, h] @ k[b, h // G].T)
            if causal:
                i = np.arange(Nq)[:, None] + (Nkv - Nq)
                s = np.where(np.arange(Nkv)[None, :] <= i, s, -np.inf)
            m = s.max(axis=1) if Nkv else np.full(Nq, -np.inf)
            live = np.isfinite(m)
            e = np.where(live[:, None], np.exp(s - np.where(live, m, 0.0)[:, None]), 0.0)
            l = e.sum(axis=1)
            o[b, h] = np.where(live[:, None], (e @ v[b, h // G]) / np.where(l > 0, l, 1.0)[:, None],
                               0.0)
            lse[b, h] = np.where(live, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return o, lse


def fp8_attention(q, k, v, signs, causal, scale):
    """The FP8 forward's reference: exact attention of the dequantised rotated operands.
    q, k, v float32 (the 16-bit inputs' values).  Returns (o, lse, prep)."""
    B, Hq, Nq, d = q.shape
    _, Hkv, Nkv, _ = k.shape
    prep = prepare(q, k, v, signs)
    qd, kd, vd = dequantized(prep, B, Hq, Hkv, Nq, Nkv, d)
    o, lse = attention_f64(qd, kd, vd, causal, scale)
    return o, lse, prep


def fp8_attention_per_tensor(q, k, v, causal, scale):
    """The baseline FP8 attention the pages compare incoherent processing against ("FlashAttention
    Explained", section "FP8 Attention and Incoherent Processing"): no rotation and one scale per
    tensor (all of Q, all of K, all of V; the same power-of-two rule as the blocks), then exact
    attention of the dequantised operands.  q, k, v float32.  Returns (o, lse)."""
    B, Hq, Nq, d = q.shape
    _, Hkv, Nkv, _ = k.shape
    deq = []
    for x in (q, k, v):
        codes, sc = quantize_planes(np.asarray(x, np.float32).reshape(1, -1, d))
        deq.append(e4m3_decode(codes).reshape(x.shape) * np.float64(sc[0]))
    return attention_f64(deq[0], deq[1], deq[2], causal, scale)
