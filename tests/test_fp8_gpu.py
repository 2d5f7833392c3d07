"""GPU parity of the FP8 forward with incoherent processing (attn_fwd_fp8) against the FP8 oracle.

"FlashAttention Explained", section "FP8 Attention and Incoherent Processing".

Three layers:
  * the preparation (rotation, block scales, E4M3 codes, V transposed) is integer work decided in
    fp32 on both sides: codes and scales must be bit-identical to the oracle's;
  * O and L against the exact (fp64) attention of the dequantised operands.  The kernel feeds P
    to the P V product as E4M3 codes (of 2^5 p), which the oracle does not: the tolerance is that
    rounding's bound.  A code is within half a step of 2^5 p: 2^-4 of it for a normal code, 2^-10
    for a subnormal one (2^5 p < 2^-6).  The kernel's p are in units where its running maximum is
    at or below the row maximum (so p >= p' = exp(s - max s), and a subnormal code needs
    p' < 2^-11), earlier tiles are rescaled by factors <= 1, and its row sum l is taken from the
    unrounded p, so per element
        |dO_ic| <= 2^-4 sum_j p'_j |v_jc| / l' + 2^-15 sum_{j: p'_j < 2^-11} |v_jc| / l'
    over the visible keys, l' = sum_j p'_j.  Added to it: 2^-9 of the first term for the fp32
    sums and exp2, and half a unit of the stored output type.  L is the log of the unrounded row
    sum: within 1e-3.
  * an accuracy gate on inputs with 0.1% large outliers (16 times the rest) in Q and K: against
    the exact attention of the original inputs, the rotation must lower the RMS error of O, and
    the GPU's error must stay within that of the oracle's FP8 model plus the P rounding.
"""
import numpy as np
import pytest

import oracle
import synthetic as syn
from oracle import fp8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    import exact_io_aware_09_gb300 as m

    return m


def as_f32(bits, dt):
    return syn.bits_to_float32(bits, dt)


def run_fp8(attn, q, k, v, dt, causal, scale, signs, keep_workspace=False):
    import torch

    qt, kt, vt = (syn.bits_to_tensor(x, dt, "cuda") for x in (q, k, v))
    B, Hq, Nq, d = q.shape
    _, Hkv, Nkv, _ = k.shape
    st = torch.from_numpy(signs).to("cuda") if signs is not None else None
    ws = torch.full((max(1, attn.attn_fwd_fp8_workspace_bytes(B, Hq, Hkv, Nq, Nkv, d)),), 0xA5,
                    dtype=torch.uint8, device="cuda")
    o = torch.full_like(qt, float("nan"))
    lse = torch.full((B, Hq, Nq), float("nan"), device="cuda")
    o, lse = attn.attn_fwd_fp8(qt, kt, vt, st, o=o, lse=lse, causal=causal, scale=scale,
                               workspace=ws)
    assert attn.attn_poll_status() == 0
    og = o.float().cpu().numpy().astype(np.float64)
    lg = lse.cpu().numpy().astype(np.float64)
    return (og, lg, ws.cpu().numpy()) if keep_workspace else (og, lg)


P_SHIFT = 5                         # P enters the P V product as E4M3(2^5 p)
P_SUBNORMAL = 2.0 ** -(6 + P_SHIFT)  # p' below this may get a subnormal code
P_SUB_ERR = 2.0 ** -(10 + P_SHIFT)   # ... within this of 2^5 p / 2^5


def rounding_bounds(qd, kd, vd, causal, scale):
    """Per element: sum_j p_j |v_jc| / l and sum_{j: p_j < 2^-11} |v_jc| / l over the visible
    keys, p_j = exp(s_j - max s), from the dequantised operands (fp64)."""
    B, Hq, Nq, d = qd.shape
    Hkv, Nkv = kd.shape[1], kd.shape[2]
    G = Hq // Hkv
    A = np.zeros((B, Hq, Nq, d))
    Bs = np.zeros((B, Hq, Nq, d))
    for b in range(B):
        for h in range(Hq):
            s = scale * (qd[b, h] @ kd[b, h // G].T)
            vis = np.ones_like(s, dtype=bool)
            if causal:
                vis = np.arange(Nkv)[None, :] <= (np.arange(Nq)[:, None] + (Nkv - Nq))
            s = np.where(vis, s, -np.inf)
            m = s.max(axis=1)
            live = np.isfinite(m)
            p = np.where(vis & live[:, None], np.exp(s - np.where(live, m, 0.0)[:, None]), 0.0)
            l = np.where(live, p.sum(axis=1), 1.0)
            av = np.abs(vd[b, h // G])
            A[b, h] = (p @ av) / l[:, None]
            Bs[b, h] = ((vis & (p < P_SUBNORMAL)).astype(np.float64) @ av) / l[:, None]
    return A, Bs


def check_o_lse(og, lg, ro, rl, A, Bs, dt, what):
    half_unit = 2.0 ** -8 if dt == "bf16" else 2.0 ** -11
    tol = (2.0 ** -4 + 2.0 ** -9) * A + P_SUB_ERR * Bs + half_unit * np.abs(ro) + 1e-6
    err = np.abs(og - ro)
    assert np.all(np.isfinite(og)), f"{what}: non-finite O"
    bad = err > tol
    if bad.any():
        i = np.unravel_index(int(np.argmax(err / tol)), err.shape)
        raise AssertionError(f"{what}: O{tuple(int(x) for x in i)} err {err[i]:.3e} > "
                             f"{tol[i]:.3e} ({int(bad.sum())} elements)")
    empty = ~np.isfinite(rl)
    assert np.all(lg[empty] == -np.inf), f"{what}: L of a row with no key"
    assert np.all(og[empty] == 0.0), f"{what}: O of a row with no key"
    dl = np.abs(lg[~empty] - rl[~empty])
    assert dl.size == 0 or dl.max() <= 1e-3, f"{what}: |dL| {dl.max():.3e}"
    return float((err / tol).max()) if err.size else 0.0


def workspace_parts(ws, attn, B, Hq, Hkv, Nq, Nkv, d):
    off = attn.attn_fwd_fp8_workspace_offsets(B, Hq, Hkv, Nq, Nkv, d)
    nqt, nkt = -(-Nq // 128), -(-Nkv // 128)
    nkvp = nkt * 128
    pq, pk = B * Hq, B * Hkv
    take = lambda i, n: ws[off[i]:off[i] + n]
    return dict(
        q8=take(0, pq * Nq * d).reshape(pq, Nq, d),
        k8=take(1, pk * Nkv * d).reshape(pk, Nkv, d),
        vt8=take(2, pk * d * nkvp).reshape(pk, d, nkvp),
        sq=take(3, pq * nqt * 4).view(np.float32).reshape(pq, nqt),
        sk=take(4, pk * nkt * 4).view(np.float32).reshape(pk, nkt),
        sv=take(5, pk * 4).view(np.float32).reshape(pk),
    )


PREP = [
    # (B, Hq, Hkv, N_q, N_kv, dtype, rotate)
    (1, 2, 2, 128, 128, "bf16", True),
    (2, 4, 2, 200, 333, "f16", True),     # ragged tiles on both sides
    (1, 3, 1, 517, 300, "bf16", False),   # no rotation: plain block scaling
    (1, 2, 1, 1, 1000, "bf16", True),     # a one-row query tile
    (2, 32, 4, 2000, 1024, "bf16", True),  # 1,088 tiles: each block of the persistent preparation
                                           # walks about seven, around its four-stage ring
]


@pytest.mark.parametrize("shape", PREP, ids=lambda s: "x".join(map(str, s)))
def test_preparation_is_bit_exact(attn, shape):
    B, Hq, Hkv, Nq, Nkv, dt, rotate = shape
    d = 128
    cfg = syn.PrefillConfig("fp8", B, Hq, Hkv, Nq, Nkv, d, dt, True, 900 + sum(shape[:5]))
    q, k, v = cfg.host_inputs()
    q = syn.with_outliers(q, dt, cfg.seed + 11)
    signs = syn.random_signs(d, cfg.seed + 12) if rotate else None
    _, _, ws = run_fp8(attn, q, k, v, dt, True, cfg.scale, signs, keep_workspace=True)
    got = workspace_parts(ws, attn, B, Hq, Hkv, Nq, Nkv, d)
    ref = fp8.prepare(as_f32(q, dt), as_f32(k, dt), as_f32(v, dt), signs)
    np.testing.assert_array_equal(got["q8"], ref["q8"])
    np.testing.assert_array_equal(got["k8"], ref["k8"])
    np.testing.assert_array_equal(got["sq"], ref["sq"])
    np.testing.assert_array_equal(got["sk"], ref["sk"])
    np.testing.assert_array_equal(got["sv"], ref["sv"])
    np.testing.assert_array_equal(got["vt8"][:, :, :Nkv], ref["v8"].transpose(0, 2, 1))
    assert not got["vt8"][:, :, Nkv:].any(), "V^T padding keys must hold code 0"


@pytest.mark.parametrize("shape", [s for s in PREP if s[-1]], ids=lambda s: "x".join(map(str, s)))
def test_codes_are_within_a_step_of_the_exact_rotation(attn, shape):
    """Independent of the butterfly order: the kernel's Q and K codes against the rows rotated
    in fp64 by the explicit Sylvester-Hadamard matrix (oracle.fp8.rotate_exact) and divided by
    the kernel's block scales. A correctly rounded code lies within half an E4M3 spacing of that
    value; the fp32 rotation's rounding may tip one to its neighbour, never further. The scales
    are the smallest powers of two above amax / 448 of the exact rotation."""
    B, Hq, Hkv, Nq, Nkv, dt, _ = shape
    d = 128
    cfg = syn.PrefillConfig("fp8", B, Hq, Hkv, Nq, Nkv, d, dt, True, 900 + sum(shape[:5]))
    q, k, v = cfg.host_inputs()
    q = syn.with_outliers(q, dt, cfg.seed + 11)
    signs = syn.random_signs(d, cfg.seed + 12)
    _, _, ws = run_fp8(attn, q, k, v, dt, True, cfg.scale, signs, keep_workspace=True)
    got = workspace_parts(ws, attn, B, Hq, Hkv, Nq, Nkv, d)
    for x, codes, sc, N in ((q, got["q8"], got["sq"], Nq), (k, got["k8"], got["sk"], Nkv)):
        exact = fp8.rotate_exact(as_f32(x, dt).reshape(-1, N, d), signs)
        s_rows = np.repeat(sc.astype(np.float64), 128, axis=1)[:, :N, None]
        y = exact / s_rows
        deq = fp8.e4m3_decode(codes)
        far = np.abs(deq - y) > fp8.e4m3_spacing(y)
        assert not far.any(), f"{int(far.sum())} codes more than one step from the exact value"
        assert (codes == fp8.e4m3_encode(y)).mean() > 0.99
        for pl in range(exact.shape[0]):
            for t in range(sc.shape[1]):
                a = np.abs(exact[pl, t * 128:(t + 1) * 128]).max()
                assert a <= 448.0 * sc[pl, t] * (1 + 1e-6) and 448.0 * sc[pl, t] < 2 * a * (1 + 1e-6)


PARITY = [
    # (B, Hq, Hkv, N_q, N_kv, dtype, causal)
    (1, 1, 1, 128, 128, "bf16", False),
    (1, 2, 2, 256, 256, "f16", True),
    (2, 4, 2, 200, 333, "bf16", True),    # ragged, bottom-right causal
    (2, 4, 2, 200, 333, "bf16", False),
    (1, 2, 2, 400, 100, "f16", True),     # N_kv < N_q: top rows see no key
    (1, 3, 1, 517, 517, "bf16", True),    # 3 query heads per key/value head
    (1, 8, 1, 384, 384, "bf16", True),
    (1, 2, 2, 1, 1000, "bf16", True),     # one row sees every key
    (1, 2, 2, 1000, 1000, "bf16", True),  # several tiles: the lazy rescale at work
    (1, 1, 1, 255, 3000, "f16", False),
]


@pytest.mark.parametrize("shape", PARITY, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("rotate", [True, False], ids=["rot", "plain"])
def test_fp8_parity(attn, shape, rotate):
    B, Hq, Hkv, Nq, Nkv, dt, causal = shape
    d = 128
    cfg = syn.PrefillConfig("fp8", B, Hq, Hkv, Nq, Nkv, d, dt, causal, 950 + sum(shape[:5]))
    q, k, v = cfg.host_inputs()
    signs = syn.random_signs(d, cfg.seed + 3) if rotate else None
    og, lg = run_fp8(attn, q, k, v, dt, causal, cfg.scale, signs)
    ro, rl, prep = fp8.fp8_attention(as_f32(q, dt), as_f32(k, dt), as_f32(v, dt), signs, causal,
                                     cfg.scale)
    qd, kd, vd = fp8.dequantized(prep, B, Hq, Hkv, Nq, Nkv, d)
    A, Bs = rounding_bounds(qd, kd, vd, causal, cfg.scale)
    check_o_lse(og, lg, ro, rl, A, Bs, dt, f"shape {shape} rotate={rotate}")


def test_fp8_large_scores(attn):
    """Q scaled by 8: sharp rows, the maximum moving often (rescales), P near its bound."""
    B, Hq, Hkv, Nq, Nkv, d, dt = 1, 2, 1, 700, 700, 128, "bf16"
    cfg = syn.PrefillConfig("fp8", B, Hq, Hkv, Nq, Nkv, d, dt, True, 977, q_scale_pow2=3)
    q, k, v = cfg.host_inputs()
    signs = syn.random_signs(d, 978)
    og, lg = run_fp8(attn, q, k, v, dt, True, cfg.scale, signs)
    ro, rl, prep = fp8.fp8_attention(as_f32(q, dt), as_f32(k, dt), as_f32(v, dt), signs, True,
                                     cfg.scale)
    A, Bs = rounding_bounds(*fp8.dequantized(prep, B, Hq, Hkv, Nq, Nkv, d), True, cfg.scale)
    check_o_lse(og, lg, ro, rl, A, Bs, dt, "large scores")


def test_fp8_empty_key_side(attn):
    import torch

    q = torch.randn(1, 2, 64, 128, device="cuda").to(torch.bfloat16)
    k = torch.empty(1, 2, 0, 128, device="cuda", dtype=torch.bfloat16)
    o, lse = attn.attn_fwd_fp8(q, k, k, None)
    assert attn.attn_poll_status() == 0
    assert torch.all(o == 0) and torch.all(lse == float("-inf"))


def test_fp8_rejects_bad_signs(attn):
    import torch

    q = torch.randn(1, 1, 128, 128, device="cuda").to(torch.bfloat16)
    with pytest.raises(attn.AttnError):
        attn.attn_fwd_fp8(q, q, q, torch.ones(64, dtype=torch.int8, device="cuda"))
    x = q[..., :64].contiguous()
    with pytest.raises(attn.AttnError):
        attn.attn_fwd_fp8(x, x, x, None)   # d = 64: the FP8 kernel is built for d = 128


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_fp8_outlier_accuracy_gate(attn, causal):
    """0.1% of the Q and K entries 16 times larger than the rest: the randomised Hadamard
    rotation lowers the RMS error of O against exact attention of the original inputs, and the
    kernel's error is well below that of the pages' baseline FP8 attention (one scale per
    tensor, no rotation; modelled by the oracle without rounding P, which favours it)."""
    B, Hq, Hkv, Nq, Nkv, d, dt = 1, 4, 4, 1024, 1024, 128, "bf16"
    cfg = syn.PrefillConfig("fp8", B, Hq, Hkv, Nq, Nkv, d, dt, causal, 1200 + causal)
    q, k, v = cfg.host_inputs()
    q = syn.with_outliers(q, dt, 1210)
    k = syn.with_outliers(k, dt, 1211)
    exact, _ = oracle.attention_rows(q, k, v, dt, B, Hq, Hkv, Nq, Nkv, d, causal, cfg.scale)
    exact = exact.reshape(B, Hq, Nq, d)
    signs = syn.random_signs(d, 1212)
    rms = lambda o: float(np.sqrt(np.mean((o - exact) ** 2)))
    gpu_rot = rms(run_fp8(attn, q, k, v, dt, causal, cfg.scale, signs)[0])
    gpu_plain = rms(run_fp8(attn, q, k, v, dt, causal, cfg.scale, None)[0])
    model_rot = rms(fp8.fp8_attention(as_f32(q, dt), as_f32(k, dt), as_f32(v, dt), signs, causal,
                                      cfg.scale)[0])
    model_base = rms(fp8.fp8_attention_per_tensor(as_f32(q, dt), as_f32(k, dt), as_f32(v, dt),
                                                  causal, cfg.scale)[0])
    print(f"fp8 gate causal={causal}: gpu rotated {gpu_rot:.4g}, gpu unrotated {gpu_plain:.4g}, "
          f"model rotated {model_rot:.4g}, per-tensor baseline model {model_base:.4g}")
    assert gpu_rot < gpu_plain / 1.15, (gpu_rot, gpu_plain)
    assert gpu_rot < model_base / 1.2, (gpu_rot, model_base)
    assert gpu_rot <= 1.25 * model_rot + 2e-3, (gpu_rot, model_rot)


def test_fp8_full_size_sampled(attn):
    """The 70B-class GQA causal prefill (B=1, Hq=64, Hkv=8, N=8192, d=128): the query heads of
    key/value head 3, sampled rows, against the oracle (block scales are per head and tile, so a
    subset of heads is quantised exactly as in the full problem)."""
    import torch

    B, Hq, Hkv, N, d, dt = 1, 64, 8, 8192, 128, "bf16"
    cfg = syn.PrefillConfig("fp8", B, Hq, Hkv, N, N, d, dt, True, 1300)
    qt, kt, vt = cfg.device_inputs()
    signs = syn.random_signs(d, 1301)
    o, lse = attn.attn_fwd_fp8(qt, kt, vt, torch.from_numpy(signs).cuda(), causal=True,
                               scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    kv = 3
    heads = list(range(kv * 8, kv * 8 + 8))
    q = as_f32(syn.tensor_to_bits(qt[:, heads]), dt)
    k = as_f32(syn.tensor_to_bits(kt[:, kv:kv + 1]), dt)
    v = as_f32(syn.tensor_to_bits(vt[:, kv:kv + 1]), dt)
    prep = fp8.prepare(q, k, v, signs)
    qd, kd, vd = fp8.dequantized(prep, 1, 8, 1, N, N, d)
    rows = np.sort(np.random.default_rng(1302).choice(N, 96, replace=False))
    rows = np.unique(np.concatenate([rows, [0, 1, 127, 128, N - 1]]))
    og = o[:, heads].float().cpu().numpy()[:, :, rows].astype(np.float64)
    lg = lse[:, heads].cpu().numpy()[:, :, rows].astype(np.float64)
    ro = np.zeros_like(og)
    rl = np.zeros_like(lg)
    A = np.zeros_like(og)
    Bs = np.zeros_like(og)
    for hi in range(8):
        for ri, r in enumerate(rows):
            s = cfg.scale * (kd[0, 0, :r + 1] @ qd[0, hi, r])
            m = s.max()
            p = np.exp(s - m)
            l = p.sum()
            ro[0, hi, ri] = (p @ vd[0, 0, :r + 1]) / l
            rl[0, hi, ri] = m + np.log(l)
            av = np.abs(vd[0, 0, :r + 1])
            A[0, hi, ri] = (p @ av) / l
            Bs[0, hi, ri] = (p < P_SUBNORMAL).astype(np.float64) @ av / l
    check_o_lse(og, lg, ro, rl, A, Bs, dt, "GQA N=8192 sampled")
