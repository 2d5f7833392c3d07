"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and rounds them to the storage type.  It holds
none of the attention arithmetic, so both the fp64 oracle (``oracle/``) and the CUDA
path (``exact_io_aware_09_gb300``) may use it without sharing any of the method.

Recipe (the pages' workloads use iid N(0, 1) inputs and fp16/bf16 storage):

* host draws: ``numpy.random.Generator(PCG64(seed)).standard_normal(..., float32)``,
  rounded to the storage type with round-to-nearest-even;
* Q, K and V of a configuration use seeds ``seed``, ``seed + 1`` and ``seed + 2``;
* the x8 stress variant multiplies the ROUNDED Q by 8 (a power of two, so exact);
* decode lengths: ``Generator(PCG64(5000)).integers(1024, 32768, B, endpoint=True)``;
* large tensors may be drawn on the device instead, with a seeded
  ``torch.Generator('cuda')`` (``device_normal``); the bits are then copied back to the
  host for any oracle comparison, so both sides still see the same inputs.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

F16 = "f16"
BF16 = "bf16"


def _torch():
    import torch  # imported lazily: the oracle's CPU tests need only numpy

    return torch


def round_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to fp16 / bf16 (nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        torch = _torch()
        t = torch.from_numpy(x).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(f"unknown dtype {dtype!r}")


def host_normal_bits(shape, seed: int, dtype: str, scale_pow2: int = 0) -> np.ndarray:
    """iid N(0,1) draws rounded to ``dtype``; optional exact power-of-two scaling after rounding."""
    g = np.random.Generator(np.random.PCG64(seed))
    x = g.standard_normal(size=shape, dtype=np.float32)
    bits = round_bits(x, dtype)
    if scale_pow2:
        bits = scale_bits_pow2(bits, dtype, scale_pow2)
    return bits


def scale_bits_pow2(bits: np.ndarray, dtype: str, k: int) -> np.ndarray:
    """Multiply stored values by 2**k exactly (no overflow/underflow for N(0,1) draws, k <= 8)."""
    torch = _torch()
    tdt = torch.float16 if dtype == F16 else torch.bfloat16
    t = torch.from_numpy(bits.view(np.int16).copy()).view(tdt)
    y = (t.float() * float(2 ** k)).to(tdt)
    return y.view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_float32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Values of stored fp16 / bf16 bits as float32 (exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    if dtype == BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


def random_signs(d: int, seed: int) -> np.ndarray:
    """int8 [d] of independent, equally likely +-1 (the sign flips of a randomised Hadamard
    rotation)."""
    g = np.random.Generator(np.random.PCG64(seed))
    return np.where(g.random(d) < 0.5, -1, 1).astype(np.int8)


def with_outliers(bits: np.ndarray, dtype: str, seed: int, frac: float = 1e-3,
                  pow2: int = 4) -> np.ndarray:
    """A fraction ``frac`` of the entries, chosen at random, multiplied by 2**pow2 exactly
    (large outliers among N(0,1) activations)."""
    g = np.random.Generator(np.random.PCG64(seed))
    pick = g.random(bits.shape) < frac
    big = scale_bits_pow2(bits, dtype, pow2)
    return np.where(pick, big, bits).astype(np.uint16)


def torch_dtype(dtype: str):
    torch = _torch()
    return torch.float16 if dtype == F16 else torch.bfloat16


def bits_to_tensor(bits: np.ndarray, dtype: str, device="cpu"):
    """View uint16 bits as a torch fp16/bf16 tensor (copy to ``device``)."""
    torch = _torch()
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch_dtype(dtype))
    return t.to(device) if str(device) != "cpu" else t.clone()


def tensor_to_bits(t) -> np.ndarray:
    torch = _torch()
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16).copy()


def device_normal(shape, seed: int, dtype: str, device="cuda", scale_pow2: int = 0):
    """Seeded N(0,1) draws made on the device (for inputs too large to draw on the host)."""
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    t = x.to(torch_dtype(dtype))
    del x
    if scale_pow2:
        t = (t.float() * float(2 ** scale_pow2)).to(torch_dtype(dtype))
    return t


def decode_lengths(B: int, lo: int = 1024, hi: int = 32768, seed: int = 5000) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(seed))
    return g.integers(lo, hi, size=B, endpoint=True).astype(np.int64)


def cu_seqlens(lengths) -> np.ndarray:
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=cu[1:])
    return cu.astype(np.int32)


@dataclasses.dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    N_q: int
    N_kv: int
    d: int
    dtype: str
    causal: bool
    seed: int
    q_scale_pow2: int = 0  # 3 -> Q multiplied by 8 after rounding (stress)

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    def shapes(self):
        return ((self.B, self.Hq, self.N_q, self.d), (self.B, self.Hkv, self.N_kv, self.d))

    def flops(self) -> float:
        """4*B*Hq*N_q*N_kv*d, halved for causal (the pages' convention)."""
        f = 4.0 * self.B * self.Hq * self.N_q * self.N_kv * self.d
        return f / 2 if self.causal else f

    def host_inputs(self):
        qs, ks = self.shapes()
        q = host_normal_bits(qs, self.seed, self.dtype, self.q_scale_pow2)
        k = host_normal_bits(ks, self.seed + 1, self.dtype)
        v = host_normal_bits(ks, self.seed + 2, self.dtype)
        return q, k, v

    def device_inputs(self, device="cuda"):
        qs, ks = self.shapes()
        q = device_normal(qs, self.seed, self.dtype, device, self.q_scale_pow2)
        k = device_normal(ks, self.seed + 1, self.dtype, device)
        v = device_normal(ks, self.seed + 2, self.dtype, device)
        return q, k, v


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    dtype: str
    seed: int
    len_lo: int = 1024
    len_hi: int = 32768
    len_seed: int = 5000
    split: int = 512
    lengths_override: Optional[tuple] = None

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    def lengths(self) -> np.ndarray:
        if self.lengths_override is not None:
            return np.asarray(self.lengths_override, dtype=np.int64)
        return decode_lengths(self.B, self.len_lo, self.len_hi, self.len_seed)

    def kv_bytes(self) -> int:
        return int(self.lengths().sum()) * 2 * self.Hkv * self.d * 2

    def host_inputs(self):
        T = int(self.lengths().sum())
        q = host_normal_bits((self.B, self.Hq, self.d), self.seed, self.dtype)
        k = host_normal_bits((T, self.Hkv, self.d), self.seed + 1, self.dtype)
        v = host_normal_bits((T, self.Hkv, self.d), self.seed + 2, self.dtype)
        return q, k, v

    def device_inputs(self, device="cuda"):
        T = int(self.lengths().sum())
        q = device_normal((self.B, self.Hq, self.d), self.seed, self.dtype, device)
        k = device_normal((T, self.Hkv, self.d), self.seed + 1, self.dtype, device)
        v = device_normal((T, self.Hkv, self.d), self.seed + 2, self.dtype, device)
        return q, k, v


# The five workloads of the benchmark (shapes from the pages; seeds fixed here).
CONFIG1 = PrefillConfig("single_head_n256_d64_f16", 1, 1, 1, 256, 256, 64, F16, False, 1001)
CONFIG2 = PrefillConfig("gpt2_causal_b8_h12_n1024_d64_bf16", 8, 12, 12, 1024, 1024, 64, BF16, True, 2001)
CONFIG3A = PrefillConfig("long_b4_h32_n4096_d128_f16", 4, 32, 32, 4096, 4096, 128, F16, False, 3001)
CONFIG3B = PrefillConfig("long_causal_b4_h32_n4096_d128_f16", 4, 32, 32, 4096, 4096, 128, F16, True, 3001)
CONFIG3SA = PrefillConfig("long_x8_b4_h32_n4096_d128_f16", 4, 32, 32, 4096, 4096, 128, F16, False, 3001, 3)
CONFIG3SB = PrefillConfig("long_x8_causal_b4_h32_n4096_d128_f16", 4, 32, 32, 4096, 4096, 128, F16, True, 3001, 3)
CONFIG4 = PrefillConfig("gqa_causal_b1_hq64_hkv8_n8192_d128_bf16", 1, 64, 8, 8192, 8192, 128, BF16, True, 4001)
CONFIG5 = DecodeConfig("splitkv_decode_b64_hq64_hkv8_d128_bf16", 64, 64, 8, 128, BF16, 5001)

PREFILL_CONFIGS = [CONFIG1, CONFIG2, CONFIG3A, CONFIG3B, CONFIG3SA, CONFIG3SB, CONFIG4]


# ----------------------------------------------------------------------------------------
# paged KV cache layout (input generation only: where each token of a packed cache goes)
# ----------------------------------------------------------------------------------------
def causal_block_pattern(N_q: int, N_kv: int, seed: int = 11, block: int = 128) -> np.ndarray:
    """Block pattern of the block-sparse measurement, [ceil(N_q/block), ceil(N_kv/block)] uint8:
    each block on or below the diagonal kept with probability 1/2, plus the diagonal block and
    the first key block of every query tile (so that every row sees a key)."""
    nq, nk = -(-N_q // block), -(-N_kv // block)
    rng = np.random.default_rng(seed)
    m = (rng.random((nq, nk)) < 0.5).astype(np.uint8)
    for r in range(nq):
        m[r, r + 1:] = 0
        m[r, min(r, nk - 1)] = 1
        m[r, 0] = 1
    return m


def paged_layout(lengths, page_size: int, seed: int, spare_pages: int = 3):
    """A shuffled page pool for sequences of the given lengths.

    Returns (block_table int32 [B, max_pages] padded with -1, num_pages, page_of_token,
    slot_of_token): packed token cu[b] + t of sequence b goes to row slot_of_token of page
    page_of_token.  spare_pages unused pages are added to the pool.
    """
    lengths = np.asarray(lengths, dtype=np.int64)
    n_pages = (lengths + page_size - 1) // page_size
    num_pages = int(n_pages.sum()) + spare_pages
    perm = np.random.default_rng(seed).permutation(num_pages).astype(np.int32)
    max_pages = max(1, int(n_pages.max()) if len(n_pages) else 1)
    table = np.full((len(lengths), max_pages), -1, dtype=np.int32)
    page_of_token, slot_of_token = [], []
    used = 0
    for b, L in enumerate(lengths):
        table[b, :n_pages[b]] = perm[used:used + n_pages[b]]
        used += int(n_pages[b])
        t = np.arange(int(L), dtype=np.int64)
        page_of_token.append(table[b][t // page_size].astype(np.int64))
        slot_of_token.append(t % page_size)
    cat = lambda xs: np.concatenate(xs) if xs else np.zeros(0, dtype=np.int64)
    return table, num_pages, cat(page_of_token), cat(slot_of_token)


def scatter_to_pages(cache, num_pages, page_size, page_of_token, slot_of_token, fill=None):
    """[T, Hkv, d] packed cache (numpy or torch) -> [num_pages, page_size, Hkv, d] pool; rows no
    token occupies hold `fill` (numpy: random bits of the given generator seed; torch: NaN)."""
    if isinstance(cache, np.ndarray):
        shape = (num_pages, page_size) + cache.shape[1:]
        if fill is None:
            pool = np.zeros(shape, dtype=cache.dtype)
        else:
            pool = np.random.default_rng(fill).integers(0, 65535, size=shape).astype(cache.dtype)
        pool[page_of_token, slot_of_token] = cache
        return pool
    import torch

    pool = torch.full((num_pages, page_size) + tuple(cache.shape[1:]), float("nan"),
                      dtype=cache.dtype, device=cache.device)
    pool[torch.from_numpy(page_of_token).to(cache.device),
         torch.from_numpy(slot_of_token).to(cache.device)] = cache
    return pool
