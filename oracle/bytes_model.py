"""Logical HBM-traffic model of one attention head (test infrastructure).

Written from "FlashAttention and GPU Data Movement", section 1.1 (the three-kernel
materialising baseline, table of reads and writes per kernel) and section 4 (the tiled FA-2
loop: Q read once, O written once, K and V re-read once per query tile; causal tiles are
skipped past the diagonal).  The model is cold-cache, exact bytes, no sector padding and
no logsumexp write unless ``lse=True`` (section 3.3 adds 4 bytes per query row).
"""
from __future__ import annotations


def _ceil(a: int, b: int) -> int:
    return -(-a // b)


def naive_traffic(N: int, d: int, b: int, causal: bool = False):
    """(reads, writes) of the explicit three-kernel baseline for one head.

    Kernel 1 reads Q, K and writes S; kernel 2 reads S and writes P; kernel 3 reads P, V and
    writes O.  ``causal=True`` is the pages' idealised lower-triangular variant that stores
    exactly half of each N x N matrix.
    """
    row = N * d * b                   # one of Q, K, V, O
    mat = N * N * b                   # S or P
    if causal:
        mat = mat // 2
    reads = (row + row) + mat + (mat + row)
    writes = mat + mat + row
    return reads, writes


def flash_traffic(N: int, d: int, b: int, Br: int, Bc: int, causal: bool = False,
                  lse: bool = False):
    """(reads, writes) of the FA-2 loop (Q outer, K/V inner) for one head.

    Query tile i covers rows [i*Br, min((i+1)*Br, N)).  Unmasked, it loads every K/V tile;
    causal, it loads the K/V tiles up to the one holding its last row (the skip bound).
    """
    n_q_tiles = _ceil(N, Br)
    n_kv_tiles = _ceil(N, Bc)
    kv_tile_bytes = Bc * d * b * 2    # one K tile and one V tile
    reads = N * d * b                 # Q, once
    for i in range(n_q_tiles):
        if causal:
            last_row = min((i + 1) * Br, N) - 1
            loaded = last_row // Bc + 1
        else:
            loaded = n_kv_tiles
        reads += loaded * kv_tile_bytes
    writes = N * d * b                # O, once
    if lse:
        writes += 4 * N
    return reads, writes


def bytes_model(N: int, d: int, b: int, scheme: str, causal: bool = False, Br: int = 128,
                Bc: int = 64, lse: bool = False) -> int:
    """Total logical traffic in bytes: scheme 'naive' or 'flash'."""
    if scheme == "naive":
        r, w = naive_traffic(N, d, b, causal)
    elif scheme == "flash":
        r, w = flash_traffic(N, d, b, Br, Bc, causal, lse)
    else:
        raise ValueError(scheme)
    return r + w
