"""Causal tile listing of the FA-2 loop (test infrastructure).

Written from "FlashAttention and GPU Data Movement", section 2.1 ("Skip bound and causal
mask are two different operations") and exercise 4: with 1-based tiles, query tile i covers
rows Br*(i-1)+1 .. Br*i and K/V tile j covers columns Bc*(j-1)+1 .. Bc*j.  A K/V tile is
loaded when it holds at least one column at or before the query tile's last row (the skip
bound), and it needs the element mask when some column lies after some row of the tile.
"""
from __future__ import annotations


def causal_tiles(i: int, Br: int, Bc: int, N: int):
    """For 1-based query tile ``i`` of a square causal problem of length N.

    Returns a dict:
      loaded   - 1-based K/V tiles the skip bound keeps,
      unmasked - the loaded tiles every row of the query tile may see in full,
      masked   - the loaded tiles that need the element mask,
      empty_rows[j] - for each masked tile j, the 1-based rows of the query tile that see
                      no column of tile j at all.
    """
    first_row = Br * (i - 1) + 1
    last_row = min(Br * i, N)
    loaded = []
    j = 1
    while Bc * (j - 1) + 1 <= last_row and Bc * (j - 1) + 1 <= N:
        loaded.append(j)
        j += 1
    unmasked = [j for j in loaded if min(Bc * j, N) <= first_row]
    masked = [j for j in loaded if j not in unmasked]
    empty_rows = {}
    for j in masked:
        first_col = Bc * (j - 1) + 1
        empty_rows[j] = [r for r in range(first_row, last_row + 1) if first_col > r]
    return {"loaded": loaded, "unmasked": unmasked, "masked": masked, "empty_rows": empty_rows}
