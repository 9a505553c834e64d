"""Partitions of the emulator's work over ranks (one GPU each), host side only.

The work splits into independent units with no collective on the data path:
  - block-FMA vector sets by contiguous index ranges;
  - GEMM outputs by bands of rows (whole CTA tiles), never by K: a chain over K is
    sequential, and splitting it would change the result;
  - multi-word GEMMs by word pairs, whose fp32 products the owner of the output adds
    in the fixed order (i + j descending, then i ascending).
Concatenating the ranks' results in rank order gives the single-rank result.
"""
from __future__ import annotations


def vector_range(n: int, rank: int, world: int) -> tuple[int, int]:
    """[lo, hi) of the vector sets rank `rank` of `world` evaluates (sizes differ by at
    most one)."""
    q, r = divmod(n, world)
    lo = rank * q + min(rank, r)
    return lo, lo + q + (1 if rank < r else 0)


def row_band(M: int, rank: int, world: int, tile: int = 64) -> tuple[int, int]:
    """[lo, hi) of the output rows of rank `rank`: whole tiles of `tile` rows, the last
    band ragged."""
    tiles = (M + tile - 1) // tile
    lo_t, hi_t = vector_range(tiles, rank, world)
    return min(lo_t * tile, M), min(hi_t * tile, M)


def combine_order(n_words: int, truncated: bool) -> list[tuple[int, int]]:
    """The word pairs (i, j), 1-based, in the order their products are added."""
    out = []
    for s in range(2 * n_words, 1, -1):
        for i in range(1, n_words + 1):
            j = s - i
            if 1 <= j <= n_words and not (truncated and i + j > n_words + 1):
                out.append((i, j))
    return out


def word_pairs(n_words: int, truncated: bool, rank: int, world: int) -> list[tuple[int, int]]:
    """The word pairs whose products rank `rank` evaluates (round robin over the
    combine order); the combine itself runs on the rank that owns the output."""
    return [p for k, p in enumerate(combine_order(n_words, truncated)) if k % world == rank]
