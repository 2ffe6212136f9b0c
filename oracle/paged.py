"""Paged latent cache: the logical-to-physical page table, written out (test
infrastructure, like the rest of ``oracle/``).

Source: "Enabling dynamic computation in Looped LMs" (arXiv 2610.09013), §"Ragged
KV" (memory savings through page tables, as in vLLM: a pool of physical memory and
a logical-to-physical table) and Appendix A.1 "Page-table aliases for compact K/V
storage" (one page identifier per logical entry; several entries may name the same
physical page, reads may alias, writes may not).

Layout this module states: a pool ``[num_pages][H][page_size][r]`` and a table
``bt [B][max_pages]``; token j of (sequence b, head h) is row ``j % page_size`` of
head h of physical page ``bt[b][j // page_size]``.  The dense view of sequence b is
therefore the concatenation, over its logical pages in order, of those pages' rows.

Nothing here does arithmetic on latents: it only moves rows, so every function is
exact.
"""
from __future__ import annotations

import numpy as np


def gather(pool: np.ndarray, bt: np.ndarray, page_size: int, lens) -> np.ndarray:
    """Dense cache ``[B][H][max_pages * page_size][r]`` of a paged pool.  Rows of the
    logical pages that hold tokens j < lens[b] are copied from their physical pages;
    every other row is NaN (it names no stored token)."""
    B, max_pages = bt.shape
    _, H, P, r = pool.shape
    assert P == page_size
    out = np.full((B, H, max_pages * P, r), np.nan, dtype=np.float64)
    for b in range(B):
        used = (int(lens[b]) + P - 1) // P
        for lp in range(used):
            pg = int(bt[b, lp])
            out[b, :, lp * P:(lp + 1) * P, :] = pool[pg]
    return out


def scatter(dense: np.ndarray, bt: np.ndarray, page_size: int, lens, num_pages: int,
            fill: float = np.nan) -> np.ndarray:
    """Pool ``[num_pages][H][page_size][r]`` holding the rows of a dense cache
    ``[B][H][L][r]`` at the places the table names (the inverse of :func:`gather`
    for a table without aliases).  Pages no used entry names keep ``fill``."""
    B, max_pages = bt.shape
    _, H, L, r = dense.shape
    P = page_size
    pool = np.full((num_pages, H, P, r), fill, dtype=np.float64)
    for b in range(B):
        used = (int(lens[b]) + P - 1) // P
        for lp in range(used):
            pg = int(bt[b, lp])
            rows = dense[b, :, lp * P:min((lp + 1) * P, L), :]
            pool[pg, :, :rows.shape[1], :] = rows
    return pool


def slot(bt: np.ndarray, page_size: int, b: int, j: int):
    """(physical page, row) of token j of sequence b."""
    return int(bt[b, j // page_size]), j % page_size
