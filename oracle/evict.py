"""Token eviction over the latent cache, written out (test infrastructure, like the
rest of ``oracle/``).

Source: "Looped Latent Attention: Cross-Loop KV Compression for Looped Transformers"
(arXiv 2607.15456v2), Appendix D "Token-eviction composition table" (Table 9: a
StreamingLLM/H2O-style budget of sink 4 + window 256 composed with LLA) and
Appendix J "Eviction and long-context prefill" (the sequence and recurrence axes
compose multiplicatively: only the kept tokens' latents are stored).

Budget kept for a sequence of L cached tokens, sink S and window W: tokens 0..S-1
and the W newest, L-W..L-1.  When L > S + W the kept latents are stored in order in
slots 0..S+W-1 (sinks first, then the window, oldest first) and the sequence's length
becomes S + W; at or below the budget nothing changes.  A decode over the kept cache
rotates slot j at position j: positions within the kept cache, the re-indexing of
StreamingLLM.

Only rows move here, so every function is exact.
"""
from __future__ import annotations

import numpy as np


def kept_tokens(L: int, sink: int, window: int):
    """Indices of the tokens a budget of (sink, window) keeps, in cache order."""
    if L <= sink + window:
        return list(range(L))
    return list(range(sink)) + list(range(L - window, L))


def evict(cache: np.ndarray, lens, sink: int, window: int):
    """(new cache, new lengths) for a dense per-head cache [B][H][L_max][r]: every
    sequence over budget keeps its sinks and its window, compacted in order; rows past
    the new length are left as they were."""
    out = cache.copy()
    new_lens = np.array(lens, dtype=np.int64).copy()
    for b in range(cache.shape[0]):
        keep = kept_tokens(int(lens[b]), sink, window)
        if len(keep) == int(lens[b]):
            continue
        out[b, :, :len(keep)] = cache[b][:, keep]
        new_lens[b] = len(keep)
    return out, new_lens
