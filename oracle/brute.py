"""Brute-force numpy statement of LLA decode, for tiny shapes only.

TEST INFRASTRUCTURE ONLY.  Independent of ``lla_oracle.c``: it materialises the
whole reconstructed K/V stack with matrix products, builds each RoPE rotation
as an explicit d x d matrix, and takes the softmax directly.  Used to check the
C oracle on shapes small enough for both to agree to ~1e-12.

Source: "Looped Latent Attention: Cross-Loop KV Compression for Looped
Transformers" (arXiv 2607.15456v2), §3 Eq. (2)-(3) and "RoPE and
reconstruction"; attention is the standard scaled dot product the paper leaves
unchanged.
"""
from __future__ import annotations

import numpy as np


def rotation_matrix(d: int, pos: float, base: float, style: int = 0) -> np.ndarray:
    """The d x d rotary matrix R(pos): block rotation of each frequency pair."""
    R = np.zeros((d, d))
    for f in range(d // 2):
        i0, i1 = (f, f + d // 2) if style == 0 else (2 * f, 2 * f + 1)
        ang = pos * base ** (-2.0 * f / d)
        c, s = np.cos(ang), np.sin(ang)
        R[i0, i0], R[i0, i1] = c, -s
        R[i1, i0], R[i1, i1] = s, c
    return R


def encode(x_stack: np.ndarray, mu: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """Eq. (2) for a batch of stacked-loop rows: (x - mu) @ W_down."""
    return (x_stack - mu) @ w_down


def reconstruct(c: np.ndarray, w_up_t: np.ndarray, mu_t: np.ndarray) -> np.ndarray:
    """Eq. (3): rows c [L][r] -> [L][d] = c @ W_up,t^T + mu_t."""
    return c @ w_up_t.T + mu_t


def decode_per_head(t, q, cache_k, cache_v, seq_lens, q_pos, w_up_k, w_up_v, mu_k, mu_v,
                    base=10000.0, style=0, pos_offset=0):
    """Per-head LLA decode at loop t.  Shapes as the C oracle: q [B][H][d],
    cache_* [B][H][L_max][r], w_up_* [T][H][d][r], mu_* [H][T*d]."""
    B, H, d = q.shape
    out = np.zeros((B, H, d))
    lse = np.zeros((B, H))
    for b in range(B):
        L = int(seq_lens[b])
        for h in range(H):
            if L == 0:
                lse[b, h] = -np.inf
                continue
            mu_kt = mu_k[h, t * d:(t + 1) * d]
            mu_vt = mu_v[h, t * d:(t + 1) * d]
            K = reconstruct(cache_k[b, h, :L], w_up_k[t, h], mu_kt)
            V = reconstruct(cache_v[b, h, :L], w_up_v[t, h], mu_vt)
            qr = rotation_matrix(d, q_pos[b] + pos_offset, base, style) @ q[b, h]
            Kr = np.stack([rotation_matrix(d, j + pos_offset, base, style) @ K[j]
                           for j in range(L)])
            s = Kr @ qr / np.sqrt(d)
            w = np.exp(s - s.max())
            out[b, h] = (w / w.sum()) @ V
            lse[b, h] = s.max() + np.log(w.sum())
    return out, lse


def decode_2d(t, q, cache_k, cache_v, seq_lens, q_pos, w_up_k, w_up_v, mu_k, mu_v,
              base=10000.0, style=0):
    """LLA-2D decode at loop t: one latent per token shared by all heads.
    cache_* [B][L_max][r], w_up_* [T][H*d][r], mu_* [T*H*d] (index (t*H+h)*d+e)."""
    B, H, d = q.shape
    out = np.zeros((B, H, d))
    lse = np.zeros((B, H))
    for b in range(B):
        L = int(seq_lens[b])
        for h in range(H):
            if L == 0:
                lse[b, h] = -np.inf
                continue
            rows = slice(h * d, (h + 1) * d)
            mu_kt = mu_k[(t * H + h) * d:(t * H + h + 1) * d]
            mu_vt = mu_v[(t * H + h) * d:(t * H + h + 1) * d]
            K = reconstruct(cache_k[b, :L], w_up_k[t][rows], mu_kt)
            V = reconstruct(cache_v[b, :L], w_up_v[t][rows], mu_vt)
            qr = rotation_matrix(d, q_pos[b], base, style) @ q[b, h]
            Kr = np.stack([rotation_matrix(d, j, base, style) @ K[j] for j in range(L)])
            s = Kr @ qr / np.sqrt(d)
            w = np.exp(s - s.max())
            out[b, h] = (w / w.sum()) @ V
            lse[b, h] = s.max() + np.log(w.sum())
    return out, lse


def hybrid_per_head(t, q, cache_k, cache_v, n_lat, q_pos, w_up_k, w_up_v, mu_k, mu_v,
                    k_win, v_win, n_win, win_pos, base=10000.0, style=0):
    """Hybrid attention with an exact window ("Hybrid Latent Attention for Looped
    Language Models", §3.4 Eq. (4)): the latent tokens' K/V stacks (Eq. (3) of the
    LLA page) and the window's exact K/V are concatenated, every key is rotated by
    its own rotation matrix, and one softmax runs over the whole row.  k_win /
    v_win [B][H][W][d] (keys before RoPE), window token w at position win_pos[b] + w."""
    B, H, d = q.shape
    out = np.zeros((B, H, d))
    lse = np.zeros((B, H))
    for b in range(B):
        nl, nw = int(n_lat[b]), int(n_win[b])
        for h in range(H):
            if nl + nw == 0:
                lse[b, h] = -np.inf
                continue
            K = reconstruct(cache_k[b, h, :nl], w_up_k[t, h], mu_k[h, t * d:(t + 1) * d])
            V = reconstruct(cache_v[b, h, :nl], w_up_v[t, h], mu_v[h, t * d:(t + 1) * d])
            K = np.concatenate([K, k_win[b, h, :nw]], axis=0)
            V = np.concatenate([V, v_win[b, h, :nw]], axis=0)
            pos = list(range(nl)) + [int(win_pos[b]) + w for w in range(nw)]
            qr = rotation_matrix(d, q_pos[b], base, style) @ q[b, h]
            Kr = np.stack([rotation_matrix(d, pos[j], base, style) @ K[j] for j in range(nl + nw)])
            s = Kr @ qr / np.sqrt(d)
            w = np.exp(s - s.max())
            out[b, h] = (w / w.sum()) @ V
            lse[b, h] = s.max() + np.log(w.sum())
    return out, lse


def decoupled_per_head(t, q, cache_k, cache_v, k_rope, seq_lens, q_pos, w_up_k, w_up_v, mu_k, mu_v,
                       base=10000.0, style=0):
    """Absorbed decoupled-RoPE decode (LLA page, Appendix J "Absorbed attention"):
    concatenated keys [content (Eq. (3), unrotated) ; R(j) r_j] against the query
    [q_c ; R(q_pos) q_r], the d_rope-wide rotation an explicit matrix, one softmax,
    scale 1/sqrt(d + d_rope).  q [B][H][d + d_rope], k_rope [B][H][L_max][d_rope]."""
    B, H, dq = q.shape
    d_rope = k_rope.shape[3]
    d = dq - d_rope
    out = np.zeros((B, H, d))
    lse = np.zeros((B, H))
    for b in range(B):
        L = int(seq_lens[b])
        for h in range(H):
            if L == 0:
                lse[b, h] = -np.inf
                continue
            K = reconstruct(cache_k[b, h, :L], w_up_k[t, h], mu_k[h, t * d:(t + 1) * d])
            V = reconstruct(cache_v[b, h, :L], w_up_v[t, h], mu_v[h, t * d:(t + 1) * d])
            Rk = np.stack([rotation_matrix(d_rope, j, base, style) @ k_rope[b, h, j] for j in range(L)])
            qfull = np.concatenate([q[b, h, :d], rotation_matrix(d_rope, q_pos[b], base, style) @ q[b, h, d:]])
            Kfull = np.concatenate([K, Rk], axis=1)
            s = Kfull @ qfull / np.sqrt(dq)
            w = np.exp(s - s.max())
            out[b, h] = (w / w.sum()) @ V
            lse[b, h] = s.max() + np.log(w.sum())
    return out, lse
