"""Pins for the oracle: what the paper and the mathematics fix, independent of the oracle.

Each test pins one part of ``oracle/lla_oracle.c`` to something other than
itself: values the paper prints (``tests/golden``), closed forms, exact
identities, special cases and an independent numpy brute force.  A dropped term,
a wrong sign or index, or a transposed operand in the oracle fails at least one.

Source: "Looped Latent Attention: Cross-Loop KV Compression for Looped
Transformers" (arXiv 2607.15456v2).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "compression.json")


def _rng(seed):
    return np.random.default_rng(seed)


def _random_case(seed, B, H, T, d, rk, rv, L_max, lens, variant=0):
    g = _rng(seed)
    if variant == 0:
        ck = g.standard_normal((B, H, L_max, rk))
        cv = g.standard_normal((B, H, L_max, rv))
        wk = g.standard_normal((T, H, d, rk)) / math.sqrt(rk)
        wv = g.standard_normal((T, H, d, rv)) / math.sqrt(rv)
        mk = g.standard_normal((H, T * d)) * math.sqrt(0.1)
        mv = g.standard_normal((H, T * d)) * math.sqrt(0.1)
    else:
        ck = g.standard_normal((B, L_max, rk))
        cv = g.standard_normal((B, L_max, rv))
        wk = g.standard_normal((T, H * d, rk)) / math.sqrt(rk)
        wv = g.standard_normal((T, H * d, rv)) / math.sqrt(rv)
        mk = g.standard_normal((T * H * d,)) * math.sqrt(0.1)
        mv = g.standard_normal((T * H * d,)) * math.sqrt(0.1)
    q = g.standard_normal((B, H, d))
    sl = np.array(lens, dtype=np.int32)
    qp = np.maximum(sl - 1, 0).astype(np.int32)
    return dict(q=q, cache_k=ck, cache_v=cv, seq_lens=sl, q_pos=qp, w_up_k=wk, w_up_v=wv,
                mu_k=mk, mu_v=mv)


# ---------------------------------------------------------------- sizes (Eq. 4, Table 5, 8)

def test_compression_ratio_matches_printed_values():
    gold = json.load(open(GOLDEN))
    for row in gold["rho"]:
        dm = oracle.dims(row["T"], 16, row["d"], row["r_k"], row["r_v"])
        assert round(oracle.compression_ratio(dm), 2) == pytest.approx(row["rho"], abs=1e-9), row


def test_cache_bytes_per_token_match_table5():
    gold = json.load(open(GOLDEN))
    for row in gold["kib_per_token_16bit"]:
        dm = oracle.dims(row["T"], row["H"], row["d"], row["r_k"], row["r_v"])
        teacher = oracle.teacher_scalars_per_token(dm, row["D"]) * 2 / 1024
        lla = oracle.latent_scalars_per_token(dm, row["D"]) * 2 / 1024
        assert teacher == row["teacher"] and lla == row["lla"], row
    row = gold["gib_at_1m_context_16bit"][0]
    for (rk, rv), key in (((96, 160), "lla_4x"), ((16, 32), "lla_21x")):
        dm = oracle.dims(row["T"], row["H"], row["d"], rk, rv)
        gib = oracle.latent_scalars_per_token(dm, row["D"]) * 2 * 2 ** 20 / 2 ** 30
        assert gib == row[key]
        assert oracle.teacher_scalars_per_token(dm, row["D"]) * 2 * 2 ** 20 / 2 ** 30 == row["teacher"]


def test_lla2d_ratio_folds_heads():
    # §3 "The LLA-2D variant": the cache drops by a further factor H.
    per_head = oracle.dims(4, 16, 128, 128, 256, variant=0)
    two_d = oracle.dims(4, 16, 128, 128, 256, variant=1)
    assert oracle.compression_ratio(two_d) == pytest.approx(16 * oracle.compression_ratio(per_head))
    assert oracle.compression_ratio(two_d) == pytest.approx(2 * 4 * 16 * 128 / 384)


# ---------------------------------------------------------------- bf16 rounding

def test_round_bf16_matches_library_conversion():
    g = _rng(1)
    vals = np.concatenate([g.standard_normal(20000).astype(np.float32),
                           (g.standard_normal(2000) * 1e-30).astype(np.float32),
                           (g.standard_normal(2000) * 1e30).astype(np.float32),
                           # below 2^-126: bf16 subnormals, spaced 2^-133
                           (g.standard_normal(2000) * 2.0 ** -128).astype(np.float32),
                           (g.standard_normal(500) * 2.0 ** -136).astype(np.float32),
                           # next to the largest finite bf16 (2^127 (2 - 2^-7)): some
                           # stay finite, the rest round to infinity
                           (np.sign(g.standard_normal(2000)) *
                            g.uniform(3.37e38, 3.40e38, 2000)).astype(np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in vals])
    assert np.isinf(ref).any() and np.isfinite(ref[-2000:]).any()
    assert (np.abs(ref[(ref != 0) & np.isfinite(ref)]) < 2.0 ** -126).any()
    assert np.array_equal(got, ref)


def test_round_bf16_edges():
    """Edges of the bf16 range written out: the largest finite value, the midpoint to
    2^128 (ties to the even neighbour, which is past the range: infinity), the smallest
    subnormal 2^-133 and half of it (a tie to the even neighbour, zero)."""
    big = 2.0 ** 127 * (2 - 2.0 ** -7)
    assert oracle.round_bf16(big) == big
    assert oracle.round_bf16(2.0 ** 127 * (2 - 2.0 ** -8)) == np.inf
    assert oracle.round_bf16(-(2.0 ** 127 * (2 - 2.0 ** -8) - 2.0 ** 110)) == -big
    assert oracle.round_bf16(2.0 ** -133) == 2.0 ** -133
    assert oracle.round_bf16(2.0 ** -134) == 0.0
    assert oracle.round_bf16(3 * 2.0 ** -134) == 2.0 ** -132
    assert oracle.round_bf16(1.4 * 2.0 ** -130) == 2.0 ** -130 + 3 * 2.0 ** -133


def test_round_bf16_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> even mantissa (1.0)
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3*2^-8 lies halfway between 1+2^-7 and 1+2^-6 -> even (1+2^-6)
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert oracle.round_bf16(-(1.0 + 2.0 ** -8 + 2.0 ** -30)) == -(1.0 + 2.0 ** -7)


# ---------------------------------------------------------------- brute force (tiny shapes)

@pytest.mark.parametrize("style", [0, 1])
@pytest.mark.parametrize("T,rk,rv", [(1, 16, 32), (2, 32, 16), (2, 16, 16)])
def test_decode_matches_brute_force(T, rk, rv, style):
    B, H, d, L_max = 2, 2, 128, 8
    c = _random_case(100 + T + rk + style, B, H, T, d, rk, rv, L_max, [8, 5])
    dm = oracle.dims(T, H, d, rk, rv, rope_style=style)
    for t in range(T):
        o, l, _ = oracle.decode(dm, t, **c)
        ob, lb = brute.decode_per_head(t, base=10000.0, style=style, **c)
        np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, lb, rtol=0, atol=1e-12)


def test_decode_2d_matches_brute_force():
    B, H, T, d, rk, rv, L_max = 2, 2, 2, 128, 32, 16, 7
    c = _random_case(7, B, H, T, d, rk, rv, L_max, [7, 3], variant=1)
    dm = oracle.dims(T, H, d, rk, rv, variant=1)
    for t in range(T):
        o, l, _ = oracle.decode(dm, t, **c)
        ob, lb = brute.decode_2d(t, **c)
        np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("variant", [0, 1])
def test_encode_matches_brute_force(variant):
    g = _rng(3)
    T, H, d, r, B, L_max, N = 2, 2, 128, 32, 2, 6, 5
    width = T * d if variant == 0 else T * H * d
    if variant == 0:
        x = g.standard_normal((N, H, width))
        w = g.standard_normal((H, width, r))
        mu = g.standard_normal((H, width))
        cache = np.full((B, H, L_max, r), -7.0)
    else:
        x = g.standard_normal((N, width))
        w = g.standard_normal((width, r))
        mu = g.standard_normal((width,))
        cache = np.full((B, L_max, r), -7.0)
    seq_idx = np.array([0, 1, 1, 0, 1], np.int32)
    pos = np.array([0, 5, 2, 3, 0], np.int32)
    dm = oracle.dims(T, H, d, r, r, variant=variant)
    oracle.encode(dm, x, seq_idx, pos, w, mu, r, cache)
    for n in range(N):
        if variant == 0:
            for h in range(H):
                ref = brute.encode(x[n, h], mu[h], w[h])
                np.testing.assert_allclose(cache[seq_idx[n], h, pos[n]], ref, atol=1e-11)
        else:
            ref = brute.encode(x[n], mu, w)
            np.testing.assert_allclose(cache[seq_idx[n], pos[n]], ref, atol=1e-11)


# ---------------------------------------------------------------- exact identities

@pytest.mark.parametrize("T", [4, 2, 1])
def test_exact_recovery_with_full_rank_orthonormal_codec(T):
    """§3 "Initialization and conversion": with W_down orthonormal of rank T*d and
    W_up,t its loop-t row slice, Eq. (2)-(3) return every loop's K/V exactly, so LLA
    decode equals uncompressed attention (the teacher)."""
    H, d, B, L_max = 2, 128, 2, 9
    r = T * d
    g = _rng(40 + T)
    lens = np.array([9, 4], np.int32)
    q_pos = lens - 1
    dm = oracle.dims(T, H, d, r, r)
    # teacher K/V per loop: [B][H][L][T][d]
    Kt = g.standard_normal((B, H, L_max, T, d))
    Vt = g.standard_normal((B, H, L_max, T, d))
    mu_k = g.standard_normal((H, T * d)) * 0.3
    mu_v = g.standard_normal((H, T * d)) * 0.3
    wd_k = np.stack([np.linalg.qr(g.standard_normal((r, r)))[0] for _ in range(H)])
    wd_v = np.stack([np.linalg.qr(g.standard_normal((r, r)))[0] for _ in range(H)])
    # W_up,t[h] = rows t*d..(t+1)*d of W_down[h]  ->  [T][H][d][r]
    wu_k = np.stack([wd_k[:, t * d:(t + 1) * d, :] for t in range(T)])
    wu_v = np.stack([wd_v[:, t * d:(t + 1) * d, :] for t in range(T)])
    cache_k = np.zeros((B, H, L_max, r))
    cache_v = np.zeros((B, H, L_max, r))
    N = B * L_max
    seq_idx = np.repeat(np.arange(B, dtype=np.int32), L_max)
    pos = np.tile(np.arange(L_max, dtype=np.int32), B)
    xk = Kt.transpose(0, 2, 1, 3, 4).reshape(N, H, T * d)   # Eq. (1) stacking t*d+i
    xv = Vt.transpose(0, 2, 1, 3, 4).reshape(N, H, T * d)
    oracle.encode(dm, xk, seq_idx, pos, wd_k, mu_k, r, cache_k)
    oracle.encode(dm, xv, seq_idx, pos, wd_v, mu_v, r, cache_v)
    q = g.standard_normal((B, H, d))
    for t in range(T):
        o, l, _ = oracle.decode(dm, t, q, cache_k, cache_v, lens, q_pos, wu_k, wu_v, mu_k, mu_v)
        os_, ls_ = oracle.sdpa(dm, q, np.ascontiguousarray(Kt[:, :, :, t]),
                               np.ascontiguousarray(Vt[:, :, :, t]), lens, q_pos)
        np.testing.assert_allclose(o, os_, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, ls_, rtol=0, atol=1e-12)


def test_absorbed_value_path_identity():
    """Appendix J "Absorbed attention": sum_i a_i W c_i = W sum_i a_i c_i."""
    c = _random_case(5, 2, 3, 4, 128, 96, 160, 33, [33, 17])
    dm = oracle.dims(4, 3, 128, 96, 160)
    for t in range(4):
        o0, l0, _ = oracle.decode(dm, t, v_mode=0, **c)
        o1, l1, _ = oracle.decode(dm, t, v_mode=1, **c)
        np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
        assert np.array_equal(l0, l1)


# ---------------------------------------------------------------- special cases

def test_softmax_weights_sum_to_one_constant_values():
    """W_up,v = 0 and mu_v = 1 make every v_j = 1: the output is sum_j p_j = 1."""
    c = _random_case(8, 3, 2, 4, 128, 96, 160, 40, [40, 1, 23])
    c["w_up_v"] = np.zeros_like(c["w_up_v"])
    c["mu_v"] = np.ones_like(c["mu_v"])
    o, _, _ = oracle.decode(oracle.dims(4, 2, 128, 96, 160), 2, **c)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-14)


def _one_hot_wup(T, H, d, r):
    w = np.zeros((T, H, d, r))
    for e in range(min(d, r)):
        w[:, :, e, e] = 1.0
    return w


def test_single_token_returns_its_value():
    """L = 1: all weight on token 0, out = v_0 = c_v,0 W^T + mu_v,t; lse = s_0."""
    T, H, d, rk, rv = 2, 2, 128, 32, 128
    c = _random_case(9, 2, H, T, d, rk, rv, 4, [1, 1])
    c["w_up_v"] = _one_hot_wup(T, H, d, rv)
    dm = oracle.dims(T, H, d, rk, rv)
    for t in range(T):
        o, l, s = oracle.decode(dm, t, want_scores=True, **c)
        expect = c["cache_v"][:, :, 0, :] + c["mu_v"][None, :, t * d:(t + 1) * d]
        np.testing.assert_array_equal(o, expect)
        np.testing.assert_array_equal(l, s[:, :, 0])


def test_zero_query_gives_uniform_mean_over_exactly_L_tokens():
    """q = 0: every score is 0, weights 1/L, lse = ln L; slots >= L must not count."""
    T, H, d, rk, rv = 2, 2, 128, 16, 128
    c = _random_case(10, 3, H, T, d, rk, rv, 12, [12, 5, 1])
    c["q"] = np.zeros_like(c["q"])
    c["w_up_v"] = _one_hot_wup(T, H, d, rv)
    c["cache_v"][1, :, 5:, :] = 1e6      # padding beyond seq_lens[1]
    dm = oracle.dims(T, H, d, rk, rv)
    o, l, _ = oracle.decode(dm, 1, **c)
    for b, L in enumerate([12, 5, 1]):
        expect = c["cache_v"][b, :, :L, :].mean(axis=1) + c["mu_v"][:, d:2 * d]
        np.testing.assert_allclose(o[b], expect, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l[b], math.log(L), rtol=0, atol=1e-14)


def test_empty_sequence():
    c = _random_case(11, 2, 2, 2, 128, 16, 32, 4, [0, 3])
    o, l, _ = oracle.decode(oracle.dims(2, 2, 128, 16, 32), 0, **c)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(l[0]))
    assert np.all(np.isfinite(l[1]))


@pytest.mark.parametrize("style", [0, 1])
def test_rope_and_scale_closed_form(style):
    """RoPE after reconstruction with theta_f = base^(-2f/d), scale 1/sqrt(d):
    q = a*e_i0, k_j = e_i0 gives s_j = a*cos((p-j)theta_f)/sqrt(d); k_j = e_i1 gives
    a*sin((p-j)theta_f)/sqrt(d), where (i0, i1) is frequency f's pair."""
    T, H, d, r = 1, 1, 128, 16
    L, p, a, base = 50, 49, 3.0, 10000.0
    for f in (0, 1, 17, 63):
        i0, i1 = (f, f + 64) if style == 0 else (2 * f, 2 * f + 1)
        for tgt, fn in ((i0, math.cos), (i1, math.sin)):
            wk = np.zeros((T, H, d, r)); wk[0, 0, tgt, 0] = 1.0
            ck = np.zeros((1, H, L, r)); ck[..., 0] = 1.0
            q = np.zeros((1, H, d)); q[0, 0, i0] = a
            c = dict(q=q, cache_k=ck, cache_v=np.zeros((1, H, L, r)),
                     seq_lens=np.array([L], np.int32), q_pos=np.array([p], np.int32),
                     w_up_k=wk, w_up_v=np.zeros((T, H, d, r)),
                     mu_k=np.zeros((H, T * d)), mu_v=np.zeros((H, T * d)))
            _, _, s = oracle.decode(oracle.dims(T, H, d, r, r, rope_style=style), 0,
                                    want_scores=True, **c)
            theta = base ** (-2.0 * f / d)
            expect = np.array([a * fn((p - j) * theta) / math.sqrt(d) for j in range(L)])
            np.testing.assert_allclose(s[0, 0, :L], expect, rtol=0, atol=1e-13)


def test_rope_shift_invariance():
    """Shifting the query and every key position by the same offset leaves attention unchanged."""
    c = _random_case(12, 2, 2, 2, 128, 32, 64, 20, [20, 9])
    dm = oracle.dims(2, 2, 128, 32, 64)
    o0, l0, _ = oracle.decode(dm, 1, **c)
    o1, l1, _ = oracle.decode(dm, 1, pos_offset=777, **c)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-10)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-10)


def test_mean_is_loop_slice():
    """Eq. (3) adds mu_t, the t-th d-slice of the codec mean: zero latents give out = mu_v,t."""
    T, H, d = 4, 2, 128
    c = _random_case(13, 1, H, T, d, 16, 32, 6, [6])
    c["cache_v"] = np.zeros_like(c["cache_v"])
    dm = oracle.dims(T, H, d, 16, 32)
    for t in range(T):
        o, _, _ = oracle.decode(dm, t, **c)
        np.testing.assert_allclose(o[0], c["mu_v"][:, t * d:(t + 1) * d], rtol=0, atol=1e-14)


def test_encode_of_mean_is_zero():
    """Eq. (2) is centred: x = mu gives c = 0."""
    g = _rng(14)
    T, H, d, r = 2, 2, 128, 48
    mu = g.standard_normal((H, T * d))
    w = g.standard_normal((H, T * d, r))
    cache = np.full((1, H, 3, r), 5.0)
    oracle.encode(oracle.dims(T, H, d, r, r), mu[None], np.array([0], np.int32),
                  np.array([1], np.int32), w, mu, r, cache)
    assert np.all(cache[0, :, 1] == 0.0)
    assert np.all(cache[0, :, 0] == 5.0) and np.all(cache[0, :, 2] == 5.0)


@pytest.mark.parametrize("variant", [0, 1])
def test_encode_rounds_each_latent_once_to_bf16(variant):
    """With rounding asked for, each stored latent is the nearest bf16 of the exact sum
    (R6): equal to the unrounded encode rounded element by element, every value on the
    bf16 grid (a float32 -> bf16 library round trip leaves it unchanged), and most of the
    written values differ from the unrounded ones."""
    g = _rng(31)
    T, H, d, r, B, L_max, N = 2, 2, 128, 32, 2, 4, 3
    width = T * d if variant == 0 else T * H * d
    shape_x = (N, H, width) if variant == 0 else (N, width)
    shape_w = (H, width, r) if variant == 0 else (width, r)
    shape_mu = (H, width) if variant == 0 else (width,)
    shape_c = (B, H, L_max, r) if variant == 0 else (B, L_max, r)
    x, w, mu = g.standard_normal(shape_x), g.standard_normal(shape_w), g.standard_normal(shape_mu)
    seq_idx, pos = np.array([1, 0, 1], np.int32), np.array([3, 0, 1], np.int32)
    dm = oracle.dims(T, H, d, r, r, variant=variant)
    exact = oracle.encode(dm, x, seq_idx, pos, w, mu, r, np.zeros(shape_c))
    rounded = oracle.encode(dm, x, seq_idx, pos, w, mu, r, np.zeros(shape_c), round_to_bf16=True)
    np.testing.assert_array_equal(rounded, np.vectorize(oracle.round_bf16)(exact))
    lib = torch.from_numpy(rounded.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(rounded, lib)
    written = N * r * (H if variant == 0 else 1)
    assert np.count_nonzero(rounded != exact) > written // 2


def test_encode_layout_structured_exact():
    """Selector W_down and integer x: c[k] = x[u(k)] exactly, in slot (seq_idx, pos) of head h;
    every other slot keeps its canary."""
    T, H, d, r, B, L_max = 2, 3, 128, 32, 3, 5
    N = 4
    seq_idx = np.array([2, 0, 2, 1], np.int32)
    pos = np.array([4, 0, 1, 3], np.int32)
    u_of_k = (np.arange(r) * 7 + 3) % (T * d)
    w = np.zeros((H, T * d, r))
    for h in range(H):
        w[h, u_of_k, np.arange(r)] = 1.0
    x = np.zeros((N, H, T * d))
    for n in range(N):
        for h in range(H):
            x[n, h] = 1000 * n + 100 * h + (np.arange(T * d) % 97)
    cache = np.full((B, H, L_max, r), -12345.0)
    oracle.encode(oracle.dims(T, H, d, r, r), x, seq_idx, pos, w, np.zeros((H, T * d)), r,
                  cache, round_to_bf16=False)
    touched = np.zeros((B, H, L_max), bool)
    for n in range(N):
        for h in range(H):
            np.testing.assert_array_equal(cache[seq_idx[n], h, pos[n]],
                                          1000 * n + 100 * h + (u_of_k % 97))
            touched[seq_idx[n], h, pos[n]] = True
    assert np.all(cache[~touched] == -12345.0)
