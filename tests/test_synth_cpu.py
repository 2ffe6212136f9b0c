"""The seeded input recipe, checked on the CPU: shapes and layouts of every tensor a
workload draws, each distribution's spread, the length range, q_pos = seq_lens - 1,
the storage rounding, and that a seed fixes every value (the GPU arm, the oracle and the
reference arm all draw their inputs through these calls)."""
import dataclasses
import math

import numpy as np
import pytest
import torch

from looped_transformer_cross_gb300.synth import (WORKLOADS, Workload, make_decode_inputs,
                                                 make_decoupled_inputs, make_window_inputs, widen)


def _small(name, B=3, L_max=256, lo=100, hi=256):
    """A workload's geometry (T, H, d, ranks, variant) at a CPU-sized batch and length."""
    return dataclasses.replace(WORKLOADS[name], B=B, L_max=L_max, len_lo=lo, len_hi=hi, N_encode=5)


@pytest.mark.parametrize("name", ["ouro1.4b_rho4_b32_4k", "ouro1.4b_rho21_b768_4k", "lla2d_b256_8k"])
def test_shapes_layouts_and_dtypes(name):
    w = _small(name)
    x = make_decode_inputs(w, 11, with_encode=True)
    T, H, d, rk, rv, B, L = w.T, w.H, w.d, w.r_k, w.r_v, w.B, w.L_max
    if w.variant == 0:
        want = {"cache_k": (B, H, L, rk), "cache_v": (B, H, L, rv), "w_up_k": (T, H, d, rk),
                "w_up_v": (T, H, d, rv), "mu_k": (H, T * d), "w_down_k": (H, T * d, rk),
                "x_k": (5, H, T * d)}
    else:
        want = {"cache_k": (B, L, rk), "cache_v": (B, L, rv), "w_up_k": (T, H * d, rk),
                "w_up_v": (T, H * d, rv), "mu_k": (T * H * d,), "w_down_k": (T * H * d, rk),
                "x_k": (5, T * H * d)}
    want["q"] = (B, H, d)
    for k, s in want.items():
        assert tuple(x[k].shape) == s, k
    for k in ("cache_k", "cache_v", "w_up_k", "w_up_v", "w_down_k", "w_down_v", "x_k", "x_v", "q"):
        assert x[k].dtype == torch.bfloat16, k
    assert x["mu_k"].dtype == torch.float32 and x["mu_v"].dtype == torch.float32
    assert x["seq_lens"].dtype == torch.int32 and x["q_pos"].dtype == torch.int32


def test_distributions_follow_the_recipe():
    """Variances as stated: latents, x and q 1; W_up 1/r; mu 0.1; W_down 1/(T d)
    (LLA-2D: 1/(T H d)); means 0.  Large draws, loose bounds (a few standard errors)."""
    w = _small("ouro1.4b_rho4_b32_4k", B=4, L_max=512)
    x = make_decode_inputs(w, 5, with_encode=True)
    T, d = w.T, w.d
    want = {"cache_k": 1.0, "cache_v": 1.0, "w_up_k": 1.0 / w.r_k, "w_up_v": 1.0 / w.r_v,
            "mu_k": 0.1, "mu_v": 0.1, "w_down_k": 1.0 / (T * d), "w_down_v": 1.0 / (T * d),
            "x_k": 1.0, "x_v": 1.0, "q": 1.0}
    for k, var in want.items():
        v = widen(x[k]).ravel()
        n = v.size
        assert abs(v.mean()) < 5 * math.sqrt(var / n), k
        assert abs(v.var() / var - 1) < 5 * math.sqrt(2.0 / n) + 0.01, (k, v.var(), var)
    w2 = _small("lla2d_b256_8k", B=2, L_max=128)
    x2 = make_decode_inputs(w2, 5, with_encode=True)
    v = widen(x2["w_down_k"]).ravel()
    assert abs(v.var() * (w2.T * w2.H * w2.d) - 1) < 0.05


def test_lengths_and_query_positions():
    w = _small("ouro1.4b_rho4_b32_4k", B=64, L_max=300, lo=7, hi=300)
    x = make_decode_inputs(w, 3)
    L = x["seq_lens"].numpy()
    assert L.min() >= 7 and L.max() <= 300 and len(set(L.tolist())) > 20
    np.testing.assert_array_equal(x["q_pos"].numpy(), L - 1)
    fixed = torch.tensor([0, 5, 300], dtype=torch.int32)
    y = make_decode_inputs(dataclasses.replace(w, B=3), 3, seq_lens=fixed)
    np.testing.assert_array_equal(y["seq_lens"].numpy(), [0, 5, 300])
    np.testing.assert_array_equal(y["q_pos"].numpy(), [0, 4, 299])      # an empty row clamps to 0


def test_a_seed_fixes_every_value():
    w = _small("ouro1.4b_rho4_b32_4k")
    a, b, c = (make_decode_inputs(w, s, with_encode=True) for s in (9, 9, 10))
    for k in a:
        assert torch.equal(a[k], b[k]), k
    assert not torch.equal(a["cache_k"], c["cache_k"]) and not torch.equal(a["q"], c["q"])
    da, db = make_decoupled_inputs(w, 4), make_decoupled_inputs(w, 4)
    assert torch.equal(da["k_rope"], db["k_rope"]) and da["q"].shape == (w.B, w.H, w.d + 64)


def test_storage_rounding_is_one_rounding_of_the_fp32_draw():
    """bf16 values are the fp32 draw rounded once: the same generator calls drawn in fp32
    and rounded by the library give the same tensor; fp32 workloads keep the draw."""
    w = _small("ouro1.4b_rho4_b32_4k")
    bf = make_decode_inputs(w, 21)
    f32 = make_decode_inputs(dataclasses.replace(w, dtype="f32"), 21)
    for k in ("cache_k", "cache_v", "w_up_k", "w_up_v", "q"):
        assert f32[k].dtype == torch.float32
        assert torch.equal(f32[k].to(torch.bfloat16), bf[k]), k
    assert torch.equal(f32["mu_k"], bf["mu_k"])


def test_window_inputs_follow_the_latent_tokens():
    w = _small("ouro1.4b_rho4_b32_4k", B=3)
    lens = torch.tensor([10, 0, 40], dtype=torch.int32)
    win_len = torch.tensor([128, 0, 5], dtype=torch.int32)
    x = make_window_inputs(w, 128, 2, lens, win_len=win_len)
    assert tuple(x["k_win"].shape) == (3, w.H, 128, w.d)
    np.testing.assert_array_equal(x["win_pos"].numpy(), [10, 0, 40])
    # the query is the newest window token; with an empty window the newest latent one
    np.testing.assert_array_equal(x["q_pos"].numpy(), [137, 0, 44])


def test_tiny_parity_case_is_fp32():
    w = WORKLOADS["tiny_f32"]
    assert isinstance(w, Workload) and w.dtype == "f32" and w.len_lo == w.len_hi == 256
    x = make_decode_inputs(w, 1)
    assert x["cache_k"].dtype == torch.float32 and int(x["seq_lens"][0]) == 256
