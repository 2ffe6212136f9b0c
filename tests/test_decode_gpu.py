"""Parity of lla_decode_attn (CUDA, through the C ABI) with the oracle.

Every case draws its inputs with the shared seeded generator, runs the kernel and
the fp64 oracle on exactly the same stored tensors, and applies the tolerance of
``lla_cases`` (2e-2 for bf16 storage, 1e-5 for fp32).  Small cases span several
128-token tiles and a ragged tail; full-size cases compare sampled sequences.
"""
import numpy as np
import pytest
import torch

from lla_cases import (compare, gpu_decode, make_decode_inputs, oracle_decode, rel_err, lse_err,
                       workload)
from looped_transformer_cross_gb300 import lla
from looped_transformer_cross_gb300.synth import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from looped_transformer_cross_gb300 import build
    build.build()


def _inputs(w, seed, lens=None):
    sl = None if lens is None else torch.tensor(lens, dtype=torch.int32)
    return make_decode_inputs(w, seed, device="cuda", seq_lens=sl)


def test_tiny_f32_all_loops():
    """The fp32 parity workload: 1 sequence, 256 tokens, H=2, (96,160), t = 1..4."""
    w = WORKLOADS["tiny_f32"]
    inp = _inputs(w, 20260000)
    for t in range(w.T):
        compare(w, inp, t)


@pytest.mark.parametrize("rk,rv", [(96, 160), (16, 32), (32, 64), (48, 80), (112, 240), (64, 128),
                                   (128, 256), (256, 256), (160, 96)])
def test_bf16_ranks_ragged(rk, rv):
    w = workload(r_k=rk, r_v=rv, B=3, L_max=300)
    inp = _inputs(w, 1000 + rk + rv, lens=[300, 1, 129])
    for t in range(w.T):
        compare(w, inp, t)


@pytest.mark.parametrize("style", [0, 1])
def test_bf16_rope_styles(style):
    w = workload(r_k=96, r_v=160, B=2, L_max=520, T=4)
    inp = _inputs(w, 77 + style, lens=[520, 385])
    compare(w, inp, 3, rope_style=style)


def test_f32_ragged_and_interleaved():
    w = workload(r_k=48, r_v=80, B=3, L_max=260, dtype="f32")
    inp = _inputs(w, 5, lens=[260, 7, 128])
    for style in (0, 1):
        compare(w, inp, 1, rope_style=style)


def test_empty_and_single_token_sequences():
    w = workload(r_k=96, r_v=160, B=4, L_max=200)
    inp = _inputs(w, 9, lens=[0, 1, 0, 200])
    out, lse, st = gpu_decode(w, inp, 0)
    assert st == lla.LLA_OK
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert np.all(o[[0, 2]] == 0.0) and np.all(np.isneginf(l[[0, 2]]))
    compare(w, inp, 0)


def test_all_sequences_empty():
    w = workload(B=3, L_max=64)
    inp = _inputs(w, 10, lens=[0, 0, 0])
    out, lse, st = gpu_decode(w, inp, 1)
    assert st == lla.LLA_OK
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_padding_is_never_read():
    """NaN in every slot at or beyond seq_lens must not change a single output bit."""
    w = workload(r_k=96, r_v=160, B=3, L_max=384)
    inp = _inputs(w, 11, lens=[300, 129, 1])
    ref_out, ref_lse, _ = gpu_decode(w, inp, 1)
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
    for b, L in enumerate([300, 129, 1]):
        inp["cache_k"][b, :, L:] = float("nan")
        inp["cache_v"][b, :, L:] = float("nan")
    out, lse, st = gpu_decode(w, inp, 1)
    assert st == lla.LLA_OK
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_softmax_weights_normalised():
    """Constant V latents with a one-hot W_up,v and mu_v = 0 give out[e] = 1 for e < r_v:
    the tile weights and the denominator must come from the same values."""
    w = workload(r_k=32, r_v=128, B=2, L_max=700)
    inp = _inputs(w, 12, lens=[700, 333])
    inp["cache_v"].fill_(1.0)
    wv = torch.zeros_like(inp["w_up_v"])
    for e in range(128):
        wv[:, :, e, e] = 1.0
    inp["w_up_v"] = wv
    inp["mu_v"].zero_()
    out, _, st = gpu_decode(w, inp, 0)
    assert st == lla.LLA_OK
    np.testing.assert_allclose(out.cpu().numpy(), 1.0, rtol=0, atol=2e-6)


def test_growing_scores_rescale_accumulators():
    """K latents scaled up along each sequence (x1 .. x4): later tiles' score maxima
    exceed the running reference by more than the lazy-rescale threshold (2^8), so
    accumulators are rescaled (16 times over these 12 units, at warp level, by the
    oracle's scores) and once more across CTA splits.  The ramp stays moderate:
    the bf16 query operand carries a ~2^-9 relative error per score term, so the
    lse error grows with the score magnitude (|lse| <= 12 here)."""
    w = workload(T=2, H=4, r_k=96, r_v=160, B=3, L_max=1500)
    inp = _inputs(w, 15, lens=[1500, 1200, 700])
    ramp = torch.linspace(1.0, 4.0, w.L_max, device="cuda").view(1, 1, w.L_max, 1)
    inp["cache_k"] = (inp["cache_k"].float() * ramp).to(inp["cache_k"].dtype).contiguous()
    for t in range(w.T):
        compare(w, inp, t)
    # and the mirror image: the largest scores first, no rescale after the first tile
    inp["cache_k"] = inp["cache_k"].flip(2).contiguous()
    compare(w, inp, 0)


def test_out_of_range_lengths_flagged():
    w = workload(B=2, L_max=128)
    inp = _inputs(w, 13, lens=[128, 5])
    inp["seq_lens"][0] = 500          # beyond L_max: clamped, status recorded
    out, lse, st = gpu_decode(w, inp, 0)
    assert st == lla.LLA_ERR_DEVICE_ARG
    inp["seq_lens"][0] = 128
    ref, _, st2 = gpu_decode(w, inp, 0)
    assert st2 == lla.LLA_OK and torch.equal(out, ref)


def test_many_splits_across_ctas():
    """Enough tiles that most (sequence, head) units are cut between CTAs."""
    w = workload(T=4, H=16, r_k=96, r_v=160, B=8, L_max=1100)
    inp = _inputs(w, 14, lens=[1100, 1000, 257, 128, 129, 640, 1, 999])
    compare(w, inp, 2)


def test_repeated_calls_are_deterministic():
    w = workload(T=4, H=16, B=6, L_max=900)
    inp = _inputs(w, 15, lens=[900, 800, 700, 600, 500, 400])
    a, la, _ = gpu_decode(w, inp, 1)
    a, la = a.clone(), la.clone()
    for _ in range(3):
        b, lb, st = gpu_decode(w, inp, 1)
        assert st == lla.LLA_OK and torch.equal(a, b) and torch.equal(la, lb)


def _sampled_full_size(name, bsel, t=0):
    w = WORKLOADS[name]
    inp = make_decode_inputs(w, 20260000 + 1, device="cuda")
    out, lse, st = gpu_decode(w, inp, t)
    assert st == lla.LLA_OK
    go, gl = out.cpu().double().numpy(), lse.cpu().double().numpy()
    assert np.all(np.isfinite(go)) and np.all(np.isfinite(gl))
    ro, rl = oracle_decode(w, inp, t, bsel=bsel)
    e_o, e_l = rel_err(go[list(bsel)], ro), lse_err(gl[list(bsel)], rl)
    assert e_o <= 2e-2 and e_l <= 2e-2, (e_o, e_l)
    return e_o, e_l


def test_ouro_rho4_b32_4k_sampled():
    """The benchmarked workload (Ouro-1.4B shape, rho = 4, 32 ragged sequences of
    3584..4096 tokens), same launch as the bench; four sequences checked in full."""
    _sampled_full_size("ouro1.4b_rho4_b32_4k", [0, 9, 22, 31], t=3)


def test_ouro_rho21_b768_4k_sampled():
    """rho = 21.3 at serving batch (768 x 4096, one layer); three sequences checked."""
    _sampled_full_size("ouro1.4b_rho21_b768_4k", [0, 400, 767], t=1)


def test_ouro_rho4_b64_16k_sampled():
    """The long-context layer (64 sequences x 16384 tokens, rho = 4) in the launch the
    bench times: all 1024 (sequence, head) units of 128 tiles in one call.  Every
    sequence spans 2048 tiles, more than twice one CTA's equal share of the 131,072
    tiles, so each checked sequence has units cut between CTAs; positions reach 16383
    and each unit's running maximum and sum cover 128 tiles.  Four sequences (first,
    last and two inside) are checked against the oracle at two loops."""
    w = WORKLOADS["ouro_rho4_b64_16k"]
    inp = make_decode_inputs(w, 20260000 + 3, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles_per_seq = w.H * (w.L_max // 128)
    assert tiles_per_seq > 2 * (w.B * tiles_per_seq) // min(sms, 1024)
    bsel = [0, 21, 42, 63]
    for t in (0, 3):
        out, lse, st = gpu_decode(w, inp, t)
        assert st == lla.LLA_OK
        go, gl = out.cpu().double().numpy(), lse.cpu().double().numpy()
        assert np.all(np.isfinite(go)) and np.all(np.isfinite(gl))
        ro, rl = oracle_decode(w, inp, t, bsel=bsel)
        e_o, e_l = rel_err(go[bsel], ro), lse_err(gl[bsel], rl)
        assert e_o <= 2e-2 and e_l <= 2e-2, (t, e_o, e_l)
