"""Parity of the small-rank per-head decode kernel (r_k in {16, 32}, r_v in {32, 64},
even H <= 16) with the oracle, through the C ABI.

The kernel splits positions (sequence, 128-token tile) over CTAs with every head of
a position in one CTA, applies RoPE through an f16 MMA against the tile's RoPE rows,
and leaves per-(sequence, CTA, head, warp) records for the combine kernel; these
cases cover every instantiation, runs that start and end inside a CTA range, runs
cut between CTAs, empty and one-token sequences, both RoPE pairings, padding that
must never be read, reference rescaling and the f16 range flag.
"""
import numpy as np
import pytest
import torch

from lla_cases import compare, gpu_decode, lla_dims, make_decode_inputs, workload
from looped_transformer_cross_gb300 import lla

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from looped_transformer_cross_gb300 import build
    build.build()


def _inputs(w, seed, lens):
    return make_decode_inputs(w, seed, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32))


def _small(w):
    assert lla.decode_kernel(lla_dims(w)) == "small-rank"


@pytest.mark.parametrize("rk,rv,H", [(16, 32, 2), (16, 32, 16), (16, 64, 4), (32, 32, 8), (32, 64, 6),
                                     (32, 64, 2), (16, 32, 6)])
def test_instances_ragged(rk, rv, H):
    w = workload(T=2, H=H, r_k=rk, r_v=rv, B=4, L_max=520)
    _small(w)
    inp = _inputs(w, 3000 + rk + rv + H, [520, 1, 129, 384])
    for t in range(w.T):
        compare(w, inp, t)


@pytest.mark.parametrize("style", [0, 1])
def test_rope_styles(style):
    w = workload(T=4, H=4, r_k=16, r_v=32, B=2, L_max=700)
    _small(w)
    inp = _inputs(w, 310 + style, [700, 257])
    compare(w, inp, 3, rope_style=style)


def test_runs_within_and_across_ctas():
    """320 positions over at most 152 CTAs: ranges of 2-3 positions that start and end
    mid-sequence, sequences that end inside a range, and empty sequences between."""
    lens = [900, 0, 130, 1, 1024, 777, 0, 256, 255, 640] * 5
    w = workload(T=4, H=16, r_k=16, r_v=32, B=len(lens), L_max=1024)
    _small(w)
    inp = _inputs(w, 321, lens)
    out, lse, st = gpu_decode(w, inp, 2)
    assert st == lla.LLA_OK
    empty = [i for i, L in enumerate(lens) if L == 0]
    assert torch.all(out[empty] == 0) and torch.all(torch.isneginf(lse[empty]))
    compare(w, inp, 2, bsel=[0, 2, 3, 4, 9, 13, 24, 38, 45, 49])


def test_one_position_per_cta():
    """Fewer positions than SMs: every CTA holds one position, every run is one tile."""
    w = workload(T=2, H=16, r_k=16, r_v=32, B=5, L_max=1000)
    _small(w)
    inp = _inputs(w, 322, [1000, 999, 129, 128, 512])
    compare(w, inp, 1)


def test_padding_is_never_read():
    """NaN in every slot at or beyond seq_lens must not change a single output bit."""
    w = workload(T=2, H=4, r_k=16, r_v=32, B=3, L_max=384)
    _small(w)
    lens = [300, 129, 1]
    inp = _inputs(w, 323, lens)
    ref_out, ref_lse, _ = gpu_decode(w, inp, 1)
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
    for b, L in enumerate(lens):
        inp["cache_k"][b, :, L:] = float("nan")
        inp["cache_v"][b, :, L:] = float("nan")
    out, lse, st = gpu_decode(w, inp, 1)
    assert st == lla.LLA_OK
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_softmax_weights_normalised():
    """Constant V latents with a one-hot W_up,v and mu_v = 0 give out[e] = 1 for e < r_v."""
    w = workload(T=2, H=4, r_k=16, r_v=64, B=2, L_max=700)
    _small(w)
    inp = _inputs(w, 324, [700, 333])
    inp["cache_v"].fill_(1.0)
    wv = torch.zeros_like(inp["w_up_v"])
    for e in range(64):
        wv[:, :, e, e] = 1.0
    inp["w_up_v"] = wv
    inp["mu_v"].zero_()
    out, _, st = gpu_decode(w, inp, 0)
    assert st == lla.LLA_OK
    o = out.cpu().numpy()
    np.testing.assert_allclose(o[..., :64], 1.0, rtol=0, atol=2e-6)
    np.testing.assert_allclose(o[..., 64:], 0.0, rtol=0, atol=0)


def test_growing_scores_rescale_accumulators():
    """K latents ramped x1 .. x6 along each sequence: warp references are raised many
    times inside a run, and the mirror image (largest scores first) never rescales."""
    w = workload(T=2, H=4, r_k=16, r_v=32, B=3, L_max=1500)
    _small(w)
    inp = _inputs(w, 325, [1500, 1200, 700])
    ramp = torch.linspace(1.0, 6.0, w.L_max, device="cuda").view(1, 1, w.L_max, 1)
    inp["cache_k"] = (inp["cache_k"].float() * ramp).to(inp["cache_k"].dtype).contiguous()
    for t in range(w.T):
        compare(w, inp, t)
    inp["cache_k"] = inp["cache_k"].flip(2).contiguous()
    compare(w, inp, 0)


def test_repeated_calls_are_deterministic():
    w = workload(T=4, H=16, r_k=16, r_v=32, B=12, L_max=900)
    _small(w)
    inp = _inputs(w, 326, [900, 800, 700, 600, 500, 400] * 2)
    a, la, _ = gpu_decode(w, inp, 1)
    a, la = a.clone(), la.clone()
    for _ in range(3):
        b, lb, st = gpu_decode(w, inp, 1)
        assert st == lla.LLA_OK and torch.equal(a, b) and torch.equal(la, lb)


def test_out_of_range_lengths_flagged():
    w = workload(T=2, H=2, r_k=16, r_v=32, B=2, L_max=128)
    _small(w)
    inp = _inputs(w, 327, [128, 5])
    inp["seq_lens"][0] = 500          # beyond L_max: clamped, status recorded
    out, _, st = gpu_decode(w, inp, 0)
    assert st == lla.LLA_ERR_DEVICE_ARG
    inp["seq_lens"][0] = 128
    ref, _, st2 = gpu_decode(w, inp, 0)
    assert st2 == lla.LLA_OK and torch.equal(out, ref)


def test_f16_range_flagged():
    """A query large enough that its folded operand leaves the f16 range is flagged."""
    w = workload(T=2, H=2, r_k=16, r_v=32, B=2, L_max=256)
    _small(w)
    inp = _inputs(w, 328, [256, 100])
    inp["q"][1] = 3.0e6
    _, _, st = gpu_decode(w, inp, 0)
    assert st == lla.LLA_ERR_RANGE
