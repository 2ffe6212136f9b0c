"""Parity of the absorbed decoupled-RoPE decode (lla_decode_attn_decoupled; LLA paper,
Appendix J "Absorbed attention") with the oracle's ``decoupled``, through the C ABI:
bf16 storage (2e-2) and the fp32 mode (1e-5), ragged lengths spanning several tiles,
both RoPE pairings of the rotary branch, empty and one-token sequences, padding that
must never be read, many CTA splits, the small-rank tensor-core kernel on every rank
pair it takes, and the Ouro-1.4B rho = 4 and rho = 21.3 layers on sampled sequences.
"""
import numpy as np
import pytest
import torch

import oracle
from lla_cases import TOL, lla_dims, lse_err, oracle_dims, rel_err, widen, workload
from looped_transformer_cross_gb300 import lla
from looped_transformer_cross_gb300.synth import make_decode_inputs, make_decoupled_inputs

pytestmark = pytest.mark.gpu
D_ROPE = 64


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from looped_transformer_cross_gb300 import build
    build.build()


def _inputs(w, seed, lens):
    inp = make_decode_inputs(w, seed, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32))
    inp.update(make_decoupled_inputs(w, seed + 1, device="cuda"))
    return inp


def _gpu(w, inp, t, style=0):
    dm = lla_dims(w, style)
    rdm = lla.dims(w.T, w.H, w.r_k, w.r_v, d_head=D_ROPE, rope_base=w.rope_base)
    cos, sin = lla.rope_table(rdm, max(w.L_max, 128))
    cos, sin = cos.cuda(), sin.cuda()
    B, H = inp["q"].shape[0], inp["q"].shape[1]
    ws = lla.decoupled_workspace(dm, D_ROPE, B, w.L_max)
    out = torch.empty((B, H, w.d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    lla.decode_attn_decoupled(dm, t, inp["q"], inp["cache_k"], inp["cache_v"], inp["k_rope"], inp["seq_lens"],
                              inp["q_pos"], inp["w_up_k"], inp["w_up_v"], inp["mu_k"], inp["mu_v"], cos, sin,
                              out, lse, ws)
    return out, lse, lla.device_status(ws)


def _compare(w, inp, t, style=0, bsel=None):
    out, lse, st = _gpu(w, inp, t, style)
    assert st == lla.LLA_OK, lla.status_string(st)
    sel = (lambda x: x) if bsel is None else (lambda x: x[list(bsel)])
    ro, rl = oracle.decoupled(oracle_dims(w, style), t, widen(sel(inp["q"])), widen(sel(inp["cache_k"])),
                              widen(sel(inp["cache_v"])), widen(sel(inp["k_rope"])),
                              sel(inp["seq_lens"]).cpu().numpy(), sel(inp["q_pos"]).cpu().numpy(),
                              widen(inp["w_up_k"]), widen(inp["w_up_v"]), widen(inp["mu_k"]), widen(inp["mu_v"]))
    go, gl = out.cpu().double().numpy(), lse.cpu().double().numpy()
    if bsel is not None:
        go, gl = go[list(bsel)], gl[list(bsel)]
    assert np.all(np.isfinite(go))
    e_o, e_l = rel_err(go, ro), lse_err(gl, rl)
    assert e_o <= TOL[w.dtype] and e_l <= TOL[w.dtype], (e_o, e_l)


@pytest.mark.parametrize("rk,rv", [(96, 160), (16, 32), (128, 256), (48, 80)])
def test_ranks_ragged(rk, rv):
    w = workload(T=2, H=2, r_k=rk, r_v=rv, B=4, L_max=400)
    inp = _inputs(w, 500 + rk, [400, 1, 129, 0])
    for t in range(w.T):
        _compare(w, inp, t)


@pytest.mark.parametrize("style", [0, 1])
def test_rope_styles(style):
    w = workload(T=2, H=4, r_k=96, r_v=160, B=2, L_max=520)
    inp = _inputs(w, 510 + style, [520, 300])
    _compare(w, inp, 1, style)


def test_fp32_mode():
    w = workload(T=2, H=2, r_k=48, r_v=80, B=3, L_max=260, dtype="f32")
    inp = _inputs(w, 520, [260, 7, 128])
    for style in (0, 1):
        _compare(w, inp, 0, style)


def test_many_splits_across_ctas():
    w = workload(T=4, H=16, r_k=96, r_v=160, B=8, L_max=1100)
    inp = _inputs(w, 530, [1100, 1000, 257, 128, 129, 640, 1, 999])
    _compare(w, inp, 2)


def test_padding_is_never_read():
    w = workload(T=2, H=2, r_k=96, r_v=160, B=3, L_max=384)
    lens = [300, 129, 1]
    inp = _inputs(w, 540, lens)
    ref, refl, _ = _gpu(w, inp, 1)
    ref, refl = ref.clone(), refl.clone()
    for b, L in enumerate(lens):
        inp["cache_k"][b, :, L:] = float("nan")
        inp["cache_v"][b, :, L:] = float("nan")
        inp["k_rope"][b, :, L:] = float("nan")
    out, lse, st = _gpu(w, inp, 1)
    assert st == lla.LLA_OK and torch.equal(out, ref) and torch.equal(lse, refl)


@pytest.mark.parametrize("style", [0, 1])
@pytest.mark.parametrize("rk,rv", [(16, 32), (16, 64), (32, 32), (32, 64)])
def test_small_ranks_tensor_core_kernel(rk, rv, style):
    """Small ranks take the tensor-core rotary kernel: every rank pair, both RoPE
    pairings (their K-step grouping differs), H = 6 (three heads per epilogue group),
    lengths ragged across tiles, an empty and a one-token sequence, every loop."""
    w = workload(T=2, H=6, r_k=rk, r_v=rv, B=5, L_max=520)
    assert lla.decoupled_kernel(lla_dims(w, style)) == "small-rank"
    inp = _inputs(w, 560 + rk + rv + style, [520, 1, 0, 129, 256])
    for t in range(w.T):
        _compare(w, inp, t, style)


def test_small_ranks_many_splits_across_ctas():
    """H = 16 and 40 sequences of 0..1100 tokens: positions split over many CTAs,
    sequences cut between CTAs (several records per unit), runs that start and end
    inside a sequence."""
    w = workload(T=3, H=16, r_k=16, r_v=32, B=40, L_max=1100)
    rng = np.random.default_rng(570)
    lens = rng.integers(0, 1101, size=w.B)
    lens[:6] = [1100, 0, 1, 128, 129, 1099]
    inp = _inputs(w, 571, lens.tolist())
    _compare(w, inp, 2, bsel=[0, 2, 3, 4, 5, 17, 39])
    _compare(w, inp, 0, bsel=[1, 20, 38])


def test_small_ranks_padding_is_never_read():
    """NaN in every slot past a sequence's length (K, V and rotary keys) leaves the
    small-rank kernel's results bit for bit unchanged."""
    w = workload(T=2, H=4, r_k=16, r_v=32, B=3, L_max=384)
    lens = [300, 129, 1]
    inp = _inputs(w, 575, lens)
    ref, refl, _ = _gpu(w, inp, 1)
    ref, refl = ref.clone(), refl.clone()
    for b, L in enumerate(lens):
        inp["cache_k"][b, :, L:] = float("nan")
        inp["cache_v"][b, :, L:] = float("nan")
        inp["k_rope"][b, :, L:] = float("nan")
    out, lse, st = _gpu(w, inp, 1)
    assert st == lla.LLA_OK and torch.equal(out, ref) and torch.equal(lse, refl)


def test_small_ranks_repeatable():
    """Two calls on the same inputs give the same bits (static split, no atomics)."""
    w = workload(T=2, H=16, r_k=16, r_v=32, B=12, L_max=700)
    inp = _inputs(w, 580, [700, 650, 1, 0, 300, 128, 129, 699, 512, 77, 640, 256])
    a, al, _ = _gpu(w, inp, 1)
    a, al = a.clone(), al.clone()
    b, bl, st = _gpu(w, inp, 1)
    assert st == lla.LLA_OK and torch.equal(a, b) and torch.equal(al, bl)


def test_ouro_rho21_layer_sampled():
    """The rho = 21.3 serving layer (768 x 4096, H = 16, (16, 32)) in the bench's
    launch, three sequences against the oracle."""
    from looped_transformer_cross_gb300.synth import WORKLOADS
    w = WORKLOADS["ouro1.4b_rho21_b768_4k"]
    assert lla.decoupled_kernel(lla_dims(w)) == "small-rank"
    inp = make_decode_inputs(w, 20260011, device="cuda")
    inp.update(make_decoupled_inputs(w, 20260012, device="cuda"))
    _compare(w, inp, 1, bsel=[0, 383, 767])


def test_ouro_rho4_layer_sampled():
    from looped_transformer_cross_gb300.synth import WORKLOADS
    w = WORKLOADS["ouro1.4b_rho4_b32_4k"]
    inp = make_decode_inputs(w, 20260001, device="cuda")
    inp.update(make_decoupled_inputs(w, 20260002, device="cuda"))
    _compare(w, inp, 3, bsel=[0, 17, 31])
