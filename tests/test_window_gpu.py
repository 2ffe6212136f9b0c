"""Parity of the exact-window path (lla_decode_attn over the latent tokens, then
lla_window_attn over the window) with the oracle's hybrid attention, Eq. (4) of
"Hybrid Latent Attention for Looped Language Models" §3.4, through the C ABI.

The window of W = 128 tokens is the HLA page's main setting; smaller and ragged
windows, empty latent parts, empty windows, both RoPE pairings, the fp32 mode,
both per-head decode kernels (tile and small-rank) and the LLA-2D decode are
covered, with the tolerance of ``lla_cases``.
"""
import numpy as np
import pytest
import torch

import oracle
from lla_cases import TOL, lla_dims, lse_err, oracle_dims, rel_err, widen, workload
from looped_transformer_cross_gb300 import lla
from looped_transformer_cross_gb300.synth import make_decode_inputs, make_window_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from looped_transformer_cross_gb300 import build
    build.build()


def _inputs(w, W, seed, lens, win_len=None):
    inp = make_decode_inputs(w, seed, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32))
    wl = None if win_len is None else torch.tensor(win_len, dtype=torch.int32)
    win = make_window_inputs(w, W, seed + 1, inp["seq_lens"], device="cuda", win_len=wl)
    inp["q_pos"] = win["q_pos"]
    return inp, win


def _gpu(w, inp, win, t, style=0):
    dm = lla_dims(w, style)
    n = int(max(w.L_max + win["k_win"].shape[2], 128))
    cos, sin = lla.rope_table(dm, n)
    cos, sin = cos.cuda(), sin.cuda()
    B, H = inp["q"].shape[0], inp["q"].shape[1]
    ws = lla.make_workspace(dm, B, w.L_max)
    out = torch.empty((B, H, w.d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    lla.decode_attn(dm, t, inp["q"], inp["cache_k"], inp["cache_v"], inp["seq_lens"], inp["q_pos"],
                    inp["w_up_k"], inp["w_up_v"], inp["mu_k"], inp["mu_v"], cos, sin, out, lse, ws)
    lla.window_attn(dm, inp["q"], win["k_win"], win["v_win"], win["win_len"], win["win_pos"], inp["q_pos"],
                    cos, sin, out, lse, ws)
    return out, lse, lla.device_status(ws)


def _oracle(w, inp, win, t, style=0, bsel=None):
    sel = (lambda x: x) if bsel is None else (lambda x: x[list(bsel)])
    return oracle.hybrid(oracle_dims(w, style), t, widen(sel(inp["q"])), widen(sel(inp["cache_k"])),
                         widen(sel(inp["cache_v"])), sel(inp["seq_lens"]).cpu().numpy(),
                         sel(inp["q_pos"]).cpu().numpy(), widen(inp["w_up_k"]), widen(inp["w_up_v"]),
                         widen(inp["mu_k"]), widen(inp["mu_v"]), widen(sel(win["k_win"])),
                         widen(sel(win["v_win"])), sel(win["win_len"]).cpu().numpy(),
                         sel(win["win_pos"]).cpu().numpy())


def _compare(w, inp, win, t, style=0, bsel=None):
    out, lse, st = _gpu(w, inp, win, t, style)
    assert st == lla.LLA_OK, lla.status_string(st)
    ro, rl = _oracle(w, inp, win, t, style, bsel)
    go, gl = out.cpu().double().numpy(), lse.cpu().double().numpy()
    if bsel is not None:
        go, gl = go[list(bsel)], gl[list(bsel)]
    assert np.all(np.isfinite(go))
    e_o, e_l = rel_err(go, ro), lse_err(gl, rl)
    assert e_o <= TOL[w.dtype] and e_l <= TOL[w.dtype], (e_o, e_l)
    return e_o, e_l


@pytest.mark.parametrize("rk,rv,H", [(16, 32, 16), (96, 160, 4), (32, 64, 2)])
def test_window_128_after_ragged_latents(rk, rv, H):
    w = workload(T=2, H=H, r_k=rk, r_v=rv, B=4, L_max=400)
    inp, win = _inputs(w, 128, 40 + rk, [400, 1, 129, 0])
    for t in range(w.T):
        _compare(w, inp, win, t)


@pytest.mark.parametrize("style", [0, 1])
def test_ragged_windows_and_rope_styles(style):
    w = workload(T=2, H=4, r_k=16, r_v=32, B=5, L_max=300)
    inp, win = _inputs(w, 40, 50 + style, [300, 77, 0, 128, 5], win_len=[40, 1, 17, 0, 33])
    _compare(w, inp, win, 1, style)


def test_fp32_mode():
    w = workload(T=2, H=2, r_k=48, r_v=80, B=3, L_max=260, dtype="f32")
    inp, win = _inputs(w, 24, 60, [260, 7, 0], win_len=[24, 3, 10])
    _compare(w, inp, win, 0)


def test_lla2d_latents_with_exact_window():
    w = workload(T=2, H=4, r_k=64, r_v=128, B=2, L_max=300, variant=1)
    inp, win = _inputs(w, 32, 70, [300, 150])
    dm = lla_dims(w)
    out, lse, st = _gpu(w, inp, win, 1)
    assert st == lla.LLA_OK
    # oracle: the 2D latent part by decode and the window by sdpa, one softmax via
    # the (pinned) log-sum-exp merge; the 2D hybrid is not a separate oracle function
    od = oracle_dims(w)
    ol, ll, _ = oracle.decode(od, 1, widen(inp["q"]), widen(inp["cache_k"]), widen(inp["cache_v"]),
                              inp["seq_lens"].cpu().numpy(), inp["q_pos"].cpu().numpy(), widen(inp["w_up_k"]),
                              widen(inp["w_up_v"]), widen(inp["mu_k"]), widen(inp["mu_v"]))
    for b in range(w.B):
        p0 = int(win["win_pos"][b])
        ow, lw = oracle.sdpa(od, widen(inp["q"][b:b + 1]), widen(win["k_win"][b:b + 1]),
                             widen(win["v_win"][b:b + 1]), win["win_len"][b:b + 1].cpu().numpy(),
                             (inp["q_pos"][b:b + 1] - p0).cpu().numpy(), pos_offset=p0)
        M = np.maximum(ll[b], lw[0])
        wa, wb = np.exp(ll[b] - M), np.exp(lw[0] - M)
        ref = (wa[:, None] * ol[b] + wb[:, None] * ow[0]) / (wa + wb)[:, None]
        refl = M + np.log(wa + wb)
        assert rel_err(out[b].cpu().double().numpy(), ref) <= 2e-2
        assert lse_err(lse[b].cpu().double().numpy(), refl) <= 2e-2


def test_empty_window_leaves_latent_result():
    w = workload(T=2, H=2, r_k=16, r_v=32, B=3, L_max=200)
    inp, win = _inputs(w, 16, 80, [200, 60, 0], win_len=[0, 0, 0])
    dm = lla_dims(w)
    cos, sin = lla.rope_table(dm, 256)
    cos, sin = cos.cuda(), sin.cuda()
    ws = lla.make_workspace(dm, 3, w.L_max)
    out = torch.empty((3, 2, 128), device="cuda")
    lse = torch.empty((3, 2), device="cuda")
    lla.decode_attn(dm, 0, inp["q"], inp["cache_k"], inp["cache_v"], inp["seq_lens"], inp["q_pos"],
                    inp["w_up_k"], inp["w_up_v"], inp["mu_k"], inp["mu_v"], cos, sin, out, lse, ws)
    o0, l0 = out.clone(), lse.clone()
    lla.window_attn(dm, inp["q"], win["k_win"], win["v_win"], win["win_len"], win["win_pos"], inp["q_pos"],
                    cos, sin, out, lse, ws)
    assert lla.device_status(ws) == lla.LLA_OK
    assert torch.equal(out, o0) and torch.equal(lse, l0)


def test_bad_window_length_is_flagged_and_skipped():
    w = workload(T=2, H=2, r_k=16, r_v=32, B=2, L_max=128)
    inp, win = _inputs(w, 8, 90, [128, 40], win_len=[8, 8])
    win["win_len"][1] = 9                 # beyond W
    out, lse, st = _gpu(w, inp, win, 0)
    assert st == lla.LLA_ERR_DEVICE_ARG
    win["win_len"][1] = 0                 # what the kernel fell back to
    ref, refl, st2 = _gpu(w, inp, win, 0)
    assert st2 == lla.LLA_OK and torch.equal(out, ref) and torch.equal(lse, refl)


def test_serving_batch_window_sampled():
    """768 sequences x 4096 latent tokens (rho = 21.3) plus a 128-token exact window:
    three sequences against the oracle."""
    from looped_transformer_cross_gb300.synth import WORKLOADS
    w = WORKLOADS["ouro1.4b_rho21_b768_4k"]
    inp = make_decode_inputs(w, 7, device="cuda")
    win = make_window_inputs(w, 128, 8, inp["seq_lens"], device="cuda")
    inp["q_pos"] = win["q_pos"]
    _compare(w, inp, win, 2, bsel=[0, 383, 767])
