"""Parity of lla_evict_window (token eviction composed with LLA; LLA paper, Appendix D
"Token-eviction composition table" and Appendix J) with the oracle, through the C ABI.

Eviction only moves rows, so the whole cache after the call (kept rows, untouched
sequences, rows past the new lengths) must equal ``oracle.evict`` bit for bit, and the
new lengths exactly.  Cases cover a shift of one row (every chunk a single row, source
and destination overlapping almost entirely), zero sinks, a zero window, LLA-2D, fp32,
and decode after eviction against the oracle on the oracle's evicted cache.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import evict
from lla_cases import TOL, lla_dims, lse_err, oracle_dims, rel_err, widen, workload
from looped_transformer_cross_gb300 import lla
from looped_transformer_cross_gb300.synth import make_decode_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from looped_transformer_cross_gb300 import build
    build.build()


def _evict_gpu(w, inp, sink, window):
    dm = lla_dims(w)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    lens = inp["seq_lens"].clone()
    lla.evict_window(dm, inp["cache_k"], inp["cache_v"], lens, sink, window, ws)
    return lens, lla.device_status(ws)


def _as4(x, w):
    """[B][H][L][r] view of a cache (LLA-2D: one latent row set per sequence)."""
    return x if w.variant == 0 else x[:, None]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("sink,window", [(4, 256), (0, 10), (5, 0)])
def test_evict_layout_exact(dtype, sink, window):
    w = workload(T=2, H=3, r_k=96, r_v=160, B=5, L_max=300, dtype=dtype)
    lens = [300, 50, sink + window + 1, 0, 299]
    inp = make_decode_inputs(w, 800 + sink + window, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32))
    ref_k, ref_lens = evict.evict(widen(inp["cache_k"]), lens, sink, window)
    ref_v, _ = evict.evict(widen(inp["cache_v"]), lens, sink, window)
    new_lens, st = _evict_gpu(w, inp, sink, window)
    assert st == lla.LLA_OK
    assert new_lens.cpu().tolist() == list(ref_lens)
    np.testing.assert_array_equal(widen(inp["cache_k"]), ref_k)
    np.testing.assert_array_equal(widen(inp["cache_v"]), ref_v)


def test_evict_layout_exact_lla2d():
    w = workload(T=2, H=4, r_k=128, r_v=256, B=3, L_max=700, variant=1)
    lens = [700, 300, 261]
    inp = make_decode_inputs(w, 810, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32))
    ref_k, ref_lens = evict.evict(_as4(widen(inp["cache_k"]), w), lens, 4, 256)
    ref_v, _ = evict.evict(_as4(widen(inp["cache_v"]), w), lens, 4, 256)
    new_lens, st = _evict_gpu(w, inp, 4, 256)
    assert st == lla.LLA_OK
    assert new_lens.cpu().tolist() == list(ref_lens)
    np.testing.assert_array_equal(_as4(widen(inp["cache_k"]), w), ref_k)
    np.testing.assert_array_equal(_as4(widen(inp["cache_v"]), w), ref_v)


@pytest.mark.parametrize("rk,rv", [(96, 160), (16, 32)])
def test_decode_after_eviction(rk, rv):
    """Evict to sink 4 + window 256, then decode with the query at the newest kept slot."""
    w = workload(T=2, H=4, r_k=rk, r_v=rv, B=4, L_max=1100)
    lens = [1100, 700, 200, 261]
    inp = make_decode_inputs(w, 820 + rk, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32))
    ref_k, ref_lens = evict.evict(widen(inp["cache_k"]), lens, 4, 256)
    ref_v, _ = evict.evict(widen(inp["cache_v"]), lens, 4, 256)
    new_lens, st = _evict_gpu(w, inp, 4, 256)
    assert st == lla.LLA_OK
    inp["seq_lens"] = new_lens
    inp["q_pos"] = (new_lens - 1).clamp(min=0).to(torch.int32)
    dm = lla_dims(w)
    cos, sin = lla.rope_table(dm, max(w.L_max, 128))
    cos, sin = cos.cuda(), sin.cuda()
    ws = lla.make_workspace(dm, w.B, w.L_max)
    out = torch.empty((w.B, w.H, w.d), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    for t in range(w.T):
        lla.decode_attn(dm, t, inp["q"], inp["cache_k"], inp["cache_v"], inp["seq_lens"], inp["q_pos"],
                        inp["w_up_k"], inp["w_up_v"], inp["mu_k"], inp["mu_v"], cos, sin, out, lse, ws)
        assert lla.device_status(ws) == lla.LLA_OK
        ro, rl, _ = oracle.decode(oracle_dims(w), t, widen(inp["q"]), ref_k, ref_v, np.asarray(ref_lens),
                                  np.asarray(ref_lens) - 1, widen(inp["w_up_k"]), widen(inp["w_up_v"]),
                                  widen(inp["mu_k"]), widen(inp["mu_v"]))
        go, gl = out.double().cpu().numpy(), lse.double().cpu().numpy()
        assert rel_err(go, ro) <= TOL["bf16"] and lse_err(gl, rl) <= TOL["bf16"]


def test_evict_bad_length_flagged_and_untouched():
    w = workload(T=2, H=2, r_k=96, r_v=160, B=2, L_max=300)
    inp = make_decode_inputs(w, 830, device="cuda", seq_lens=torch.tensor([300, 280], dtype=torch.int32))
    inp["seq_lens"][1] = 301                      # beyond L_max
    before_k = inp["cache_k"].clone()
    new_lens, st = _evict_gpu(w, inp, 4, 256)
    assert st == lla.LLA_ERR_DEVICE_ARG
    assert new_lens.cpu().tolist() == [260, 301]
    assert torch.equal(inp["cache_k"][1], before_k[1])
