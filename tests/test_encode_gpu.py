"""Parity of lla_encode (CUDA, through the C ABI) with the oracle.

Layout and indexing are checked bit-exactly with structured inputs whose
arithmetic is exact in bf16/fp32; random inputs are compared with the oracle's
fp64 latents rounded to bf16 (at most one bf16 ulp apart: the kernel rounds an
fp32 sum, the oracle an fp64 one).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from lla_cases import gpu_decode, lla_dims, oracle_dims, workload
from looped_transformer_cross_gb300 import lla
from looped_transformer_cross_gb300.synth import make_decode_inputs, widen

pytestmark = pytest.mark.gpu

CANARY = -3072.0  # exactly representable in bf16 and fp32


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from looped_transformer_cross_gb300 import build
    build.build()


def _encode(w, x_k, x_v, seq_idx, pos, wdk, wdv, mu_k, mu_v, ck, cv):
    dm = lla_dims(w)
    ws = lla.make_workspace(dm, ck.shape[0], w.L_max, seq_idx.shape[0])
    lla.encode(dm, x_k, x_v, seq_idx, pos, wdk, wdv, mu_k, mu_v, ck, cv, ws)
    return lla.device_status(ws)


@pytest.mark.parametrize("dtype,rk,rv,N", [
    ("bf16", 96, 160, 130), ("bf16", 16, 32, 130), ("bf16", 48, 80, 130), ("bf16", 256, 240, 130),
    ("f32", 96, 160, 130), ("f32", 16, 32, 130), ("f32", 48, 80, 130), ("f32", 256, 240, 130),
    # a batch of 33 tiles with a 4-token tail, spread over the persistent grid
    ("bf16", 96, 160, 4100), ("bf16", 128, 256, 4100), ("bf16", 32, 64, 4100)])
def test_encode_layout_structured_exact(dtype, rk, rv, N):
    """Selector W_down and small-integer x: every latent is one x entry exactly, it lands in
    slot (seq_idx[n], h, pos[n]) and every other slot keeps its canary."""
    T, H, d, B = 2, 3, 128, 3
    L_max = 200 if N <= 200 else 1400   # N spans two token tiles, or 33
    w = workload(T=T, H=H, r_k=rk, r_v=rv, B=B, L_max=L_max, dtype=dtype)
    sd = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = np.random.default_rng(3)
    slots = g.choice(B * L_max, size=N, replace=False)
    seq_idx = torch.tensor(slots // L_max, dtype=torch.int32)
    pos = torch.tensor(slots % L_max, dtype=torch.int32)
    Td = T * d
    expect = {}
    tensors = []
    for axis, r in ((0, rk), (1, rv)):
        u_of_k = (np.arange(r) * 37 + 11 + axis) % Td
        W = np.zeros((H, Td, r), np.float32)
        W[:, u_of_k, np.arange(r)] = 1.0
        x = ((np.arange(N)[:, None, None] * 3 + np.arange(H)[None, :, None] * 5 +
              np.arange(Td)[None, None, :] + axis) % 241 - 120).astype(np.float32)
        expect[axis] = x[:, :, u_of_k]                     # [N][H][r]
        tensors.append((torch.from_numpy(x).to(sd).cuda(), torch.from_numpy(W).to(sd).cuda()))
    mu = torch.zeros((H, Td), dtype=torch.float32, device="cuda")
    ck = torch.full((B, H, L_max, rk), CANARY, dtype=sd, device="cuda")
    cv = torch.full((B, H, L_max, rv), CANARY, dtype=sd, device="cuda")
    st = _encode(w, tensors[0][0], tensors[1][0], seq_idx.cuda(), pos.cuda(), tensors[0][1],
                 tensors[1][1], mu, mu, ck, cv)
    assert st == lla.LLA_OK
    for axis, cache in ((0, ck), (1, cv)):
        got = cache.float().cpu().numpy()
        touched = np.zeros(got.shape[:3], bool)
        for n in range(N):
            b, p = int(seq_idx[n]), int(pos[n])
            np.testing.assert_array_equal(got[b, :, p], expect[axis][n])
            touched[b, :, p] = True
        assert np.all(got[~touched] == CANARY)


@pytest.mark.parametrize("rk,rv,N", [(96, 160, 300), (16, 32, 300), (96, 160, 4100)])
def test_encode_random_vs_oracle_bf16(rk, rv, N):
    """Each GPU latent must be the bf16 rounding of a value within the fp32
    accumulation bound 2^-20 * sum_u |x_u - mu_u| |W_uk| of the exact sum (the
    kernel rounds an fp32 dot product of T*d terms), and almost all must equal the
    oracle's fp64 sum rounded to bf16.  N = 4100: 33 tiles over the persistent grid."""
    T, H, d, B = 4, 4, 128, 4
    L_max = 160 if N <= 640 else 1100
    w = workload(T=T, H=H, r_k=rk, r_v=rv, B=B, L_max=L_max, N_encode=N)
    inp = make_decode_inputs(w, 31, device="cuda", with_encode=True)
    g = np.random.default_rng(4)
    slots = g.choice(B * L_max, size=N, replace=False)
    seq_idx = torch.tensor(slots // L_max, dtype=torch.int32, device="cuda")
    pos = torch.tensor(slots % L_max, dtype=torch.int32, device="cuda")
    ck = torch.full((B, H, L_max, rk), CANARY, dtype=torch.bfloat16, device="cuda")
    cv = torch.full((B, H, L_max, rv), CANARY, dtype=torch.bfloat16, device="cuda")
    st = _encode(w, inp["x_k"], inp["x_v"], seq_idx, pos, inp["w_down_k"], inp["w_down_v"],
                 inp["mu_k"], inp["mu_v"], ck, cv)
    assert st == lla.LLA_OK
    dm = oracle_dims(w)
    si, po = seq_idx.cpu().numpy(), pos.cpu().numpy()
    for cache, x, wd, mu, r in ((ck, "x_k", "w_down_k", "mu_k", rk), (cv, "x_v", "w_down_v", "mu_v", rv)):
        exact = np.full((B, H, L_max, r), CANARY)
        oracle.encode(dm, widen(inp[x]), si, po, widen(inp[wd]), widen(inp[mu]), r, exact)
        rounded = np.full((B, H, L_max, r), CANARY)
        oracle.encode(dm, widen(inp[x]), si, po, widen(inp[wd]), widen(inp[mu]), r, rounded,
                      round_to_bf16=True)
        mag = np.full((B, H, L_max, r), 0.0)     # sum |x - mu| |W| in the same slots
        oracle.encode(dm, np.abs(widen(inp[x]) - widen(inp[mu])[None]), si, po,
                      np.abs(widen(inp[wd])), np.zeros_like(widen(inp[mu])), r, mag)
        got = cache.double().cpu().numpy()
        touched = got != CANARY
        assert np.all(rounded[~touched] == CANARY) and touched.sum() == N * H * r
        # half a bf16 spacing at |got| (2^(e-8) for 2^e <= |got| < 2^(e+1)) plus the bound
        half_ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(got), 2.0 ** -126))) - 8)
        bound = half_ulp + 2.0 ** -20 * mag
        assert np.all(np.abs(got - exact)[touched] <= bound[touched])
        assert (got == rounded)[touched].mean() > 0.99


def test_encode_random_vs_oracle_f32():
    T, H, d, B, L_max, N = 2, 2, 128, 2, 64, 50
    w = workload(T=T, H=H, r_k=48, r_v=80, B=B, L_max=L_max, N_encode=N, dtype="f32")
    inp = make_decode_inputs(w, 32, device="cuda", with_encode=True)
    seq_idx = torch.tensor(np.arange(N) % B, dtype=torch.int32, device="cuda")
    pos = torch.tensor(np.arange(N) // B, dtype=torch.int32, device="cuda")
    ck = torch.zeros((B, H, L_max, 48), dtype=torch.float32, device="cuda")
    cv = torch.zeros((B, H, L_max, 80), dtype=torch.float32, device="cuda")
    assert _encode(w, inp["x_k"], inp["x_v"], seq_idx, pos, inp["w_down_k"], inp["w_down_v"],
                   inp["mu_k"], inp["mu_v"], ck, cv) == lla.LLA_OK
    dm = oracle_dims(w)
    ref = np.zeros((B, H, L_max, 48))
    oracle.encode(dm, widen(inp["x_k"]), seq_idx.cpu().numpy(), pos.cpu().numpy(),
                  widen(inp["w_down_k"]), widen(inp["mu_k"]), 48, ref)
    np.testing.assert_allclose(ck.double().cpu().numpy(), ref, rtol=0, atol=1e-5)


def test_encode_rejects_bad_slots():
    w = workload(T=1, H=1, r_k=16, r_v=16, B=2, L_max=8, N_encode=3)
    inp = make_decode_inputs(w, 33, device="cuda", with_encode=True)
    seq_idx = torch.tensor([0, 5, 1], dtype=torch.int32, device="cuda")   # 5 >= B
    pos = torch.tensor([0, 1, 8], dtype=torch.int32, device="cuda")       # 8 >= L_max
    ck = torch.full((2, 1, 8, 16), CANARY, dtype=torch.bfloat16, device="cuda")
    cv = torch.full((2, 1, 8, 16), CANARY, dtype=torch.bfloat16, device="cuda")
    st = _encode(w, inp["x_k"], inp["x_v"], seq_idx, pos, inp["w_down_k"], inp["w_down_v"],
                 inp["mu_k"], inp["mu_v"], ck, cv)
    assert st == lla.LLA_ERR_DEVICE_ARG
    c = ck.float().cpu().numpy()
    assert np.any(c[0, 0, 0] != CANARY)                # the valid token was written
    c[0, 0, 0] = CANARY
    assert np.all(c == CANARY)                          # nothing else was touched


def test_encode_then_decode_recovers_teacher_attention_f32():
    """Full-rank orthonormal codec (the paper's SVD-initialisation structure, r = T*d):
    encode + decode must reproduce attention over the original per-loop K/V."""
    T, H, d, B, L_max = 2, 2, 128, 2, 150
    r = T * d
    w = workload(T=T, H=H, r_k=r, r_v=r, B=B, L_max=L_max, dtype="f32")
    g = np.random.default_rng(5)
    lens = np.array([150, 77], np.int32)
    Kt = g.standard_normal((B, H, L_max, T, d)).astype(np.float32)
    Vt = g.standard_normal((B, H, L_max, T, d)).astype(np.float32)
    Q = np.stack([np.linalg.qr(g.standard_normal((r, r)))[0] for _ in range(2 * H)]).astype(np.float32)
    Wd_k, Wd_v = torch.from_numpy(Q[:H]), torch.from_numpy(Q[H:])
    # W_up,t = loop-t row slice of W_down -> [T][H][d][r]
    Wu_k = torch.stack([Wd_k[:, t * d:(t + 1) * d, :] for t in range(T)]).contiguous()
    Wu_v = torch.stack([Wd_v[:, t * d:(t + 1) * d, :] for t in range(T)]).contiguous()
    mu = torch.zeros((H, T * d), dtype=torch.float32)
    N = B * L_max
    seq_idx = torch.from_numpy(np.repeat(np.arange(B), L_max).astype(np.int32))
    pos = torch.from_numpy(np.tile(np.arange(L_max), B).astype(np.int32))
    xk = torch.from_numpy(np.ascontiguousarray(Kt.transpose(0, 2, 1, 3, 4).reshape(N, H, T * d)))
    xv = torch.from_numpy(np.ascontiguousarray(Vt.transpose(0, 2, 1, 3, 4).reshape(N, H, T * d)))
    ck = torch.zeros((B, H, L_max, r), dtype=torch.float32, device="cuda")
    cv = torch.zeros_like(ck)
    assert _encode(w, xk.cuda(), xv.cuda(), seq_idx.cuda(), pos.cuda(), Wd_k.cuda(), Wd_v.cuda(),
                   mu.cuda(), mu.cuda(), ck, cv) == lla.LLA_OK
    q = torch.from_numpy(g.standard_normal((B, H, d)).astype(np.float32))
    inp = dict(q=q.cuda(), cache_k=ck, cache_v=cv, seq_lens=torch.from_numpy(lens).cuda(),
               q_pos=torch.from_numpy(lens - 1).cuda(), w_up_k=Wu_k.cuda(), w_up_v=Wu_v.cuda(),
               mu_k=mu.cuda(), mu_v=mu.cuda())
    dm = oracle_dims(w)
    for t in range(T):
        out, lse, st = gpu_decode(w, inp, t)
        assert st == lla.LLA_OK
        ro, rl = oracle.sdpa(dm, widen(q), np.ascontiguousarray(Kt[:, :, :, t], dtype=np.float64),
                             np.ascontiguousarray(Vt[:, :, :, t], dtype=np.float64), lens, lens - 1)
        go = out.double().cpu().numpy()
        err = (np.abs(go - ro).max(-1) / np.abs(ro).max(-1)).max()
        assert err <= 1e-5, err
        assert np.abs(lse.double().cpu().numpy() - rl).max() <= 1e-5


def test_encode_then_decode_chain_bf16():
    """GPU encode then GPU decode against oracle encode (rounded to bf16) then oracle decode."""
    T, H, B, L_max = 4, 4, 3, 260
    w = workload(T=T, H=H, r_k=96, r_v=160, B=B, L_max=L_max, N_encode=B * L_max)
    inp = make_decode_inputs(w, 34, device="cuda", with_encode=True,
                             seq_lens=torch.tensor([260, 131, 1], dtype=torch.int32))
    N = B * L_max
    seq_idx = torch.tensor(np.repeat(np.arange(B), L_max).astype(np.int32), device="cuda")
    pos = torch.tensor(np.tile(np.arange(L_max), B).astype(np.int32), device="cuda")
    ck = torch.zeros((B, H, L_max, 96), dtype=torch.bfloat16, device="cuda")
    cv = torch.zeros((B, H, L_max, 160), dtype=torch.bfloat16, device="cuda")
    assert _encode(w, inp["x_k"], inp["x_v"], seq_idx, pos, inp["w_down_k"], inp["w_down_v"],
                   inp["mu_k"], inp["mu_v"], ck, cv) == lla.LLA_OK
    dm = oracle_dims(w)
    rk = np.zeros((B, H, L_max, 96))
    rv = np.zeros((B, H, L_max, 160))
    si, po = seq_idx.cpu().numpy(), pos.cpu().numpy()
    oracle.encode(dm, widen(inp["x_k"]), si, po, widen(inp["w_down_k"]), widen(inp["mu_k"]), 96, rk,
                  round_to_bf16=True)
    oracle.encode(dm, widen(inp["x_v"]), si, po, widen(inp["w_down_v"]), widen(inp["mu_v"]), 160, rv,
                  round_to_bf16=True)
    inp["cache_k"], inp["cache_v"] = ck, cv
    sl, qp = inp["seq_lens"].cpu().numpy(), inp["q_pos"].cpu().numpy()
    for t in range(T):
        out, lse, st = gpu_decode(w, inp, t)
        assert st == lla.LLA_OK
        ro, rl, _ = oracle.decode(dm, t, widen(inp["q"]), rk, rv, sl, qp, widen(inp["w_up_k"]),
                                  widen(inp["w_up_v"]), widen(inp["mu_k"]), widen(inp["mu_v"]))
        go = out.double().cpu().numpy()
        err = (np.abs(go - ro).max(-1) / np.maximum(np.abs(ro).max(-1), 1e-6)).max()
        assert err <= 2e-2, err
        assert np.abs(lse.double().cpu().numpy() - rl).max() <= 2e-2


def test_encode_prefill_full_size_sampled():
    """The long-context prefill at full size, in the launch configuration the bench
    times: lla_encode of every position of 64 sequences x 16384 tokens x 16 heads
    (1,048,576 tokens, x about 34 GB) in one call.  Every cache slot must be written
    (no canary left: a property that holds at any size), and sampled tokens (the
    first and last, both sides of tile and sequence boundaries, and random ones)
    must agree with the oracle's Eq. (2) under the bound of the random-input test."""
    from looped_transformer_cross_gb300.synth import WORKLOADS
    w = WORKLOADS["ouro_rho4_b64_16k"]
    B, H, L_max, N = w.B, w.H, w.L_max, w.N_encode
    assert N == B * L_max
    if torch.cuda.mem_get_info()[0] < 90e9:
        pytest.skip("needs about 90 GB of free device memory")
    inp = make_decode_inputs(w, 20260003, device="cuda", with_encode=True)
    ck, cv = inp.pop("cache_k").fill_(CANARY), inp.pop("cache_v").fill_(CANARY)
    seq_idx = torch.arange(B, dtype=torch.int32, device="cuda").repeat_interleave(L_max)
    pos = torch.arange(L_max, dtype=torch.int32, device="cuda").repeat(B)
    st = _encode(w, inp["x_k"], inp["x_v"], seq_idx, pos, inp["w_down_k"], inp["w_down_v"],
                 inp["mu_k"], inp["mu_v"], ck, cv)
    assert st == lla.LLA_OK
    assert not bool((ck == CANARY).any()) and not bool((cv == CANARY).any())
    g = np.random.default_rng(5)
    picks = [0, 127, 128, L_max - 1, L_max, N - 129, N - 128, N - 1]
    picks = np.unique(np.concatenate([picks, g.choice(N, size=40, replace=False)]))
    S = picks.shape[0]
    idx = torch.tensor(picks, dtype=torch.int64, device="cuda")
    dm = oracle_dims(w)
    zeros = np.zeros(S, dtype=np.int32)
    for cache, x, wd, mu, r in ((ck, "x_k", "w_down_k", "mu_k", w.r_k), (cv, "x_v", "w_down_v", "mu_v", w.r_v)):
        xs = widen(inp[x][idx])                          # [S][H][T*d]
        si = np.arange(S, dtype=np.int32)
        exact, rounded, mag = (np.zeros((S, H, 1, r)) for _ in range(3))
        oracle.encode(dm, xs, si, zeros, widen(inp[wd]), widen(inp[mu]), r, exact)
        oracle.encode(dm, xs, si, zeros, widen(inp[wd]), widen(inp[mu]), r, rounded, round_to_bf16=True)
        oracle.encode(dm, np.abs(xs - widen(inp[mu])[None]), si, zeros, np.abs(widen(inp[wd])),
                      np.zeros_like(widen(inp[mu])), r, mag)
        got = cache[idx // L_max, :, idx % L_max].double().cpu().numpy()   # [S][H][r]
        exact, rounded, mag = exact[:, :, 0], rounded[:, :, 0], mag[:, :, 0]
        half_ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(got), 2.0 ** -126))) - 8)
        assert np.all(np.abs(got - exact) <= half_ulp + 2.0 ** -20 * mag)
        assert (got == rounded).mean() > 0.99
