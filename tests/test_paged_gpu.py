"""Parity of the paged-cache entries (lla_encode_paged, lla_decode_attn_paged) with
the oracle, through the C ABI.

Page tables as in "Enabling dynamic computation in Looped LMs" (§"Ragged KV",
Appendix A.1): a pool [num_pages][H][page_size][r] and a table [B][max_pages].
Pools are built from the dense test caches by moving rows exactly
(``oracle.paged.scatter``, or plain row copies at full size), physical pages are
shuffled, pages no entry names hold NaN and must never be read, and the expected
values are the oracle's on the dense view of the same rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import paged
from lla_cases import TOL, lla_dims, lse_err, oracle_dims, rel_err, widen, workload
from looped_transformer_cross_gb300 import lla
from looped_transformer_cross_gb300.synth import WORKLOADS, make_decode_inputs

pytestmark = pytest.mark.gpu
CANARY = -3072.0  # exactly representable in bf16 and fp32


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from looped_transformer_cross_gb300 import build
    build.build()


def _table(lens, P, max_pages, seed, extra=3):
    """Distinct shuffled physical pages for every logical page that holds a token;
    other entries -1 (never looked at); `extra` pages no entry names."""
    g = np.random.default_rng(seed)
    used = [(int(L) + P - 1) // P for L in lens]
    num_pages = sum(used) + extra
    perm = g.permutation(num_pages)
    bt = np.full((len(lens), max_pages), -1, np.int32)
    k = 0
    for b, u in enumerate(used):
        for lp in range(u):
            bt[b, lp] = perm[k]
            k += 1
    return bt, num_pages


def _pools(inp, bt, P, lens, num_pages):
    sd = inp["cache_k"].dtype
    return [torch.from_numpy(paged.scatter(widen(inp[n]), bt, P, lens, num_pages)).to(sd).cuda()
            for n in ("cache_k", "cache_v")]


def _gpu_paged(w, inp, pool_k, pool_v, bt, P, t, style=0):
    dm = lla_dims(w, style)
    B, H = inp["q"].shape[0], inp["q"].shape[1]
    cap = bt.shape[1] * P
    cos, sin = lla.rope_table(dm, max(cap, 128))
    cos, sin = cos.cuda(), sin.cuda()
    ws = lla.make_workspace(dm, B, cap)
    out = torch.empty((B, H, w.d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    lla.decode_attn_paged(dm, t, inp["q"], pool_k, pool_v, torch.from_numpy(bt).cuda(), P, inp["seq_lens"],
                          inp["q_pos"], inp["w_up_k"], inp["w_up_v"], inp["mu_k"], inp["mu_v"], cos, sin, out,
                          lse, ws)
    return out, lse, lla.device_status(ws)


def _oracle_dense(w, inp, ck, cv, t, style=0, bsel=None):
    sel = (lambda x: x) if bsel is None else (lambda x: x[list(bsel)])
    ro, rl, _ = oracle.decode(oracle_dims(w, style), t, widen(sel(inp["q"])), sel(ck), sel(cv),
                              sel(inp["seq_lens"]).cpu().numpy(), sel(inp["q_pos"]).cpu().numpy(),
                              widen(inp["w_up_k"]), widen(inp["w_up_v"]), widen(inp["mu_k"]), widen(inp["mu_v"]))
    return ro, rl


def _check(w, inp, pool_k, pool_v, bt, P, t, style=0):
    out, lse, st = _gpu_paged(w, inp, pool_k, pool_v, bt, P, t, style)
    assert st == lla.LLA_OK, lla.status_string(st)
    lens = inp["seq_lens"].cpu().numpy()
    ck = paged.gather(widen(pool_k), bt, P, lens)
    cv = paged.gather(widen(pool_v), bt, P, lens)
    ro, rl = _oracle_dense(w, inp, ck, cv, t, style)
    go, gl = out.double().cpu().numpy(), lse.double().cpu().numpy()
    assert np.all(np.isfinite(go))
    e_o, e_l = rel_err(go, ro), lse_err(gl, rl)
    assert e_o <= TOL[w.dtype] and e_l <= TOL[w.dtype], (e_o, e_l)


@pytest.mark.parametrize("P,r_v", [(1, 160), (8, 160), (16, 160), (32, 160), (64, 160), (100, 160),
                                   (128, 160), (256, 160), (16, 144)])
def test_paged_decode_tile_kernel(P, r_v):
    """The tile kernel's shapes in every kind of page: whole tiles inside a page
    (128, 256), a tile as 128/P page pieces (8, 16, 32, 64: with r_v a multiple of 32
    one box per page holds all of its V columns, else one box per 32-column chunk and
    page, the last zero-filled past r_v), and pages the tile copies do not take, whose
    rows are gathered one by one (1: the vLLM setting, 100)."""
    w = workload(T=2, H=4, r_k=96, r_v=r_v, B=5, L_max=400)
    lens = [400, 1, 129, 0, 256]
    inp = make_decode_inputs(w, 700 + P, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32))
    assert lla.decode_kernel(lla_dims(w)) == "tile"
    bt, npg = _table(lens, P, math.ceil(w.L_max / P), 701 + P)
    pk, pv = _pools(inp, bt, P, lens, npg)
    for t in range(w.T):
        _check(w, inp, pk, pv, bt, P, t)


@pytest.mark.parametrize("style,P", [(0, 128), (1, 128), (0, 1), (1, 16), (0, 24)])
def test_paged_decode_small_rank_kernel(style, P):
    """The small-rank kernel copies a head-tile's rows page by page, so it takes every
    page size: one-token pages, 16, 24 (a page boundary inside a tile) and 128."""
    w = workload(T=2, H=4, r_k=16, r_v=32, B=4, L_max=300)
    lens = [300, 128, 0, 5]
    inp = make_decode_inputs(w, 710 + style, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32))
    assert lla.decode_kernel(lla_dims(w, style)) == "small-rank"
    bt, npg = _table(lens, P, math.ceil(w.L_max / P), 711 + P)
    pk, pv = _pools(inp, bt, P, lens, npg)
    for t in range(w.T):
        _check(w, inp, pk, pv, bt, P, t, style)


@pytest.mark.parametrize("H,P", [(4, 8), (4, 32), (4, 64), (6, 16), (16, 16)])
def test_paged_decode_small_rank_set_pages(H, P):
    """Pages of 8..64 tokens on the small-rank kernel take the set-page layout: one
    copy per page for a whole head set (its heads lie together in a page), every
    epilogue group reading every ring slot; two-head sets (H = 6) and four-head sets,
    a last tile of a few rows in a part-filled page, an empty sequence."""
    w = workload(T=2, H=H, r_k=16, r_v=32, B=4, L_max=300)
    lens = [300, 128, 0, 5]
    inp = make_decode_inputs(w, 730 + H + P, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32))
    assert lla.decode_kernel(lla_dims(w)) == "small-rank"
    bt, npg = _table(lens, P, math.ceil(w.L_max / P), 731 + P)
    pk, pv = _pools(inp, bt, P, lens, npg)
    for t in range(w.T):
        _check(w, inp, pk, pv, bt, P, t)


@pytest.mark.parametrize("P", [1, 16])
def test_paged_decode_fp32_any_page_size(P):
    """fp32 mode takes any page size, down to the one-token pages of the page's own
    vLLM implementation."""
    w = workload(T=2, H=2, r_k=96, r_v=160, B=3, L_max=50, dtype="f32")
    lens = [50, 17, 0]
    inp = make_decode_inputs(w, 720 + P, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32))
    bt, npg = _table(lens, P, math.ceil(w.L_max / P), 721 + P)
    pk, pv = _pools(inp, bt, P, lens, npg)
    for t in range(w.T):
        _check(w, inp, pk, pv, bt, P, t)


def test_paged_decode_aliased_prefix():
    """Two sequences share their first page (a common prefix): aliased reads."""
    w = workload(T=2, H=4, r_k=96, r_v=160, B=2, L_max=300)
    lens = [300, 200]
    P = 128
    inp = make_decode_inputs(w, 730, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32))
    for n in ("cache_k", "cache_v"):
        inp[n][1, :, :P] = inp[n][0, :, :P]
    bt, npg = _table(lens, P, math.ceil(w.L_max / P), 731)
    bt[1, 0] = bt[0, 0]
    pk, pv = _pools(inp, bt, P, lens, npg)
    _check(w, inp, pk, pv, bt, P, 1)


@pytest.mark.parametrize("dtype,P", [("bf16", 128), ("bf16", 16), ("bf16", 1), ("f32", 16)])
def test_paged_encode_layout_exact(dtype, P):
    """Selector W_down and small-integer x: every latent is one x entry exactly and
    lands in row pos % P of head h of page bt[seq][pos // P]; every other pool row
    keeps its canary."""
    T, H, d, B, L_max, N = 2, 3, 128, 3, 256, 130
    rk, rv = 96, 160
    w = workload(T=T, H=H, r_k=rk, r_v=rv, B=B, L_max=L_max, dtype=dtype)
    sd = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = np.random.default_rng(740)
    slots = g.choice(B * L_max, size=N, replace=False)
    seq_idx = torch.tensor(slots // L_max, dtype=torch.int32)
    pos = torch.tensor(slots % L_max, dtype=torch.int32)
    max_pages = L_max // P
    bt, npg = _table([L_max] * B, P, max_pages, 741, extra=2)
    Td = T * d
    expect, tensors = {}, []
    for axis, r in ((0, rk), (1, rv)):
        u_of_k = (np.arange(r) * 37 + 11 + axis) % Td
        W = np.zeros((H, Td, r), np.float32)
        W[:, u_of_k, np.arange(r)] = 1.0
        x = ((np.arange(N)[:, None, None] * 3 + np.arange(H)[None, :, None] * 5 +
              np.arange(Td)[None, None, :] + axis) % 241 - 120).astype(np.float32)
        expect[axis] = x[:, :, u_of_k]
        tensors.append((torch.from_numpy(x).to(sd).cuda(), torch.from_numpy(W).to(sd).cuda()))
    mu = torch.zeros((H, Td), dtype=torch.float32, device="cuda")
    pk = torch.full((npg, H, P, rk), CANARY, dtype=sd, device="cuda")
    pv = torch.full((npg, H, P, rv), CANARY, dtype=sd, device="cuda")
    dm = lla_dims(w)
    ws = lla.make_workspace(dm, B, max_pages * P, N)
    lla.encode_paged(dm, tensors[0][0], tensors[1][0], seq_idx.cuda(), pos.cuda(), tensors[0][1], tensors[1][1],
                     mu, mu, pk, pv, torch.from_numpy(bt).cuda(), P, ws)
    assert lla.device_status(ws) == lla.LLA_OK
    for axis, pool in ((0, pk), (1, pv)):
        got = pool.float().cpu().numpy()
        touched = np.zeros(got.shape[:3], bool)
        for n in range(N):
            pg, row = paged.slot(bt, P, int(seq_idx[n]), int(pos[n]))
            np.testing.assert_array_equal(got[pg, :, row], expect[axis][n])
            touched[pg, :, row] = True
        assert np.all(got[~touched] == CANARY)


def test_paged_out_of_range_page_is_flagged():
    """A table entry outside [0, num_pages): decode reads a page inside the pool
    instead and records LLA_ERR_DEVICE_ARG; encode skips the write and records it."""
    w = workload(T=2, H=2, r_k=96, r_v=160, B=2, L_max=256)
    lens = [256, 100]
    P = 128
    inp = make_decode_inputs(w, 750, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32),
                             with_encode=True)
    bt, npg = _table(lens, P, 2, 751)
    pk, pv = _pools(inp, bt, P, lens, npg)
    bad = bt.copy()
    bad[0, 1] = npg + 7
    out, lse, st = _gpu_paged(w, inp, pk, pv, bad, P, 0)
    assert st == lla.LLA_ERR_DEVICE_ARG
    assert torch.isfinite(out[1]).all()
    before_k = pk.clone()
    dm = lla_dims(w)
    ws = lla.make_workspace(dm, 2, 2 * P, 2)
    seq_idx = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    pos = torch.tensor([200, 50], dtype=torch.int32, device="cuda")   # token 200 of seq 0: the bad page
    lla.encode_paged(dm, inp["x_k"][:2], inp["x_v"][:2], seq_idx, pos, inp["w_down_k"], inp["w_down_v"],
                     inp["mu_k"], inp["mu_v"], pk, pv, torch.from_numpy(bad).cuda(), P, ws)
    assert lla.device_status(ws) == lla.LLA_ERR_DEVICE_ARG
    # only sequence 1's slot changed (compared as bit patterns: unnamed rows hold NaN)
    pg, row = paged.slot(bt, P, 1, 50)
    changed = (pk.view(torch.int16) != before_k.view(torch.int16)).any(dim=-1).nonzero().tolist()
    assert changed and all(c[0] == pg and c[2] == row for c in changed)


@pytest.mark.parametrize("P", [256, 16])
def test_paged_bench_layer_sampled(P):
    """The Ouro-1.4B rho = 4 layer (32 x 3584..4096) in 256- and 16-token pages,
    shuffled, in the launch the bench times; sequences 0 and 31 against the oracle."""
    w = WORKLOADS["ouro1.4b_rho4_b32_4k"]
    inp = make_decode_inputs(w, 760, device="cuda")
    lens = inp["seq_lens"].cpu().numpy()
    max_pages = w.L_max // P
    bt, npg = _table(lens, P, max_pages, 761)
    pools = []
    for n in ("cache_k", "cache_v"):
        dense = inp[n]
        pool = torch.full((npg,) + (w.H, P, dense.shape[-1]), float("nan"), dtype=dense.dtype, device="cuda")
        for b in range(w.B):
            for lp in range((int(lens[b]) + P - 1) // P):
                pool[int(bt[b, lp])] = dense[b, :, lp * P:(lp + 1) * P]
        pools.append(pool)
    out, lse, st = _gpu_paged(w, inp, pools[0], pools[1], bt, P, 2)
    assert st == lla.LLA_OK
    bsel = (0, 31)
    sl = inp["seq_lens"][list(bsel)].cpu().numpy()
    qp = inp["q_pos"][list(bsel)].cpu().numpy()
    ro, rl, _ = oracle.decode(oracle_dims(w), 2, widen(inp["q"][list(bsel)]), widen(inp["cache_k"][list(bsel)]),
                              widen(inp["cache_v"][list(bsel)]), sl, qp, widen(inp["w_up_k"]), widen(inp["w_up_v"]),
                              widen(inp["mu_k"]), widen(inp["mu_v"]))
    go = out.double().cpu().numpy()[list(bsel)]
    gl = lse.double().cpu().numpy()[list(bsel)]
    assert rel_err(go, ro) <= TOL["bf16"] and lse_err(gl, rl) <= TOL["bf16"]
