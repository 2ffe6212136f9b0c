"""Parity of the LLA-2D path (one latent per token shared by all heads) with the oracle.

lla_decode_attn with variant LLA_2D runs the CTA-pair score kernel and the value
kernel (bf16, H even <= 16, r_k <= 128, r_v <= 256), else the plain kernels (fp32
storage, or bf16 at other head counts and at ranks up to 512); lla_encode maps the
whole stack x in R^{T*H*d} to one latent.  The oracle computes the plain
definition (every head's K/V reconstructed from the shared latent, RoPE, softmax)
in fp64 on the same stored tensors.  Cases span several 256-token pair blocks,
ragged tails (a CTA of the pair with no valid token, partial 16-token value
steps), empty sequences and runs split between CTA pairs and value CTAs.
"""
import numpy as np
import pytest
import torch

import oracle
from lla_cases import compare, gpu_decode, lla_dims, oracle_decode, oracle_dims, rel_err, lse_err, workload
from looped_transformer_cross_gb300 import lla
from looped_transformer_cross_gb300.synth import WORKLOADS, make_decode_inputs, widen

pytestmark = pytest.mark.gpu

CANARY = -3072.0


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from looped_transformer_cross_gb300 import build
    build.build()


def w2d(**kw):
    base = dict(variant=1, T=2, H=4, r_k=128, r_v=256, B=4, L_max=1300)
    base.update(kw)
    return workload(**base)


def _inputs(w, seed, lens):
    return make_decode_inputs(w, seed, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32))


@pytest.mark.parametrize("H,rk,rv", [(4, 128, 256), (16, 128, 256), (8, 64, 128), (4, 96, 160),
                                     (4, 32, 64), (12, 128, 192)])
def test_2d_bf16_ragged(H, rk, rv):
    """Blocks of 512 tokens cut at 1300 / 513 / 1 tokens and an empty sequence."""
    w = w2d(H=H, r_k=rk, r_v=rv)
    inp = _inputs(w, 400 + H + rk + rv, [1300, 513, 1, 0])
    for t in range(w.T):
        compare(w, inp, t)


def test_2d_bf16_interleaved_rope():
    w = w2d(H=8, B=2, L_max=700)
    inp = _inputs(w, 41, [700, 300])
    compare(w, inp, 1, rope_style=1)


def test_2d_f32_mode():
    w = w2d(H=4, r_k=64, r_v=96, B=3, L_max=300, dtype="f32")
    inp = _inputs(w, 42, [300, 129, 0])
    for t in range(w.T):
        compare(w, inp, t)


def test_2d_padding_is_never_read():
    """NaN in every slot at or beyond seq_lens must not change a single output bit
    (value chunks past the end are zeroed before the value MMA reads them)."""
    w = w2d(H=4, B=3, L_max=1100)
    lens = [1100, 700, 200]
    inp = _inputs(w, 43, lens)
    ref_out, ref_lse, _ = gpu_decode(w, inp, 1)
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
    for b, L in enumerate(lens):
        inp["cache_k"][b, L:] = float("nan")
        inp["cache_v"][b, L:] = float("nan")
    out, lse, st = gpu_decode(w, inp, 1)
    assert st == lla.LLA_OK
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_2d_softmax_weights_normalised():
    """Constant V latents with a one-hot W_up,v and mu_v = 0 give out[e] = 1 for every
    head: the value MMA's weights and the record sums come from the same bf16 p."""
    w = w2d(H=8, r_k=64, r_v=128, B=2, L_max=1500)
    inp = _inputs(w, 44, [1500, 333])
    inp["cache_v"].fill_(1.0)
    wv = torch.zeros_like(inp["w_up_v"])          # [T][H*d][r_v]
    for h in range(w.H):
        for e in range(128):
            wv[:, h * 128 + e, e] = 1.0
    inp["w_up_v"] = wv
    inp["mu_v"].zero_()
    out, _, st = gpu_decode(w, inp, 0)
    assert st == lla.LLA_OK
    np.testing.assert_allclose(out.cpu().numpy(), 1.0, rtol=0, atol=2e-6)


def test_2d_growing_scores_rescale_accumulators():
    """K latents scaled up along the sequence: the 32-token groups' references span a
    wide range, so the value kernel scales most groups' weights by large powers of two
    (and flushes the smallest to zero) before the value MMA."""
    w = w2d(H=4, B=2, L_max=2600)
    inp = _inputs(w, 45, [2600, 1800])
    ramp = torch.linspace(1.0, 4.0, w.L_max, device="cuda").view(1, w.L_max, 1)
    inp["cache_k"] = (inp["cache_k"].float() * ramp).to(inp["cache_k"].dtype).contiguous()
    compare(w, inp, 0)
    inp["cache_k"] = inp["cache_k"].flip(1).contiguous()
    compare(w, inp, 1)


def test_2d_runs_split_between_pairs():
    """More blocks than CTA pairs, ragged lengths: most sequences are cut between pairs
    and most pairs see several sequences (records merged by the combine kernel)."""
    w = w2d(H=4, r_k=64, r_v=128, B=40, L_max=3000)
    g = np.random.default_rng(46)
    lens = [int(x) for x in g.integers(1, 3001, size=40)]
    lens[3] = 0
    inp = _inputs(w, 46, lens)
    compare(w, inp, 1)


def test_2d_repeated_calls_are_deterministic():
    w = w2d(H=16, B=6, L_max=1500)
    inp = _inputs(w, 47, [1500, 1400, 900, 600, 513, 512])
    a, la, _ = gpu_decode(w, inp, 1)
    a, la = a.clone(), la.clone()
    for _ in range(3):
        b, lb, st = gpu_decode(w, inp, 1)
        assert st == lla.LLA_OK and torch.equal(a, b) and torch.equal(la, lb)


def test_2d_unsupported_shapes():
    """Ranks above 512 (the LLA-2D limit) are refused before any launch: no kernel
    family, no workspace size, LLA_ERR_UNSUPPORTED from the call itself."""
    for rk, rv in ((528, 128), (128, 528)):
        w = w2d(H=4, r_k=rk, r_v=rv, B=1, L_max=64)
        dm = lla_dims(w)
        assert lla.decode_kernel(dm) is None
        with pytest.raises(lla.LLAError):
            lla.make_workspace(dm, 1, 64)
        inp = _inputs(w, 48, [64])
        with pytest.raises(lla.LLAError) as e:
            gpu_decode(w, inp, 0, workspace=torch.zeros(1 << 20, dtype=torch.uint8, device="cuda"))
        assert e.value.status == lla.LLA_ERR_UNSUPPORTED


@pytest.mark.parametrize("H,rk,rv", [(4, 256, 512), (2, 512, 128), (3, 128, 256), (20, 64, 128),
                                     (4, 496, 384)])
def test_2d_bf16_plain_shapes(H, rk, rv):
    """Shapes outside the CTA-pair kernels' range (ranks above 128 / 256, odd or more
    than 16 heads) run the plain kernels over bf16 storage: parity, ragged lengths."""
    w = w2d(H=H, r_k=rk, r_v=rv, B=3, L_max=300)
    assert lla.decode_kernel(lla_dims(w)) == "plain-2d"
    inp = _inputs(w, 500 + H + rk + rv, [300, 129, 0])
    compare(w, inp, 1)


def test_2d_pair_shapes_take_the_pair_kernels():
    for H, rk, rv in ((2, 16, 16), (16, 128, 256), (6, 64, 96)):
        assert lla.decode_kernel(lla_dims(w2d(H=H, r_k=rk, r_v=rv))) == "pair-2d"


def test_2d_f32_rank_512():
    w = w2d(H=4, r_k=512, r_v=512, B=2, L_max=200, dtype="f32")
    inp = _inputs(w, 52, [200, 77])
    compare(w, inp, 0)


@pytest.mark.parametrize("dtype,rk,rv", [("bf16", 512, 384), ("bf16", 496, 272), ("f32", 512, 320)])
def test_2d_encode_large_ranks(dtype, rk, rv):
    """Encode at LLA-2D ranks above 256 (one 512-column accumulator in the bf16 kernel):
    each latent within half a bf16 spacing plus the fp32 accumulation bound of the
    Eq. (2) sum (bf16), or within the sequential-summation bound (fp32)."""
    T, H, B, L_max, N = 2, 4, 2, 80, 150
    w = w2d(T=T, H=H, r_k=rk, r_v=rv, B=B, L_max=L_max, N_encode=N, dtype=dtype)
    inp = make_decode_inputs(w, 53, device="cuda", with_encode=True)
    seq_idx = torch.tensor(np.arange(N) % B, dtype=torch.int32, device="cuda")
    pos = torch.tensor(np.arange(N) // B, dtype=torch.int32, device="cuda")
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    ck = torch.full((B, L_max, rk), CANARY, dtype=tdt, device="cuda")
    cv = torch.full((B, L_max, rv), CANARY, dtype=tdt, device="cuda")
    dm = lla_dims(w)
    wsp = lla.make_workspace(dm, B, L_max, N)
    lla.encode(dm, inp["x_k"], inp["x_v"], seq_idx, pos, inp["w_down_k"], inp["w_down_v"],
               inp["mu_k"], inp["mu_v"], ck, cv, wsp)
    assert lla.device_status(wsp) == lla.LLA_OK
    od = oracle_dims(w)
    si, po = seq_idx.cpu().numpy(), pos.cpu().numpy()
    for cache, x, wd, mu, r in ((ck, "x_k", "w_down_k", "mu_k", rk), (cv, "x_v", "w_down_v", "mu_v", rv)):
        exact = np.full((B, L_max, r), CANARY)
        oracle.encode(od, widen(inp[x]), si, po, widen(inp[wd]), widen(inp[mu]), r, exact)
        mag = np.zeros((B, L_max, r))
        oracle.encode(od, np.abs(widen(inp[x]) - widen(inp[mu])[None]), si, po, np.abs(widen(inp[wd])),
                      np.zeros_like(widen(inp[mu])), r, mag)
        got = cache.double().cpu().numpy()
        touched = got != CANARY
        assert touched.sum() == N * r
        if dtype == "bf16":
            half_ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(got), 2.0 ** -126))) - 8)
            bound = half_ulp + 2.0 ** -20 * mag
        else:
            # sequential fp32 sum of T*H*d products: at most n u sum|terms|
            bound = T * H * 128 * 2.0 ** -24 * mag + 1e-30
        assert np.all(np.abs(got - exact)[touched] <= bound[touched])


def test_2d_encode_layout_structured_exact():
    """Selector W_down over the T*H*d stack and small-integer x: every latent is one x
    entry exactly, in slot (seq_idx[n], pos[n]); untouched slots keep the canary."""
    T, H, d, B, L_max, N, rk, rv = 2, 4, 128, 3, 200, 130, 128, 256
    w = w2d(T=T, H=H, r_k=rk, r_v=rv, B=B, L_max=L_max)
    width = T * H * d
    g = np.random.default_rng(5)
    slots = g.choice(B * L_max, size=N, replace=False)
    seq_idx = torch.tensor(slots // L_max, dtype=torch.int32, device="cuda")
    pos = torch.tensor(slots % L_max, dtype=torch.int32, device="cuda")
    expect, xs, ws = {}, [], []
    for axis, r in ((0, rk), (1, rv)):
        u_of_k = (np.arange(r) * 53 + 7 + axis) % width
        W = np.zeros((width, r), np.float32)
        W[u_of_k, np.arange(r)] = 1.0
        x = ((np.arange(N)[:, None] * 3 + np.arange(width)[None, :] + axis) % 241 - 120).astype(np.float32)
        expect[axis] = x[:, u_of_k]
        xs.append(torch.from_numpy(x).to(torch.bfloat16).cuda())
        ws.append(torch.from_numpy(W).to(torch.bfloat16).cuda())
    mu = torch.zeros(width, dtype=torch.float32, device="cuda")
    ck = torch.full((B, L_max, rk), CANARY, dtype=torch.bfloat16, device="cuda")
    cv = torch.full((B, L_max, rv), CANARY, dtype=torch.bfloat16, device="cuda")
    dm = lla_dims(w)
    wsp = lla.make_workspace(dm, B, L_max, N)
    lla.encode(dm, xs[0], xs[1], seq_idx, pos, ws[0], ws[1], mu, mu, ck, cv, wsp)
    assert lla.device_status(wsp) == lla.LLA_OK
    for axis, cache in ((0, ck), (1, cv)):
        got = cache.float().cpu().numpy()
        touched = np.zeros(got.shape[:2], bool)
        for n in range(N):
            b, p = int(seq_idx[n]), int(pos[n])
            np.testing.assert_array_equal(got[b, p], expect[axis][n])
            touched[b, p] = True
        assert np.all(got[~touched] == CANARY)


def test_2d_encode_random_vs_oracle():
    """Random stack: each latent within half a bf16 spacing plus the fp32 accumulation
    bound of the exact Eq. (2) sum over T*H*d terms; almost all equal the oracle's
    fp64 sum rounded to bf16."""
    T, H, B, L_max, N, rk, rv = 2, 4, 2, 96, 100, 64, 128
    w = w2d(T=T, H=H, r_k=rk, r_v=rv, B=B, L_max=L_max, N_encode=N)
    inp = make_decode_inputs(w, 49, device="cuda", with_encode=True)
    seq_idx = torch.tensor(np.arange(N) % B, dtype=torch.int32, device="cuda")
    pos = torch.tensor(np.arange(N) // B, dtype=torch.int32, device="cuda")
    ck = torch.full((B, L_max, rk), CANARY, dtype=torch.bfloat16, device="cuda")
    cv = torch.full((B, L_max, rv), CANARY, dtype=torch.bfloat16, device="cuda")
    dm = lla_dims(w)
    wsp = lla.make_workspace(dm, B, L_max, N)
    lla.encode(dm, inp["x_k"], inp["x_v"], seq_idx, pos, inp["w_down_k"], inp["w_down_v"],
               inp["mu_k"], inp["mu_v"], ck, cv, wsp)
    assert lla.device_status(wsp) == lla.LLA_OK
    od = oracle_dims(w)
    si, po = seq_idx.cpu().numpy(), pos.cpu().numpy()
    for cache, x, wd, mu, r in ((ck, "x_k", "w_down_k", "mu_k", rk), (cv, "x_v", "w_down_v", "mu_v", rv)):
        exact = np.full((B, L_max, r), CANARY)
        oracle.encode(od, widen(inp[x]), si, po, widen(inp[wd]), widen(inp[mu]), r, exact)
        rounded = np.full((B, L_max, r), CANARY)
        oracle.encode(od, widen(inp[x]), si, po, widen(inp[wd]), widen(inp[mu]), r, rounded,
                      round_to_bf16=True)
        mag = np.zeros((B, L_max, r))
        oracle.encode(od, np.abs(widen(inp[x]) - widen(inp[mu])[None]), si, po, np.abs(widen(inp[wd])),
                      np.zeros_like(widen(inp[mu])), r, mag)
        got = cache.double().cpu().numpy()
        touched = got != CANARY
        assert touched.sum() == N * r
        half_ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(got), 2.0 ** -126))) - 8)
        bound = half_ulp + 2.0 ** -20 * mag
        assert np.all(np.abs(got - exact)[touched] <= bound[touched])
        assert (got == rounded)[touched].mean() > 0.99


def test_2d_encode_then_decode_chain():
    """Encode a history with lla_encode, then decode it: the same answer as the oracle
    decoding the oracle-encoded (bf16-rounded) latents, up to the bf16 tolerance."""
    T, H, B, L_max, rk, rv = 2, 4, 2, 700, 64, 128
    w = w2d(T=T, H=H, r_k=rk, r_v=rv, B=B, L_max=L_max, N_encode=B * L_max)
    inp = make_decode_inputs(w, 50, device="cuda", with_encode=True,
                             seq_lens=torch.tensor([700, 450], dtype=torch.int32))
    N = B * L_max
    seq_idx = torch.tensor(np.arange(N) // L_max, dtype=torch.int32, device="cuda")
    pos = torch.tensor(np.arange(N) % L_max, dtype=torch.int32, device="cuda")
    dm = lla_dims(w)
    wsp = lla.make_workspace(dm, B, L_max, N)
    lla.encode(dm, inp["x_k"], inp["x_v"], seq_idx, pos, inp["w_down_k"], inp["w_down_v"],
               inp["mu_k"], inp["mu_v"], inp["cache_k"], inp["cache_v"], wsp)
    assert lla.device_status(wsp) == lla.LLA_OK
    compare(w, inp, 1)


def test_lla2d_b256_8k_sampled():
    """The LLA-2D workload at full size (256 sequences x 8192 tokens, H = 16, r = (128,
    256)) in the bench's launch; three sequences checked against the oracle in full."""
    w = WORKLOADS["lla2d_b256_8k"]
    inp = make_decode_inputs(w, 20260004, device="cuda")
    out, lse, st = gpu_decode(w, inp, 2)
    assert st == lla.LLA_OK
    go, gl = out.cpu().double().numpy(), lse.cpu().double().numpy()
    assert np.all(np.isfinite(go)) and np.all(np.isfinite(gl))
    bsel = [0, 131, 255]
    ro, rl = oracle_decode(w, inp, 2, bsel=bsel)
    e_o, e_l = rel_err(go[bsel], ro), lse_err(gl[bsel], rl)
    assert e_o <= 2e-2 and e_l <= 2e-2, (e_o, e_l)
