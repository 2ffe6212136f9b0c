"""lla_decode_attn_noalloc: the decode entry point for callers that cannot allocate
device memory (a plugin whose host framework's pool owns the GPU, a serving path
that must never call cudaMalloc).  Its scratch is a fixed array inside the library.
Its results must equal, bit for bit, those of lla_decode_attn with a caller
workspace, call after call, on every kernel family (each lays its scratch out
differently), and its device status must be readable.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import pytest
import torch

from lla_cases import gpu_decode, lla_dims, make_decode_inputs, workload
from looped_transformer_cross_gb300 import lla

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from looped_transformer_cross_gb300 import build
    build.build()


def _noalloc(w, inp, t, out, lse, loop_t=None):
    dm = lla_dims(w)
    cos, sin = lla.rope_table(dm, max(w.L_max, 128))
    lla.decode_attn_noalloc(dm, t if loop_t is None else loop_t, inp["q"], inp["cache_k"],
                            inp["cache_v"], inp["seq_lens"], inp["q_pos"], inp["w_up_k"],
                            inp["w_up_v"], inp["mu_k"], inp["mu_v"], cos.cuda(), sin.cuda(), out, lse)


# one case per kernel family: tile, small-rank, LLA-2D CTA pairs, fp32
CASES = {
    "tile": (dict(T=4, H=16, r_k=96, r_v=160, B=6, L_max=1100), [1100, 1000, 257, 1, 129, 640]),
    "small-rank": (dict(T=4, H=16, r_k=16, r_v=32, B=5, L_max=1100), [1100, 0, 513, 1, 1000]),
    "pair-2d": (dict(T=2, H=16, r_k=128, r_v=256, B=3, L_max=1100, variant=1), [1100, 700, 1]),
    "fp32": (dict(T=2, H=4, r_k=48, r_v=80, B=3, L_max=300, dtype="f32"), [300, 7, 128]),
}


@pytest.mark.parametrize("family", sorted(CASES))
def test_noalloc_equals_workspace_entry_point_twice(family):
    kw, lens = CASES[family]
    w = workload(**kw)
    assert lla.decode_kernel(lla_dims(w)) == family
    inp = make_decode_inputs(w, 41, device="cuda", seq_lens=torch.tensor(lens, dtype=torch.int32))
    for t in (0, w.T - 1):
        ref_out, ref_lse, st = gpu_decode(w, inp, t)
        assert st == lla.LLA_OK
        for _ in range(2):   # two calls in a row share the same scratch
            out = torch.full_like(ref_out, float("nan"))
            lse = torch.full_like(ref_lse, float("nan"))
            _noalloc(w, inp, t, out, lse)
            assert lla.device_status(None) == lla.LLA_OK
            assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_noalloc_device_status_is_readable():
    """An out-of-range length seen by the kernels is recorded in the scratch's status
    word and read back with no workspace; a call the host checks reject enqueues
    nothing (the recorded word survives it); the next valid call starts clean."""
    w = workload(T=2, H=16, r_k=96, r_v=160, B=2, L_max=256)
    inp = make_decode_inputs(w, 43, device="cuda", seq_lens=torch.tensor([256, 100], dtype=torch.int32))
    out = torch.empty((w.B, w.H, w.d), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    inp["seq_lens"][0] = w.L_max + 100
    _noalloc(w, inp, 0, out, lse)
    assert lla.device_status(None, clear=False) == lla.LLA_ERR_DEVICE_ARG
    with pytest.raises(lla.LLAError) as e:
        _noalloc(w, inp, 0, out, lse, loop_t=w.T)          # rejected on the host
    assert e.value.status == lla.LLA_ERR_INVALID_ARG
    assert lla.device_status(None) == lla.LLA_ERR_DEVICE_ARG   # read, then cleared
    assert lla.device_status(None) == lla.LLA_OK
    inp["seq_lens"][0] = w.L_max
    _noalloc(w, inp, 1, out, lse)
    assert lla.device_status(None) == lla.LLA_OK
    ref_out, ref_lse, st = gpu_decode(w, inp, 1)
    assert st == lla.LLA_OK and torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    w = workload(T=1, H=16, r_k=16, r_v=160, B=1000, L_max=1)
    dm = lla_dims(w)
    assert lla.workspace_size(dm, w.B, w.L_max) > (64 << 20)   # LLA_NOALLOC_SCRATCH_BYTES
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(lla.LLAError) as e:
        lla.decode_attn_noalloc(dm, 0, t, torch.zeros((w.B, w.H, w.L_max, 16), dtype=torch.bfloat16, device="cuda"),
                                torch.zeros((w.B, w.H, w.L_max, 160), dtype=torch.bfloat16, device="cuda"),
                                t, t, t, t, o, o, torch.zeros((128, 64), device="cuda"),
                                torch.zeros((128, 64), device="cuda"), o, o)
    assert e.value.status == lla.LLA_ERR_UNSUPPORTED
