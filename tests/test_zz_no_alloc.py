"""lla_decode_attn_noalloc: the decode entry point for callers that cannot allocate
device memory (its scratch is a fixed array inside the library).  Its results
must match lla_decode_attn with a caller workspace, call after call.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from lla_cases import TOL, gpu_decode, lla_dims, lse_err, make_decode_inputs, rel_err, workload
from looped_transformer_cross_gb300 import lla

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from looped_transformer_cross_gb300 import build
    build.build()


def _noalloc(w, inp, t, out, lse):
    dm = lla_dims(w)
    cos, sin = lla.rope_table(dm, max(w.L_max, 128))
    lla.decode_attn_noalloc(dm, t, inp["q"], inp["cache_k"], inp["cache_v"], inp["seq_lens"],
                            inp["q_pos"], inp["w_up_k"], inp["w_up_v"], inp["mu_k"], inp["mu_v"],
                            cos.cuda(), sin.cuda(), out, lse)
    torch.cuda.synchronize()


def test_noalloc_matches_workspace_entry_point_twice():
    # split units across CTAs and ragged tails, so the scratch records are exercised
    w = workload(T=4, H=16, r_k=96, r_v=160, B=6, L_max=1100)
    inp = make_decode_inputs(w, 41, device="cuda",
                             seq_lens=torch.tensor([1100, 1000, 257, 1, 129, 640], dtype=torch.int32))
    for t in (2, 3):
        ref_out, ref_lse, st = gpu_decode(w, inp, t)
        assert st == lla.LLA_OK
        go_ref, gl_ref = ref_out.double().cpu().numpy(), ref_lse.double().cpu().numpy()
        for _ in range(2):   # two calls in a row share the same scratch
            out = torch.full_like(ref_out, float("nan"))
            lse = torch.full_like(ref_lse, float("nan"))
            _noalloc(w, inp, t, out, lse)
            go, gl = out.double().cpu().numpy(), lse.double().cpu().numpy()
            assert np.all(np.isfinite(go))
            assert rel_err(go, go_ref) <= TOL["bf16"] and lse_err(gl, gl_ref) <= TOL["bf16"]


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
