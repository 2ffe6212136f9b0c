"""The bounded wait's expiry on the GPU, made on purpose without a fault: the
workspace's test word (LLA_TEST_STALL at byte 4) makes the tile decode kernel's
first weights barrier expect one arrival more than it gets, so the value-MMA
issuer's wait runs out after about a second.  The call must report
LLA_ERR_TIMEOUT through the status word, the context must stay usable, and the
next call on the same (cleared) workspace must return the exact result."""
import os
import re
import time

import pytest
import torch

from lla_cases import gpu_decode, lla_dims, make_decode_inputs, workload
from looped_transformer_cross_gb300 import lla

pytestmark = pytest.mark.gpu

# the test word's value as include/lla.h defines it
with open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "lla.h")) as _h:
    LLA_TEST_STALL = int(re.search(r"#define\s+LLA_TEST_STALL\s+(0x[0-9A-Fa-f]+)u?", _h.read()).group(1), 16)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from looped_transformer_cross_gb300 import build
    build.build()


def test_bounded_wait_expires_then_next_call_is_exact():
    w = workload(T=2, H=4, r_k=96, r_v=160, B=3, L_max=600)
    assert lla.decode_kernel(lla_dims(w)) == "tile"
    inp = make_decode_inputs(w, 47, device="cuda", seq_lens=torch.tensor([600, 1, 300], dtype=torch.int32))
    ref_out, ref_lse, st = gpu_decode(w, inp, 1)
    assert st == lla.LLA_OK
    ws = lla.make_workspace(lla_dims(w), w.B, w.L_max)
    words = ws.view(torch.int32)
    words[1] = LLA_TEST_STALL
    t0 = time.perf_counter()
    _, _, st = gpu_decode(w, inp, 1, workspace=ws)      # reads and clears the status word
    elapsed = time.perf_counter() - t0
    assert st == lla.LLA_ERR_TIMEOUT
    assert elapsed < 30.0
    words[1] = 0
    torch.cuda.synchronize()
    out, lse, st = gpu_decode(w, inp, 1, workspace=ws)
    assert st == lla.LLA_OK
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
