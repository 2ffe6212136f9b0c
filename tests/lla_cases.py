"""Shared helpers for the parity tests: run the CUDA path and the oracle on the
same seeded inputs and compare them with the tolerance rule of the tests.

Tolerance (per output vector): max|o_gpu - o_ref| / max(max|o_ref|, 1e-6) over
every (sequence, head), and max |lse_gpu - lse_ref|; 2e-2 for bf16 storage with
fp32 accumulation, 1e-5 for fp32 storage.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
from looped_transformer_cross_gb300 import lla
from looped_transformer_cross_gb300.synth import Workload, make_decode_inputs, widen

TOL = {"bf16": 2e-2, "f32": 1e-5}


def workload(**kw) -> Workload:
    base = dict(name="test", T=2, H=2, d=128, r_k=96, r_v=160, B=3, L_max=300, len_lo=1,
                len_hi=300)
    base.update(kw)
    return Workload(**base)


def lla_dims(w: Workload, rope_style=0):
    return lla.dims(w.T, w.H, w.r_k, w.r_v, d_head=w.d, variant=w.variant,
                    dtype=lla.LLA_BF16 if w.dtype == "bf16" else lla.LLA_F32,
                    rope_base=w.rope_base, rope_style=rope_style)


def oracle_dims(w: Workload, rope_style=0):
    return oracle.dims(w.T, w.H, w.d, w.r_k, w.r_v, w.variant, w.rope_base, rope_style)


def gpu_decode(w: Workload, inp: dict, t: int, rope_style=0, workspace=None, out=None, lse=None):
    """lla_decode_attn through the C ABI; returns (out, lse, device status)."""
    dm = lla_dims(w, rope_style)
    cos, sin = lla.rope_table(dm, max(w.L_max, 128))
    cos, sin = cos.cuda(), sin.cuda()
    B, H = inp["q"].shape[0], inp["q"].shape[1]
    if workspace is None:
        workspace = lla.make_workspace(dm, B, w.L_max)
    if out is None:
        out = torch.empty((B, H, w.d), dtype=torch.float32, device="cuda")
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    lla.decode_attn(dm, t, inp["q"], inp["cache_k"], inp["cache_v"], inp["seq_lens"],
                    inp["q_pos"], inp["w_up_k"], inp["w_up_v"], inp["mu_k"], inp["mu_v"], cos, sin,
                    out, lse, workspace)
    st = lla.device_status(workspace)
    return out, lse, st


def oracle_decode(w: Workload, inp: dict, t: int, rope_style=0, bsel=None):
    """The oracle on the same stored tensors (widened exactly to fp64), optionally
    on a subset of sequences ``bsel``."""
    def sel(x):
        return x if bsel is None else x[list(bsel)]
    sl = sel(inp["seq_lens"]).cpu().numpy()
    qp = sel(inp["q_pos"]).cpu().numpy()
    out, lse, _ = oracle.decode(oracle_dims(w, rope_style), t, widen(sel(inp["q"])),
                                widen(sel(inp["cache_k"])), widen(sel(inp["cache_v"])), sl, qp,
                                widen(inp["w_up_k"]), widen(inp["w_up_v"]), widen(inp["mu_k"]),
                                widen(inp["mu_v"]))
    return out, lse


def rel_err(o_gpu: np.ndarray, o_ref: np.ndarray) -> float:
    num = np.abs(o_gpu - o_ref).max(axis=-1)
    den = np.maximum(np.abs(o_ref).max(axis=-1), 1e-6)
    return float((num / den).max()) if num.size else 0.0


def lse_err(l_gpu: np.ndarray, l_ref: np.ndarray) -> float:
    both_inf = np.isneginf(l_gpu) & np.isneginf(l_ref)
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(l_gpu - l_ref))
    return float(d.max()) if d.size else 0.0


def compare(w: Workload, inp: dict, t: int, rope_style=0, bsel=None, tol=None):
    out, lse, st = gpu_decode(w, inp, t, rope_style)
    assert st == lla.LLA_OK, lla.status_string(st)
    ro, rl = oracle_decode(w, inp, t, rope_style, bsel)
    go = out.cpu().double().numpy()
    gl = lse.cpu().double().numpy()
    if bsel is not None:
        go, gl = go[list(bsel)], gl[list(bsel)]
    e_o, e_l = rel_err(go, ro), lse_err(gl, rl)
    tol = TOL[w.dtype] if tol is None else tol
    assert np.all(np.isfinite(go)), "non-finite output"
    assert e_o <= tol and e_l <= tol, "rel err %.3g, lse err %.3g (tol %g)" % (e_o, e_l, tol)
    return e_o, e_l


__all__ = ["TOL", "workload", "lla_dims", "oracle_dims", "gpu_decode", "oracle_decode", "rel_err",
           "lse_err", "compare", "make_decode_inputs", "widen", "dataclasses"]
