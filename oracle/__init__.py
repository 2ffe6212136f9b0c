"""The oracle for Looped Latent Attention: plain fp64 CPU code, test infrastructure.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product library (``looped_transformer_cross_gb300``)
never does, and this package imports nothing from it.

Two independent statements of the method live here:

* ``lla_oracle.c`` (loaded through :func:`lib`): the paper's equations in plain C,
  fp64, parallel over (sequence, head) with OpenMP.
* ``brute.py``: a numpy restatement for tiny shapes that materialises every
  reconstructed K/V and every rotation matrix.

Source: "Looped Latent Attention: Cross-Loop KV Compression for Looped
Transformers" (arXiv 2607.15456v2), §3 and Appendix J.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lla_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


class OracleDims(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int),
        ("H", ctypes.c_int),
        ("d", ctypes.c_int),
        ("r_k", ctypes.c_int),
        ("r_v", ctypes.c_int),
        ("variant", ctypes.c_int),
        ("rope_base", ctypes.c_double),
        ("rope_style", ctypes.c_int),
    ]


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc (-O2, OpenMP) if missing or stale."""
    stale = (not os.path.exists(_SO)) or os.path.getmtime(_SO) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "lla_oracle.h")))
    if force or stale:
        tmp = _SO + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def lib():
    """Load (building first if needed) the C oracle."""
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int)
            pd = ctypes.POINTER(OracleDims)
            L.oracle_compression_ratio.argtypes = [pd]
            L.oracle_compression_ratio.restype = ctypes.c_double
            L.oracle_teacher_scalars_per_token.argtypes = [pd, ctypes.c_int]
            L.oracle_teacher_scalars_per_token.restype = ctypes.c_longlong
            L.oracle_latent_scalars_per_token.argtypes = [pd, ctypes.c_int]
            L.oracle_latent_scalars_per_token.restype = ctypes.c_longlong
            L.oracle_round_bf16.argtypes = [ctypes.c_double]
            L.oracle_round_bf16.restype = ctypes.c_double
            L.oracle_encode.argtypes = [pd, ctypes.c_int, dp, ip, ip, dp, dp, ctypes.c_int,
                                        dp, ctypes.c_int, ctypes.c_long, ctypes.c_int]
            L.oracle_encode.restype = ctypes.c_int
            L.oracle_decode.argtypes = [pd, ctypes.c_int, ctypes.c_int, ctypes.c_long, dp, dp, dp,
                                        ip, ip, ctypes.c_long, dp, dp, dp, dp, dp, dp, dp,
                                        ctypes.c_int]
            L.oracle_decode.restype = ctypes.c_int
            L.oracle_sdpa.argtypes = [pd, ctypes.c_int, ctypes.c_long, dp, dp, dp, ip, ip,
                                      ctypes.c_long, dp, dp]
            L.oracle_sdpa.restype = ctypes.c_int
            L.oracle_hybrid.argtypes = [pd, ctypes.c_int, ctypes.c_int, ctypes.c_long, ctypes.c_long, dp, dp, dp,
                                        ip, ip, dp, dp, dp, dp, dp, dp, ip, ip, dp, dp]
            L.oracle_hybrid.restype = ctypes.c_int
            L.oracle_decoupled.argtypes = [pd, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_long, dp, dp, dp,
                                           dp, ip, ip, ctypes.c_long, dp, dp, dp, dp, dp, dp]
            L.oracle_decoupled.restype = ctypes.c_int
            L.oracle_num_threads.argtypes = []
            L.oracle_num_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def dims(T, H, d, r_k, r_v, variant=0, rope_base=10000.0, rope_style=0) -> OracleDims:
    return OracleDims(T, H, d, r_k, r_v, variant, float(rope_base), rope_style)


def _d(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _i(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def num_threads() -> int:
    return lib().oracle_num_threads()


def compression_ratio(dm: OracleDims) -> float:
    return lib().oracle_compression_ratio(ctypes.byref(dm))


def teacher_scalars_per_token(dm: OracleDims, D: int) -> int:
    return lib().oracle_teacher_scalars_per_token(ctypes.byref(dm), D)


def latent_scalars_per_token(dm: OracleDims, D: int) -> int:
    return lib().oracle_latent_scalars_per_token(ctypes.byref(dm), D)


def round_bf16(x: float) -> float:
    return lib().oracle_round_bf16(float(x))


def encode(dm: OracleDims, x, seq_idx, pos, w_down, mu, r, cache, round_to_bf16=False):
    """Eq. (2) into ``cache`` (an fp64 numpy array, updated in place)."""
    assert cache.dtype == np.float64 and cache.flags.c_contiguous
    x, xp = _d(x)
    w, wp = _d(w_down)
    m, mp = _d(mu)
    si, sip = _i(seq_idx)
    po, pop = _i(pos)
    N = si.shape[0]
    B = cache.shape[0]
    L_max = cache.shape[2] if dm.variant == 0 else cache.shape[1]
    rc = lib().oracle_encode(ctypes.byref(dm), N, xp, sip, pop, wp, mp, int(r),
                             cache.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                             B, L_max, 1 if round_to_bf16 else 0)
    if rc != 0:
        raise ValueError("oracle_encode failed (%d)" % rc)
    return cache


def decode(dm: OracleDims, t, q, cache_k, cache_v, seq_lens, q_pos, w_up_k, w_up_v,
           mu_k, mu_v, pos_offset=0, want_scores=False, v_mode=0):
    """Decode attention at loop ``t``: returns (out [B][H][d], lse [B][H], scores|None)."""
    q, qp = _d(q)
    ck, ckp = _d(cache_k)
    cv, cvp = _d(cache_v)
    sl, slp = _i(seq_lens)
    qpos, qposp = _i(q_pos)
    wk, wkp = _d(w_up_k)
    wv, wvp = _d(w_up_v)
    mk, mkp = _d(mu_k)
    mv, mvp = _d(mu_v)
    B = q.shape[0]
    L_max = ck.shape[2] if dm.variant == 0 else ck.shape[1]
    out = np.zeros((B, dm.H, dm.d))
    lse = np.zeros((B, dm.H))
    scores = np.full((B, dm.H, L_max), np.nan) if want_scores else None
    sp = scores.ctypes.data_as(ctypes.POINTER(ctypes.c_double)) if want_scores else None
    rc = lib().oracle_decode(ctypes.byref(dm), int(t), B, L_max, qp, ckp, cvp, slp, qposp,
                             int(pos_offset), wkp, wvp, mkp, mvp,
                             out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                             lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), sp, int(v_mode))
    if rc != 0:
        raise ValueError("oracle_decode failed (%d)" % rc)
    return out, lse, scores


def hybrid(dm: OracleDims, t, q, cache_k, cache_v, n_lat, q_pos, w_up_k, w_up_v, mu_k, mu_v,
           k_win, v_win, n_win, win_pos):
    """Eq. (4) of the HLA page at loop ``t``: one softmax over the latent tokens
    j < n_lat[b] and the exact window tokens w < n_win[b] (positions win_pos[b] + w).
    k_win / v_win are [B][H][W][d], keys before RoPE.  Returns (out, lse)."""
    q, qp = _d(q)
    ck, ckp = _d(cache_k)
    cv, cvp = _d(cache_v)
    nl, nlp = _i(n_lat)
    qpos, qposp = _i(q_pos)
    wk, wkp = _d(w_up_k)
    wv, wvp = _d(w_up_v)
    mk, mkp = _d(mu_k)
    mv, mvp = _d(mu_v)
    kw, kwp = _d(k_win)
    vw, vwp = _d(v_win)
    nw, nwp = _i(n_win)
    wpos, wposp = _i(win_pos)
    B, L_max, W = q.shape[0], ck.shape[2], kw.shape[2]
    out = np.zeros((B, dm.H, dm.d))
    lse = np.zeros((B, dm.H))
    rc = lib().oracle_hybrid(ctypes.byref(dm), int(t), B, L_max, W, qp, ckp, cvp, nlp, qposp,
                             wkp, wvp, mkp, mvp, kwp, vwp, nwp, wposp,
                             out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                             lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError("oracle_hybrid failed (%d)" % rc)
    return out, lse


def decoupled(dm: OracleDims, t, q, cache_k, cache_v, k_rope, seq_lens, q_pos, w_up_k, w_up_v, mu_k, mu_v,
              pos_offset=0):
    """Absorbed decoupled-RoPE decode at loop ``t`` (LLA page, Appendix J): q [B][H][d + d_rope],
    k_rope [B][H][L_max][d_rope], the rest as :func:`decode`.  Returns (out, lse)."""
    q, qp = _d(q)
    ck, ckp = _d(cache_k)
    cv, cvp = _d(cache_v)
    kr, krp = _d(k_rope)
    sl, slp = _i(seq_lens)
    qpos, qposp = _i(q_pos)
    wk, wkp = _d(w_up_k)
    wv, wvp = _d(w_up_v)
    mk, mkp = _d(mu_k)
    mv, mvp = _d(mu_v)
    B, L_max, d_rope = q.shape[0], ck.shape[2], kr.shape[3]
    out = np.zeros((B, dm.H, dm.d))
    lse = np.zeros((B, dm.H))
    rc = lib().oracle_decoupled(ctypes.byref(dm), int(t), int(d_rope), B, L_max, qp, ckp, cvp, krp, slp, qposp,
                                int(pos_offset), wkp, wvp, mkp, mvp,
                                out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError("oracle_decoupled failed (%d)" % rc)
    return out, lse


def sdpa(dm: OracleDims, q, k, v, seq_lens, q_pos, pos_offset=0):
    """Uncompressed attention over pre-RoPE K/V [B][H][L_max][d]: (out, lse)."""
    q, qp = _d(q)
    k, kp = _d(k)
    v, vp = _d(v)
    sl, slp = _i(seq_lens)
    qpos, qposp = _i(q_pos)
    B, L_max = q.shape[0], k.shape[2]
    out = np.zeros((B, dm.H, dm.d))
    lse = np.zeros((B, dm.H))
    rc = lib().oracle_sdpa(ctypes.byref(dm), B, L_max, qp, kp, vp, slp, qposp, int(pos_offset),
                           out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                           lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError("oracle_sdpa failed (%d)" % rc)
    return out, lse
