"""Thin Python binding of liblla.so (include/lla.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels.  PyTorch is
used for device memory and the current stream; tensors are passed by pointer.
If the library is missing, loading raises — there is no fallback.

Names follow the C ABI: :func:`encode` = ``lla_encode``, :func:`decode_attn` =
``lla_decode_attn``, :func:`workspace_size`, :func:`rope_table`,
:func:`device_status`, :func:`status_string`.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "liblla.so")

(LLA_OK, LLA_ERR_INVALID_ARG, LLA_ERR_UNSUPPORTED, LLA_ERR_CUDA, LLA_ERR_TIMEOUT, LLA_ERR_DEVICE_ARG,
 LLA_ERR_RANGE) = range(7)
LLA_BF16, LLA_F32 = 0, 1
LLA_PER_HEAD, LLA_2D = 0, 1
LLA_ROPE_HALF, LLA_ROPE_INTERLEAVED = 0, 1


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("d_head", ctypes.c_int),
                ("r_k", ctypes.c_int), ("r_v", ctypes.c_int), ("variant", ctypes.c_int),
                ("dtype", ctypes.c_int), ("rope_base", ctypes.c_float), ("rope_style", ctypes.c_int)]


class Cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("B", ctypes.c_int),
                ("L_max", ctypes.c_int64)]


class PagedCache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("B", ctypes.c_int), ("max_pages", ctypes.c_int), ("page_size", ctypes.c_int),
                ("num_pages", ctypes.c_int64)]


class LLAError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s: %s (status %d)" % (what, status_string(status), status))
        self.status = status


_lib = None
_lock = threading.Lock()


def lib():
    """Load liblla.so (raises OSError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(LIB_PATH)
            vp, i32p, fp = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
            pd = ctypes.POINTER(Dims)
            L.lla_encode.argtypes = [pd, vp, vp, ctypes.c_int, i32p, i32p, vp, vp, fp, fp, Cache,
                                     vp, ctypes.c_size_t, vp]
            L.lla_encode.restype = ctypes.c_int
            L.lla_decode_attn.argtypes = [pd, ctypes.c_int, vp, Cache, i32p, i32p, vp, vp, fp, fp,
                                          fp, fp, ctypes.c_int64, fp, fp, vp, ctypes.c_size_t, vp]
            L.lla_decode_attn.restype = ctypes.c_int
            L.lla_workspace_size.argtypes = [pd, ctypes.c_int, ctypes.c_int64, ctypes.c_int]
            L.lla_workspace_size.restype = ctypes.c_size_t
            L.lla_rope_table.argtypes = [pd, ctypes.c_int64, fp, fp]
            L.lla_rope_table.restype = ctypes.c_int
            L.lla_device_status.argtypes = [vp, vp, ctypes.c_int]
            L.lla_device_status.restype = ctypes.c_int
            L.lla_status_string.argtypes = [ctypes.c_int]
            L.lla_status_string.restype = ctypes.c_char_p
            L.lla_window_attn.argtypes = [pd, ctypes.c_int, ctypes.c_int, vp, vp, vp, i32p, i32p, i32p,
                                          fp, fp, ctypes.c_int64, fp, fp, vp, ctypes.c_size_t, vp]
            L.lla_window_attn.restype = ctypes.c_int
            L.lla_decoupled_workspace_size.argtypes = [pd, ctypes.c_int, ctypes.c_int, ctypes.c_int64]
            L.lla_decoupled_workspace_size.restype = ctypes.c_size_t
            L.lla_decode_attn_decoupled.argtypes = [pd, ctypes.c_int, ctypes.c_int, vp, Cache, vp, i32p, i32p, vp, vp,
                                                    fp, fp, fp, fp, ctypes.c_int64, fp, fp, vp, ctypes.c_size_t, vp]
            L.lla_decode_attn_decoupled.restype = ctypes.c_int
            L.lla_encode_paged.argtypes = [pd, vp, vp, ctypes.c_int, i32p, i32p, vp, vp, fp, fp, PagedCache,
                                           vp, ctypes.c_size_t, vp]
            L.lla_encode_paged.restype = ctypes.c_int
            L.lla_decode_attn_paged.argtypes = [pd, ctypes.c_int, vp, PagedCache, i32p, i32p, vp, vp, fp, fp,
                                                fp, fp, ctypes.c_int64, fp, fp, vp, ctypes.c_size_t, vp]
            L.lla_decode_attn_paged.restype = ctypes.c_int
            L.lla_decode_attn_noalloc.argtypes = [pd, ctypes.c_int, vp, Cache, i32p, i32p, vp, vp, fp, fp,
                                                  fp, fp, ctypes.c_int64, fp, fp, vp]
            L.lla_decode_attn_noalloc.restype = ctypes.c_int
            L.lla_evict_window.argtypes = [pd, Cache, i32p, ctypes.c_int, ctypes.c_int, vp, ctypes.c_size_t, vp]
            L.lla_evict_window.restype = ctypes.c_int
            L.lla_decode_kernel.argtypes = [pd]
            L.lla_decode_kernel.restype = ctypes.c_char_p
            L.lla_decoupled_kernel.argtypes = [pd, ctypes.c_int]
            L.lla_decoupled_kernel.restype = ctypes.c_char_p
            L.lla_abi_version.argtypes = []
            L.lla_abi_version.restype = ctypes.c_int
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().lla_status_string(int(status)).decode()


def decode_kernel(dm: Dims) -> Optional[str]:
    """Kernel family lla_decode_attn runs for these dims ("tile", "small-rank",
    "pair-2d", "fp32"), or None if they are invalid or unsupported."""
    r = lib().lla_decode_kernel(ctypes.byref(dm))
    return None if r is None else r.decode()


def decoupled_kernel(dm: Dims, d_rope: int = 64) -> Optional[str]:
    """Kernel family lla_decode_attn_decoupled runs for these dims ("small-rank",
    "tile", "fp32"), or None if they are invalid or unsupported."""
    r = lib().lla_decoupled_kernel(ctypes.byref(dm), int(d_rope))
    return None if r is None else r.decode()


def dims(T, H, r_k, r_v, d_head=128, variant=LLA_PER_HEAD, dtype=LLA_BF16, rope_base=10000.0,
         rope_style=LLA_ROPE_HALF) -> Dims:
    return Dims(T, H, d_head, r_k, r_v, variant, dtype, float(rope_base), rope_style)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to liblla must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, what: str):
    if status != LLA_OK:
        raise LLAError(status, what)


def workspace_size(dm: Dims, B: int, L_max: int, max_N: int = 0) -> int:
    n = lib().lla_workspace_size(ctypes.byref(dm), int(B), int(L_max), int(max_N))
    if n == 0:
        raise LLAError(LLA_ERR_INVALID_ARG, "lla_workspace_size")
    return n


def make_workspace(dm: Dims, B: int, L_max: int, max_N: int = 0, device="cuda") -> torch.Tensor:
    """A zero-filled workspace buffer of the required size (status word cleared)."""
    return torch.zeros(workspace_size(dm, B, L_max, max_N), dtype=torch.uint8, device=device)


def rope_table(dm: Dims, n_pos: int):
    """(cos, sin) fp32 CPU tensors [n_pos][d/2] from lla_rope_table (fp64 on the host)."""
    c = torch.empty((int(n_pos), dm.d_head // 2), dtype=torch.float32)
    s = torch.empty_like(c)
    _check(lib().lla_rope_table(ctypes.byref(dm), int(n_pos), _ptr(c), _ptr(s)), "lla_rope_table")
    return c, s


def encode(dm: Dims, x_k, x_v, seq_idx, pos, w_down_k, w_down_v, mu_k, mu_v, cache_k, cache_v,
           workspace, stream=None):
    """lla_encode: latents of N tokens into cache slots (seq_idx[n], pos[n])."""
    N = int(seq_idx.shape[0])
    B = int(cache_k.shape[0])
    L_max = int(cache_k.shape[2] if dm.variant == LLA_PER_HEAD else cache_k.shape[1])
    cache = Cache(ctypes.c_void_p(cache_k.data_ptr()), ctypes.c_void_p(cache_v.data_ptr()), B, L_max)
    st = lib().lla_encode(ctypes.byref(dm), _ptr(x_k), _ptr(x_v), N, _ptr(seq_idx), _ptr(pos),
                          _ptr(w_down_k), _ptr(w_down_v), _ptr(mu_k), _ptr(mu_v), cache,
                          _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "lla_encode")


def decode_attn(dm: Dims, loop_t: int, q, cache_k, cache_v, seq_lens, q_pos, w_up_k, w_up_v,
                mu_k, mu_v, rope_cos, rope_sin, out, lse, workspace, stream=None):
    """lla_decode_attn: one layer, loop ``loop_t``, all heads and sequences, into out / lse."""
    B = int(cache_k.shape[0])
    L_max = int(cache_k.shape[2] if dm.variant == LLA_PER_HEAD else cache_k.shape[1])
    cache = Cache(ctypes.c_void_p(cache_k.data_ptr()), ctypes.c_void_p(cache_v.data_ptr()), B, L_max)
    st = lib().lla_decode_attn(ctypes.byref(dm), int(loop_t), _ptr(q), cache, _ptr(seq_lens),
                               _ptr(q_pos), _ptr(w_up_k), _ptr(w_up_v), _ptr(mu_k), _ptr(mu_v),
                               _ptr(rope_cos), _ptr(rope_sin), int(rope_cos.shape[0]), _ptr(out),
                               _ptr(lse), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "lla_decode_attn")


def paged_cache(pool_k, pool_v, block_table, page_size: int) -> PagedCache:
    """The lla_paged_cache of pools [num_pages][H][page_size][r] and a block table
    [B][max_pages] (int32, device)."""
    B, max_pages = int(block_table.shape[0]), int(block_table.shape[1])
    return PagedCache(ctypes.c_void_p(pool_k.data_ptr()), ctypes.c_void_p(pool_v.data_ptr()),
                      ctypes.c_void_p(block_table.data_ptr()), B, max_pages, int(page_size),
                      int(pool_k.shape[0]))


def encode_paged(dm: Dims, x_k, x_v, seq_idx, pos, w_down_k, w_down_v, mu_k, mu_v, pool_k, pool_v,
                 block_table, page_size: int, workspace, stream=None):
    """lla_encode_paged: latents of N tokens into paged slots (seq_idx[n], pos[n])."""
    N = int(seq_idx.shape[0])
    st = lib().lla_encode_paged(ctypes.byref(dm), _ptr(x_k), _ptr(x_v), N, _ptr(seq_idx), _ptr(pos),
                                _ptr(w_down_k), _ptr(w_down_v), _ptr(mu_k), _ptr(mu_v),
                                paged_cache(pool_k, pool_v, block_table, page_size),
                                _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "lla_encode_paged")


def decode_attn_paged(dm: Dims, loop_t: int, q, pool_k, pool_v, block_table, page_size: int, seq_lens,
                      q_pos, w_up_k, w_up_v, mu_k, mu_v, rope_cos, rope_sin, out, lse, workspace,
                      stream=None):
    """lla_decode_attn_paged: lla_decode_attn over a paged cache (pools [num_pages][H][page_size][r],
    block table [B][max_pages])."""
    st = lib().lla_decode_attn_paged(ctypes.byref(dm), int(loop_t), _ptr(q),
                                     paged_cache(pool_k, pool_v, block_table, page_size), _ptr(seq_lens),
                                     _ptr(q_pos), _ptr(w_up_k), _ptr(w_up_v), _ptr(mu_k), _ptr(mu_v),
                                     _ptr(rope_cos), _ptr(rope_sin), int(rope_cos.shape[0]), _ptr(out),
                                     _ptr(lse), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "lla_decode_attn_paged")


def evict_window(dm: Dims, cache_k, cache_v, seq_lens, sink: int, window: int, workspace, stream=None):
    """lla_evict_window: keep each sequence's `sink` first and `window` newest latents
    (moved in order to slots sink..), rewriting seq_lens in place."""
    B = int(cache_k.shape[0])
    L_max = int(cache_k.shape[2] if dm.variant == LLA_PER_HEAD else cache_k.shape[1])
    cache = Cache(ctypes.c_void_p(cache_k.data_ptr()), ctypes.c_void_p(cache_v.data_ptr()), B, L_max)
    st = lib().lla_evict_window(ctypes.byref(dm), cache, _ptr(seq_lens), int(sink), int(window), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "lla_evict_window")


def window_attn(dm: Dims, q, k_win, v_win, win_len, win_pos, q_pos, rope_cos, rope_sin, out, lse,
                workspace, stream=None):
    """lla_window_attn: exact attention over each sequence's window of recent tokens
    (k_win / v_win [B][H][W][d], keys before RoPE, token w at position win_pos[b] + w),
    merged in place into ``out`` / ``lse`` holding lla_decode_attn's latent result."""
    B, W = int(k_win.shape[0]), int(k_win.shape[2])
    st = lib().lla_window_attn(ctypes.byref(dm), B, W, _ptr(q), _ptr(k_win), _ptr(v_win), _ptr(win_len),
                               _ptr(win_pos), _ptr(q_pos), _ptr(rope_cos), _ptr(rope_sin),
                               int(rope_cos.shape[0]), _ptr(out), _ptr(lse), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "lla_window_attn")


def decoupled_workspace(dm: Dims, d_rope: int, B: int, L_max: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace for lla_decode_attn_decoupled."""
    n = lib().lla_decoupled_workspace_size(ctypes.byref(dm), int(d_rope), int(B), int(L_max))
    if n == 0:
        raise LLAError(LLA_ERR_INVALID_ARG, "lla_decoupled_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def decode_attn_decoupled(dm: Dims, loop_t: int, q, cache_k, cache_v, k_rope, seq_lens, q_pos, w_up_k,
                          w_up_v, mu_k, mu_v, rope_cos, rope_sin, out, lse, workspace, stream=None):
    """lla_decode_attn_decoupled: absorbed decoupled-RoPE decode (content on the latents,
    a d_rope = k_rope.shape[3] rotary branch); q is [B][H][d + d_rope]."""
    B, L_max = int(cache_k.shape[0]), int(cache_k.shape[2])
    cache = Cache(ctypes.c_void_p(cache_k.data_ptr()), ctypes.c_void_p(cache_v.data_ptr()), B, L_max)
    st = lib().lla_decode_attn_decoupled(ctypes.byref(dm), int(loop_t), int(k_rope.shape[3]), _ptr(q), cache,
                                         _ptr(k_rope), _ptr(seq_lens), _ptr(q_pos), _ptr(w_up_k), _ptr(w_up_v),
                                         _ptr(mu_k), _ptr(mu_v), _ptr(rope_cos), _ptr(rope_sin),
                                         int(rope_cos.shape[0]), _ptr(out), _ptr(lse), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "lla_decode_attn_decoupled")


def device_status(workspace, stream=None, clear=True) -> int:
    """Synchronise and read (then clear) the kernels' status word in ``workspace``."""
    return int(lib().lla_device_status(_ptr(workspace), _stream(stream), 1 if clear else 0))


class Decoder:
    """Convenience holder of one layer's codec parameters and a RoPE table on the device.

    ``__call__`` runs ``lla_decode_attn`` for loop t and returns (out, lse).
    """

    def __init__(self, dm: Dims, w_up_k, w_up_v, mu_k, mu_v, B: int, L_max: int, device="cuda"):
        self.dm = dm
        self.w_up_k, self.w_up_v, self.mu_k, self.mu_v = w_up_k, w_up_v, mu_k, mu_v
        n = max(int(L_max), 128)
        c, s = rope_table(dm, n)
        self.rope_cos, self.rope_sin = c.to(device), s.to(device)
        self.workspace = make_workspace(dm, B, L_max, device=device)

    def __call__(self, loop_t, q, cache_k, cache_v, seq_lens, q_pos, out=None, lse=None, stream=None):
        B, H = q.shape[0], q.shape[1]
        if out is None:
            out = torch.empty((B, H, self.dm.d_head), dtype=torch.float32, device=q.device)
        if lse is None:
            lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
        decode_attn(self.dm, loop_t, q, cache_k, cache_v, seq_lens, q_pos, self.w_up_k,
                    self.w_up_v, self.mu_k, self.mu_v, self.rope_cos, self.rope_sin, out, lse,
                    self.workspace, stream)
        return out, lse


def decode_attn_noalloc(dm: Dims, loop_t: int, q, cache_k, cache_v, seq_lens, q_pos, w_up_k,
                        w_up_v, mu_k, mu_v, rope_cos, rope_sin, out, lse, stream=None):
    """lla_decode_attn_noalloc: lla_decode_attn with the library's fixed device scratch
    instead of a caller workspace, for callers that cannot allocate device memory.
    Calls that overlap on the GPU race on that scratch; make the first call on a
    device before any stream capture."""
    f = lib().lla_decode_attn_noalloc
    B = int(cache_k.shape[0])
    L_max = int(cache_k.shape[2] if dm.variant == LLA_PER_HEAD else cache_k.shape[1])
    cache = Cache(ctypes.c_void_p(cache_k.data_ptr()), ctypes.c_void_p(cache_v.data_ptr()), B, L_max)
    st = f(ctypes.byref(dm), int(loop_t), _ptr(q), cache, _ptr(seq_lens), _ptr(q_pos), _ptr(w_up_k),
           _ptr(w_up_v), _ptr(mu_k), _ptr(mu_v), _ptr(rope_cos), _ptr(rope_sin),
           int(rope_cos.shape[0]), _ptr(out), _ptr(lse), _stream(stream))
    _check(st, "lla_decode_attn_noalloc")
