"""Seeded synthetic LLA workloads, shared by the tests, the smoke check and the bench.

This module draws random tensors and converts them to their storage dtype.  It
contains none of the method's arithmetic: no encode, reconstruction, RoPE or
attention.  Both the CUDA path and the oracle consume exactly the tensors made
here (the oracle after an exact widening to fp64).

Recipe (the same for every workload, distributions given as variances):

* cached K latents ~ N(0, 1), V latents ~ N(0, 1)
* W_up,{k,v} ~ N(0, 1/r) with r the rank of that axis
* mu_{k,v} ~ N(0, 0.1)  (the codec mean of Eq. (2); mu_t is its loop-t slice)
* W_down,{k,v} ~ N(0, 1/(T*d))  (LLA-2D: N(0, 1/(T*H*d)))
* x_{k,v} (stacked pre-RoPE loop activations for encode) ~ N(0, 1)
* q ~ N(0, 1)
* seq_lens uniform integers in [len_lo, len_hi]; q_pos = seq_lens - 1

Draw order is fixed (latents K, latents V, W_up,k, W_up,v, mu_k, mu_v, W_down,k,
W_down,v, x_k, x_v, q, seq_lens), each drawn as fp32 standard normals from one
``torch.Generator`` seeded with ``seed`` (on the CPU for small workloads, on the
GPU for the large ones), scaled by the standard deviation in fp32, then rounded
once (round-to-nearest-even) to the storage dtype: bf16 for latents, W and q in
bf16 mode, fp32 for everything in fp32 mode; mu is always fp32.

Workload shapes follow the Ouro-1.4B geometry the paper evaluates (D=24 layers,
H=16 heads, d_head=128, T=4 loops; "Looped Latent Attention", Appendix A
"Models") at the rank pairs of its Table 8 and Table 5.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    d: int
    r_k: int
    r_v: int
    B: int
    L_max: int
    len_lo: int
    len_hi: int
    variant: int = 0          # 0 per-head LLA, 1 LLA-2D
    dtype: str = "bf16"       # storage dtype: "bf16" or "f32"
    rope_base: float = 10000.0
    layers: int = 1           # layers of the synthetic stack (full-step workloads)
    N_encode: int = 0         # tokens written by lla_encode per layer (0: none)


WORKLOADS = {
    # tiny parity case: one sequence, 256 past tokens, fp32 storage
    "tiny_f32": Workload("tiny_f32", T=4, H=2, d=128, r_k=96, r_v=160, B=1, L_max=256,
                         len_lo=256, len_hi=256, dtype="f32"),
    # Ouro-1.4B-shaped single layer, rho = 4, 32 ragged sequences of 3584..4096 tokens
    "ouro1.4b_rho4_b32_4k": Workload("ouro1.4b_rho4_b32_4k", T=4, H=16, d=128, r_k=96,
                                     r_v=160, B=32, L_max=4096, len_lo=3584, len_hi=4096),
    # the same layer with 8 sequences (about 250 MB of latents, still above L2): the
    # small case for kernel profiles
    "ouro1.4b_rho4_b8_4k": Workload("ouro1.4b_rho4_b8_4k", T=4, H=16, d=128, r_k=96,
                                    r_v=160, B=8, L_max=4096, len_lo=3584, len_hi=4096),
    # rho = 21.3 at serving batch: 768 sequences x 4096, 24-layer stack + new-token encode
    "ouro1.4b_rho21_b768_4k": Workload("ouro1.4b_rho21_b768_4k", T=4, H=16, d=128, r_k=16,
                                       r_v=32, B=768, L_max=4096, len_lo=4096, len_hi=4096,
                                       layers=24, N_encode=768),
    # the same layer at 64 sequences (0.4 GB of latents, above L2): the profiling case
    "ouro1.4b_rho21_b64_4k": Workload("ouro1.4b_rho21_b64_4k", T=4, H=16, d=128, r_k=16,
                                      r_v=32, B=64, L_max=4096, len_lo=4096, len_hi=4096,
                                      N_encode=64),
    # long context: 64 sequences x 16384, 48-layer stack, prefill encode of every token
    "ouro_rho4_b64_16k": Workload("ouro_rho4_b64_16k", T=4, H=16, d=128, r_k=96, r_v=160,
                                  B=64, L_max=16384, len_lo=16384, len_hi=16384, layers=48,
                                  N_encode=64 * 16384),
    # the long-context layer with 8 sequences (1.07 GB of latents): the case for kernel
    # profiles at 16k tokens per sequence
    "ouro_rho4_b8_16k": Workload("ouro_rho4_b8_16k", T=4, H=16, d=128, r_k=96, r_v=160,
                                 B=8, L_max=16384, len_lo=16384, len_hi=16384),
    # the long-context prefill at 4 sequences (65,536 tokens x 16 heads, 2.1 GB of x):
    # the case for profiles of the prefill encode
    "ouro_rho4_b4_16k": Workload("ouro_rho4_b4_16k", T=4, H=16, d=128, r_k=96, r_v=160,
                                 B=4, L_max=16384, len_lo=16384, len_hi=16384,
                                 N_encode=4 * 16384),
    # LLA-2D: one latent per token for all heads, r = (128, 256), 256 x 8192
    "lla2d_b256_8k": Workload("lla2d_b256_8k", T=4, H=16, d=128, r_k=128, r_v=256, B=256,
                              L_max=8192, len_lo=8192, len_hi=8192, variant=1),
    # the same with 32 sequences (about 200 MB of latents, still above L2): the small
    # case for kernel profiles
    "lla2d_b32_8k": Workload("lla2d_b32_8k", T=4, H=16, d=128, r_k=128, r_v=256, B=32,
                             L_max=8192, len_lo=8192, len_hi=8192, variant=1),
}


def storage_dtype(w: Workload) -> torch.dtype:
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def _normal(gen: torch.Generator, shape, std: float, dtype: torch.dtype, device) -> torch.Tensor:
    t = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def make_decode_inputs(w: Workload, seed: int, device="cpu", with_encode: bool = False,
                       seq_lens: Optional[torch.Tensor] = None) -> dict:
    """Draw one layer's cache, codec parameters, queries and lengths.

    Layouts (row-major): cache_k [B][H][L_max][r_k] (LLA-2D: [B][L_max][r_k]);
    w_up_k [T][H][d][r_k] (LLA-2D: [T][H*d][r_k]); mu_k [H][T*d] (LLA-2D: [T*H*d]);
    w_down_k [H][T*d][r_k] (LLA-2D: [T*H*d][r_k]); x_k [N][H][T*d] (LLA-2D: [N][T*H*d]);
    q [B][H][d]; seq_lens, q_pos [B] int32.  V tensors likewise with r_v.
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed))
    sd = storage_dtype(w)
    T, H, d, rk, rv, B, L = w.T, w.H, w.d, w.r_k, w.r_v, w.B, w.L_max
    if w.variant == 0:
        ck_shape, cv_shape = (B, H, L, rk), (B, H, L, rv)
        wuk, wuv = (T, H, d, rk), (T, H, d, rv)
        mu_shape = (H, T * d)
        wdk, wdv = (H, T * d, rk), (H, T * d, rv)
        wd_std = 1.0 / math.sqrt(T * d)
        x_shape = lambda N: (N, H, T * d)  # noqa: E731
    else:
        ck_shape, cv_shape = (B, L, rk), (B, L, rv)
        wuk, wuv = (T, H * d, rk), (T, H * d, rv)
        mu_shape = (T * H * d,)
        wdk, wdv = (T * H * d, rk), (T * H * d, rv)
        wd_std = 1.0 / math.sqrt(T * H * d)
        x_shape = lambda N: (N, T * H * d)  # noqa: E731
    out = {}
    out["cache_k"] = _normal(gen, ck_shape, 1.0, sd, dev)
    out["cache_v"] = _normal(gen, cv_shape, 1.0, sd, dev)
    out["w_up_k"] = _normal(gen, wuk, 1.0 / math.sqrt(rk), sd, dev)
    out["w_up_v"] = _normal(gen, wuv, 1.0 / math.sqrt(rv), sd, dev)
    out["mu_k"] = _normal(gen, mu_shape, math.sqrt(0.1), torch.float32, dev)
    out["mu_v"] = _normal(gen, mu_shape, math.sqrt(0.1), torch.float32, dev)
    if with_encode:
        N = w.N_encode if w.N_encode > 0 else B
        out["w_down_k"] = _normal(gen, wdk, wd_std, sd, dev)
        out["w_down_v"] = _normal(gen, wdv, wd_std, sd, dev)
        out["x_k"] = _normal(gen, x_shape(N), 1.0, sd, dev)
        out["x_v"] = _normal(gen, x_shape(N), 1.0, sd, dev)
    out["q"] = _normal(gen, (B, H, d), 1.0, sd, dev)
    if seq_lens is None:
        seq_lens = torch.randint(w.len_lo, w.len_hi + 1, (B,), generator=gen, device=dev,
                                 dtype=torch.int64).to(torch.int32)
    out["seq_lens"] = seq_lens.to(device=dev, dtype=torch.int32)
    out["q_pos"] = (out["seq_lens"] - 1).clamp_min(0).to(torch.int32)
    return out


def make_window_inputs(w: Workload, W: int, seed: int, seq_lens: torch.Tensor, device="cpu",
                       win_len: Optional[torch.Tensor] = None) -> dict:
    """Exact window of the W newest tokens per sequence (the hybrid layout of the HLA
    page's §3.4): k_win / v_win [B][H][W][d] ~ N(0, 1) in the storage dtype (keys
    before RoPE), win_len [B] (default W), win_pos = seq_lens (the window follows the
    latent tokens) and q_pos = the newest window token's position."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed))
    sd = storage_dtype(w)
    B, H, d = w.B, w.H, w.d
    out = {"k_win": _normal(gen, (B, H, W, d), 1.0, sd, dev), "v_win": _normal(gen, (B, H, W, d), 1.0, sd, dev)}
    if win_len is None:
        win_len = torch.full((B,), W, dtype=torch.int32)
    out["win_len"] = win_len.to(device=dev, dtype=torch.int32)
    out["win_pos"] = seq_lens.to(device=dev, dtype=torch.int32).clone()
    last = out["win_pos"] + out["win_len"] - 1
    out["q_pos"] = torch.where(out["win_len"] > 0, last, (out["win_pos"] - 1).clamp_min(0)).to(torch.int32)
    return out


def make_decoupled_inputs(w: Workload, seed: int, device="cpu", d_rope: int = 64) -> dict:
    """The decoupled-RoPE decode's extra inputs: rotary keys k_rope [B][H][L_max][d_rope]
    ~ N(0, 1) and the query [B][H][d + d_rope] ~ N(0, 1), in the storage dtype."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed))
    sd = storage_dtype(w)
    return {"k_rope": _normal(gen, (w.B, w.H, w.L_max, d_rope), 1.0, sd, dev),
            "q": _normal(gen, (w.B, w.H, w.d + d_rope), 1.0, sd, dev)}


def widen(t: torch.Tensor):
    """Exact widening of a stored tensor to a float64 numpy array (for the oracle)."""
    return t.detach().to("cpu").to(torch.float64).numpy()
