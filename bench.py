"""Benchmark of the LLA latent-store decode hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one decode step of one layer of the workload: ``lla_encode`` of each
sequence's new token (its T-loop K/V stack) followed by ``lla_decode_attn`` for
loops t = 1..T over all heads and sequences.  The metric is decode-attention
latent-KV tokens per second per layer-loop: sum_b seq_lens[b] * T / step time.

Rank 0 prints one JSON line.  With N>1 (torchrun, one rank per GPU) every rank
runs its own sequences (the path shards by sequence with no exchange: weak
scaling) and the time is the max over ranks.  ``--impl reference`` times the
oracle (plain fp64 C on the host cores) on a bounded sample of the same
workload instead.
"""
from __future__ import annotations

import argparse
import dataclasses
import datetime
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from looped_transformer_cross_gb300 import build as lla_build  # noqa: E402
from looped_transformer_cross_gb300 import lla  # noqa: E402
from looped_transformer_cross_gb300.synth import (WORKLOADS, make_decode_inputs,  # noqa: E402
                                                  make_decoupled_inputs, make_window_inputs, widen)

METRIC = "decode-attn latent-KV tokens/s per layer-loop; % HBM or tensor-pipe roofline"

# DRAM bytes (read + write) of decode_bf16_kernel per latent token-head, from one ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum) each of the 8-sequence
# variants of the 4k-context bench layer (ouro1.4b_rho4_b8_4k) and of the long-context
# layer (ouro_rho4_b8_16k); a workload takes the capture of its context length.
# Valid only for the decode source whose sha256 starts with TRAFFIC_SRC_SHA; any other
# source reports traffic as unknown (null).
TRAFFIC_PER_TOKEN_HEAD = {4096: (263.988736e6 + 3.217408e6) / (31042 * 16),
                          16384: (1080.879104e6 + 3.529472e6) / (8 * 16384 * 16)}
TRAFFIC_SRC_SHA = "2b90f83646e16cdd"
DECODE_SRC = os.path.join(ROOT, "looped_transformer_cross_gb300", "csrc", "lla_decode.cu")
# The same for the LLA-2D score kernel (the dominant one of the LLA-2D call), per
# latent token (all heads), from the 32-sequence variant of the LLA-2D layer; valid
# only for the source whose sha256 starts with TRAFFIC2D_SRC_SHA.
TRAFFIC2D_PER_TOKEN = (90.234624e6 + 4.024320e6) / (32 * 8192)
TRAFFIC2D_SRC_SHA = "7100f488412d4d9a"
DECODE2D_SRC = os.path.join(ROOT, "looped_transformer_cross_gb300", "csrc", "lla_decode2d.cu")
# Same for decode_small_kernel (the per-head kernel at small ranks), from a capture
# of the 64-sequence variant of the rho = 21.3 layer (ouro1.4b_rho21_b64_4k).
TRAFFIC_SMALL_PER_TOKEN_HEAD = (412.849152e6 + 3.808256e6) / (64 * 4096 * 16)
TRAFFIC_SMALL_SRC_SHA = "d9a74db4c583c522"
DECODE_SMALL_SRC = os.path.join(ROOT, "looped_transformer_cross_gb300", "csrc", "lla_decode_small.cu")
# Same for decoupled_tile_kernel (the tensor-core decoupled kernel at larger ranks),
# from the 8-sequence variant of the rho = 4 layer (ouro1.4b_rho4_b8_4k).
TRAFFIC_DEC_TILE_PER_TOKEN_HEAD = (326.490112e6 + 3.213824e6) / (31042 * 16)
TRAFFIC_DEC_TILE_SRC_SHA = "682bdfb06f9c87d1"
# Same for decoupled_small_kernel (small ranks, rotary branch on the tensor cores),
# from the 64-sequence variant of the rho = 21.3 layer (ouro1.4b_rho21_b64_4k).
TRAFFIC_DEC_SMALL_PER_TOKEN_HEAD = (945.438720e6 + 2.848000e6) / (64 * 4096 * 16)
TRAFFIC_DEC_SMALL_SRC_SHA = "682bdfb06f9c87d1"
DECOUPLED_SMALL_SRC = os.path.join(ROOT, "looped_transformer_cross_gb300", "csrc", "lla_decoupled_tc.cu")
# DRAM bytes of encode_pair_kernel per prefill token (all heads, both axes), from one
# ncu capture of the 4-sequence prefill (ouro_rho4_b4_16k: 65,536 tokens); valid only
# for the encode source whose sha256 starts with TRAFFIC_ENC_SRC_SHA.
TRAFFIC_ENC_PER_TOKEN = (2198.692352e6 + 481.901568e6) / 65536
TRAFFIC_ENC_SRC_SHA = "34fa9d1b5ce18a15"
ENCODE_SRC = os.path.join(ROOT, "looped_transformer_cross_gb300", "csrc", "lla_encode.cu")
UNIT = "latent tokens/s per layer-loop"
DEFAULT_WORKLOAD = "ouro1.4b_rho4_b32_4k"
D_ROPE = 64   # rotary dimensions of the decoupled-RoPE decode


def peaks():
    """(HBM GB/s, bf16 TFLOP/s sustained, source).  The bf16 figure is the one measured
    over a seconds-long GEMM loop under the power cap: the decode calls run back to
    back for the whole timed region."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return (float(d["hbm_gbs"]), float(d.get("bf16_tflops_sustained", d.get("bf16_tflops", 1700.0))),
                "measured")
    return 6800.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms while active, each
    sample stamped with the host clock on arrival; ``summary(t0, t1)`` keeps the
    samples taken between t0 and t1."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def wait_live(self, timeout_s=3.0):
        """Wait (bounded) for the first sample, so the sampler runs before the work."""
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and time.perf_counter() - t0 < timeout_s:
            time.sleep(0.01)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        window = "timed region"
        pick = [ln for ts, ln in self.lines if (t0 is None or ts >= t0) and (t1 is None or ts <= t1)]
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in pick:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax = max(smax, float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax or None,
                "reasons": sorted(reasons), "samples": len(sm), "window": window}


# ----------------------------------------------------------------- our arm

class DecodeStep:
    """The layers' state on the device and the per-step call sequence: for each of
    ``layers`` layers, lla_encode of the sequences' new token and lla_decode_attn for
    loops 1..T.  Layer l reads layer buffer l mod nbuf, where nbuf is the number of
    distinct layer caches that fit in device memory (a stack larger than HBM cycles
    its buffers); every layer has its own queries and outputs.  With a window W > 0
    (one layer) each decode call is followed by lla_window_attn over an exact window
    of the W newest tokens (the HLA page's hybrid layout, §3.4 Eq. (4)) placed after
    the latent tokens."""

    def __init__(self, w, seed, device, window=0, decoupled=False, paged=0, layers=1, prefill=False):
        if layers > 1 and (window or decoupled or paged):
            raise ValueError("a multi-layer step runs the dense per-layer decode only")
        self.nlayers = layers
        self.w = w
        self.window = window
        self.decoupled = decoupled
        self.paged = paged
        # the prefill stack (x for every cached position) is drawn only when the prefill
        # leg will encode it; otherwise the new-token rows alone
        wd = w if prefill else dataclasses.replace(w, N_encode=min(w.N_encode, w.B))
        self.inp = make_decode_inputs(wd, seed, device=device, with_encode=True)
        # a workload with a prefill stack (x for every cached position) keeps it aside:
        # the decode step encodes only each sequence's new token, the first B rows
        self.prefill_x = None
        if self.inp["x_k"].shape[0] > w.B:
            self.prefill_x = (self.inp["x_k"], self.inp["x_v"])
            self.inp["x_k"], self.inp["x_v"] = self.inp["x_k"][:w.B], self.inp["x_v"][:w.B]
        if window > 0:
            self.win = make_window_inputs(w, window, seed + 5, self.inp["seq_lens"], device=device)
            self.inp["q_pos"] = self.win["q_pos"]
        g = torch.Generator(device=device)
        g.manual_seed(seed + 7)
        # one query per layer and loop (the model's query changes from loop to loop)
        self.qL = (torch.randn((layers, w.T, w.B, w.H, w.d), generator=g, device=device)
                   .to(self.inp["q"].dtype).contiguous())
        self.q = self.qL[0]
        # further layer buffers: each its own cache, codec and new-token stacks, drawn
        # with its own seed, the lengths shared; as many as fit in device memory
        self.bufs = [self.inp]
        if layers > 1:
            per_layer = sum(self.inp[k].numel() * self.inp[k].element_size() for k in ("cache_k", "cache_v"))
            free = torch.cuda.mem_get_info(device)[0]
            nbuf = int(min(layers, max(1, (free - 8e9 - per_layer) // per_layer)))
            wl = dataclasses.replace(w, N_encode=0)   # new-token rows only
            for l in range(1, nbuf):
                li = make_decode_inputs(wl, seed + 100 * l, device=device, with_encode=True,
                                        seq_lens=self.inp["seq_lens"])
                li["seq_lens"], li["q_pos"] = self.inp["seq_lens"], self.inp["q_pos"]
                del li["q"]
                self.bufs.append(li)
        self.dm = lla.dims(w.T, w.H, w.r_k, w.r_v, variant=w.variant, rope_base=w.rope_base)
        c, s = lla.rope_table(self.dm, max(w.L_max + window, 128))
        self.cos, self.sin = c.to(device), s.to(device)
        self.ws = lla.make_workspace(self.dm, w.B, w.L_max, w.B, device=device)
        self.seq_idx = torch.arange(w.B, dtype=torch.int32, device=device)
        self.outL = torch.empty((layers, w.T, w.B, w.H, w.d), dtype=torch.float32, device=device)
        self.lseL = torch.empty((layers, w.T, w.B, w.H), dtype=torch.float32, device=device)
        self.out, self.lse = self.outL[0], self.lseL[0]
        self.tokens = int(self.inp["seq_lens"].sum().item())
        self.enc_pos = (self.inp["seq_lens"] - 1).clamp(0, w.L_max - 1).to(torch.int32)
        if paged:
            # page pools [num_pages][H][P][r] with a shuffled page table (the page tables
            # of "Enabling dynamic computation in Looped LMs", App. A.1); the dense cache
            # rows are moved into them and the dense cache is dropped
            P = paged
            lens = self.inp["seq_lens"].cpu().tolist()
            max_pages = (w.L_max + P - 1) // P
            used = [(L + P - 1) // P for L in lens]
            num_pages = sum(used)
            perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed + 11))
            bt = torch.full((w.B, max_pages), -1, dtype=torch.int32)
            k = 0
            for b, u in enumerate(used):
                bt[b, :u] = perm[k:k + u].to(torch.int32)
                k += u
            self.block_table = bt.to(device)
            for n, pn in (("cache_k", "pool_k"), ("cache_v", "pool_v")):
                dense = self.inp[n]
                pool = torch.empty((num_pages, w.H, P, dense.shape[-1]), dtype=dense.dtype, device=device)
                for b, u in enumerate(used):
                    for lp in range(u):
                        rows = dense[b, :, lp * P:(lp + 1) * P]
                        pool[int(bt[b, lp]), :, :rows.shape[1]] = rows
                setattr(self, pn, pool)
                self.inp[n] = None
            del dense
            torch.cuda.empty_cache()
            self.ws = lla.make_workspace(self.dm, w.B, max_pages * P, w.B, device=device)
        if decoupled:
            # absorbed decoupled-RoPE decode (LLA Appendix J): rotary keys of d_rope = 64
            # per (token, head) beside the latents, queries [B][H][d + 64]
            self.k_rope = make_decoupled_inputs(w, seed + 9, device=device)["k_rope"]
            self.q = (torch.randn((w.T, w.B, w.H, w.d + D_ROPE), generator=g, device=device)
                      .to(self.inp["q"].dtype).contiguous())
            rdm = lla.dims(w.T, w.H, w.r_k, w.r_v, d_head=D_ROPE, rope_base=w.rope_base)
            c, s = lla.rope_table(rdm, max(w.L_max, 128))
            self.cos_r, self.sin_r = c.to(device), s.to(device)
            self.dws = lla.decoupled_workspace(self.dm, D_ROPE, w.B, w.L_max, device=device)

    def run(self, ev=None, group=False):
        """One step.  ``ev``: events [start][end][window end] per decode call; with
        ``group`` only the start of the first and the end of the last decode call of
        each layer are recorded (no event between consecutive calls)."""
        if self.nlayers > 1:
            return self.run_layers(ev, group)
        i, dm = self.inp, self.dm
        # the new token's latent: slot seq_lens - 1 (the query's own slot without a window)
        if self.paged:
            lla.encode_paged(dm, i["x_k"], i["x_v"], self.seq_idx, self.enc_pos, i["w_down_k"], i["w_down_v"],
                             i["mu_k"], i["mu_v"], self.pool_k, self.pool_v, self.block_table, self.paged, self.ws)
        else:
            lla.encode(dm, i["x_k"], i["x_v"], self.seq_idx, self.enc_pos, i["w_down_k"], i["w_down_v"],
                       i["mu_k"], i["mu_v"], i["cache_k"], i["cache_v"], self.ws)
        for t in range(self.w.T):
            if ev is not None and (not group or t == 0):
                ev[0][t].record()
            if self.paged:
                lla.decode_attn_paged(dm, t, self.q[t], self.pool_k, self.pool_v, self.block_table, self.paged,
                                      i["seq_lens"], i["q_pos"], i["w_up_k"], i["w_up_v"], i["mu_k"], i["mu_v"],
                                      self.cos, self.sin, self.out[t], self.lse[t], self.ws)
            elif self.decoupled:
                lla.decode_attn_decoupled(dm, t, self.q[t], i["cache_k"], i["cache_v"], self.k_rope,
                                          i["seq_lens"], i["q_pos"], i["w_up_k"], i["w_up_v"], i["mu_k"],
                                          i["mu_v"], self.cos_r, self.sin_r, self.out[t], self.lse[t], self.dws)
            else:
                lla.decode_attn(dm, t, self.q[t], i["cache_k"], i["cache_v"], i["seq_lens"], i["q_pos"],
                                i["w_up_k"], i["w_up_v"], i["mu_k"], i["mu_v"], self.cos, self.sin,
                                self.out[t], self.lse[t], self.ws)
            if ev is not None and (not group or t == self.w.T - 1):
                ev[1][t].record()
            if self.window > 0:
                v = self.win
                lla.window_attn(dm, self.q[t], v["k_win"], v["v_win"], v["win_len"], v["win_pos"],
                                i["q_pos"], self.cos, self.sin, self.out[t], self.lse[t], self.ws)
                if ev is not None:
                    ev[2][t].record()

    def run_layers(self, ev=None, group=False):
        dm, T = self.dm, self.w.T
        for l in range(self.nlayers):
            i = self.bufs[l % len(self.bufs)]
            lla.encode(dm, i["x_k"], i["x_v"], self.seq_idx, self.enc_pos, i["w_down_k"], i["w_down_v"],
                       i["mu_k"], i["mu_v"], i["cache_k"], i["cache_v"], self.ws)
            for t in range(T):
                if ev is not None and (not group or t == 0):
                    ev[0][l * T + t].record()
                lla.decode_attn(dm, t, self.qL[l, t], i["cache_k"], i["cache_v"], i["seq_lens"], i["q_pos"],
                                i["w_up_k"], i["w_up_v"], i["mu_k"], i["mu_v"], self.cos, self.sin,
                                self.outL[l, t], self.lseL[l, t], self.ws)
                if ev is not None and (not group or t == T - 1):
                    ev[1][l * T + t].record()

    def dense_view(self, nseq):
        """(cache_k, cache_v) of the first nseq sequences as dense [nseq][H][L_max][r]
        tensors (gathered from the pages when the cache is paged)."""
        if not self.paged:
            return self.inp["cache_k"][:nseq], self.inp["cache_v"][:nseq]
        P, w = self.paged, self.w
        out = []
        for pool in (self.pool_k, self.pool_v):
            d = torch.zeros((nseq, w.H, w.L_max, pool.shape[-1]), dtype=pool.dtype, device=pool.device)
            bt = self.block_table.cpu()
            for b in range(nseq):
                for lp in range(bt.shape[1]):
                    if int(bt[b, lp]) >= 0:
                        n = min(P, w.L_max - lp * P)
                        d[b, :, lp * P:lp * P + n] = pool[int(bt[b, lp]), :, :n]
            out.append(d)
        return out[0], out[1]

    # launches of this library's kernels per step: encode (bias + GEMM) + T x (query
    # images + decode + combine [+ window]); decoupled: query records + decode + combine
    def gathers_rows(self):
        """True when the paged decode runs the row-gathering kernel (tile-kernel shapes
        in pages that are neither a multiple of 128 tokens nor 8, 16, 32 or 64)."""
        P = self.paged
        return bool(P) and lla.decode_kernel(self.dm) == "tile" and not (P % 128 == 0 or (P % 8 == 0 and 128 % P == 0))

    def launches(self):
        """Library kernel launches per step: the encode's two, then per decode call its
        family's (row gather 1; fp32 and plain LLA-2D 2; tile, small-rank and decoupled
        3: images, decode, combine; LLA-2D on CTA pairs 4: images, score, value,
        combine) and the window call's one."""
        fam = lla.decode_kernel(self.dm)
        if self.gathers_rows():
            per = 1
        elif self.decoupled:
            per = 2 if lla.decoupled_kernel(self.dm, D_ROPE) == "fp32" else 3
        elif fam == "pair-2d":
            per = 4
        elif fam in ("fp32", "plain-2d"):
            per = 2
        else:
            per = 3
        return (2 + (per + (1 if self.window > 0 else 0)) * self.w.T) * self.nlayers


# A rank that dies or never joins must not hold the others forever: every collective of
# the bench (the barriers around the timed region, the max of the elapsed time, the sum of
# the tokens) ends with an error after this many seconds.
PG_TIMEOUT_S = float(os.environ.get("LLA_BENCH_PG_TIMEOUT_S", "600"))


def init_dist(backend, device=None, timeout_s=None):
    """One process group over the launcher's env (RANK, WORLD_SIZE, MASTER_*), with a
    bounded timeout on every collective."""
    kw = {"timeout": datetime.timedelta(seconds=PG_TIMEOUT_S if timeout_s is None else timeout_s)}
    if device is not None:
        kw["device_id"] = device
    torch.distributed.init_process_group(backend, **kw)


def barrier(dist_on):
    if dist_on:
        torch.distributed.barrier()


def max_over_ranks(x, dist_on, device):
    if not dist_on:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, dist_on, device):
    if not dist_on:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def prefill_run(step: DecodeStep, reps: int, hbm: float, src: str):
    """lla_encode of the workload's whole prefill stack: every cached position of every
    sequence, one [tokens x T*d] . [T*d x r] product per head and axis (Eq. (2) of the
    LLA page), written into a second cache so the decode layer stays as it was.  Each
    call is timed with CUDA events on the launching stream; x (tens of GB) is far larger
    than L2.  Algorithmic bytes: x_k and x_v read once, every latent written once
    (W_down and mu, under 1 MB, left out)."""
    w, i = step.w, step.inp
    xk, xv = step.prefill_x
    dev = xk.device
    seq_idx = torch.arange(w.B, dtype=torch.int32, device=dev).repeat_interleave(w.L_max)
    pos = torch.arange(w.L_max, dtype=torch.int32, device=dev).repeat(w.B)
    pk, pv = torch.empty_like(i["cache_k"]), torch.empty_like(i["cache_v"])
    n = int(seq_idx.shape[0])
    moved = ((xk.numel() + xv.numel()) * xk.element_size() + (pk.numel() + pv.numel()) * pk.element_size())
    flops = 2.0 * xk.numel() * (w.r_k + w.r_v)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for k in range(reps + 2):
        e0.record()
        lla.encode(step.dm, xk, xv, seq_idx, pos, i["w_down_k"], i["w_down_v"], i["mu_k"], i["mu_v"],
                   pk, pv, step.ws)
        e1.record()
        torch.cuda.synchronize()
        if k >= 2:
            times.append(e0.elapsed_time(e1) / 1e3)
    if lla.device_status(step.ws) != lla.LLA_OK:
        raise RuntimeError("device status after the prefill encode")
    t = float(np.mean(times))
    del pk, pv
    import hashlib
    with open(ENCODE_SRC, "rb") as f:
        same_src = hashlib.sha256(f.read()).hexdigest().startswith(TRAFFIC_ENC_SRC_SHA)
    traffic = TRAFFIC_ENC_PER_TOKEN * n if same_src else None
    return {"tokens": n, "heads": w.H if w.variant == 0 else 1, "encode_ms": t * 1e3,
            "value": n / t, "unit": "prefill tokens/s per layer", "tflops": flops / t / 1e12,
            "roofline": {"bound": "hbm", "achieved": moved / t / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": moved / t / 1e9 / hbm, "traffic": traffic, "traffic_kernel": "encode_pair_kernel",
                         "kernel": "lla_encode (encode_bias_kernel + encode_pair_kernel)",
                         "algorithmic_bytes_per_launch": moved, "peak_source": src}}


def arm_config(w, args, tokens, world, layers=1):
    """The bench line's ``config``: the same object on both arms."""
    return {"workload": w.name, "variant": "LLA-2D" if w.variant else "per-head",
            **({"exact_window": args.window} if args.window > 0 else {}),
            **({"decoupled_rope": D_ROPE} if args.decoupled else {}),
            **({"paged": {"page_size": args.paged, "pages_shuffled": True}} if args.paged else {}),
            "T": w.T, "H": w.H, "d_head": w.d, "r_k": w.r_k,
            "r_v": w.r_v, "batch_per_gpu": w.B, "seq_len_range": [w.len_lo, w.len_hi],
            "latent_tokens_per_gpu": tokens, "parallelism": "dp%d" % world,
            "layers_per_step": layers,
            "step": "%slla_encode of %d new tokens + %s for loops 1..%d" % (
                "per layer: " if layers > 1 else "", w.B,
                "lla_decode_attn_decoupled" if args.decoupled else "lla_decode_attn", w.T),
            "l2": "inputs larger than L2 (%.2f GB of latents per GPU)" % (
                w.B * w.H * w.L_max * (w.r_k + w.r_v) * 2 / 1e9)}


def e2e_run(step: DecodeStep, steps: int):
    """Same step through the public API with the per-step inputs coming from pinned
    host memory and the results read back: new-token stacks, queries, lengths
    (host->device) and out/lse (device->host)."""
    # every layer buffer's new-token stacks, the lengths, every layer's queries in; the
    # last layer's out / lse back (all of them for a one-layer step)
    pairs = [(b[k], b[k].cpu().pin_memory()) for b in step.bufs for k in ("x_k", "x_v")]
    pairs += [(step.inp[k], step.inp[k].cpu().pin_memory()) for k in ("seq_lens", "q_pos")]
    pairs.append((step.qL, step.qL.cpu().pin_memory()))
    out_dev, lse_dev = step.outL[-1], step.lseL[-1]
    host_out = torch.empty(out_dev.shape, dtype=torch.float32).pin_memory()
    host_lse = torch.empty(lse_dev.shape, dtype=torch.float32).pin_memory()
    h2d = sum(h.numel() * h.element_size() for _, h in pairs)
    d2h = host_out.numel() * 4 + host_lse.numel() * 4
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        for dev, h in pairs:
            dev.copy_(h, non_blocking=True)
        step.run()
        host_out.copy_(out_dev, non_blocking=True)
        host_lse.copy_(lse_dev, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    dt = time.perf_counter() - t0
    return dt, h2d, d2h


def oracle_sample(w, inp_dev, q_dev, budget_s=12.0, k_rope=None, dense=None):
    """Time the oracle on the first S sequences (all heads, all loops) of the same
    inputs; S grows from 1 until the run would take about ``budget_s``.  With
    ``k_rope`` it is the decoupled-RoPE decode's oracle."""
    import oracle
    odm = oracle.dims(w.T, w.H, w.d, w.r_k, w.r_v, w.variant, w.rope_base)
    wk, wv = widen(inp_dev["w_up_k"]), widen(inp_dev["w_up_v"])
    mk, mv = widen(inp_dev["mu_k"]), widen(inp_dev["mu_v"])
    lens = inp_dev["seq_lens"].cpu().numpy()

    def run(S, loops):
        dk, dv = dense(S) if dense is not None else (inp_dev["cache_k"][:S], inp_dev["cache_v"][:S])
        ck, cv = widen(dk), widen(dv)
        kr = widen(k_rope[:S]) if k_rope is not None else None
        t0 = time.perf_counter()
        for t in range(loops):
            if kr is not None:
                oracle.decoupled(odm, t, widen(q_dev[t][:S]), ck, cv, kr, lens[:S], lens[:S] - 1, wk, wv, mk, mv)
            else:
                oracle.decode(odm, t, widen(q_dev[t][:S]), ck, cv, lens[:S], lens[:S] - 1, wk, wv, mk, mv)
        return time.perf_counter() - t0

    t1 = run(1, 1)
    S = int(max(1, min(w.B, budget_s / max(t1 * w.T, 1e-3))))
    dt = run(S, w.T)
    tokens = float(lens[:S].sum()) * w.T
    return {"value": tokens / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "first %d of %d sequences, all %d heads, loops 1..%d (%.0f latent tokens x "
                      "loops) in %.2f s" % (S, w.B, w.H, w.T, tokens, dt)}


def oracle_prefill_sample(w, inp_dev, x_dev, budget_s=8.0):
    """Time the oracle's encode (Eq. (2), both axes, all heads) on the first S tokens of
    the prefill stack; S grows from 128 until the run would take about ``budget_s``."""
    import oracle
    odm = oracle.dims(w.T, w.H, w.d, w.r_k, w.r_v, w.variant, w.rope_base)
    wd = (widen(inp_dev["w_down_k"]), widen(inp_dev["w_down_v"]))
    mu = (widen(inp_dev["mu_k"]), widen(inp_dev["mu_v"]))
    units = w.H if w.variant == 0 else 1

    def run(S):
        xs = (widen(x_dev[0][:S]), widen(x_dev[1][:S]))
        si = np.zeros(S, dtype=np.int32)
        po = np.arange(S, dtype=np.int32)
        shape = (1, units, S) if w.variant == 0 else (1, S)
        outs = (np.zeros(shape + (w.r_k,)), np.zeros(shape + (w.r_v,)))
        t0 = time.perf_counter()
        for a in range(2):
            oracle.encode(odm, xs[a], si, po, wd[a], mu[a], (w.r_k, w.r_v)[a], outs[a], round_to_bf16=True)
        return time.perf_counter() - t0

    t1 = run(128)
    S = int(max(128, min(x_dev[0].shape[0], 128 * budget_s / max(t1, 1e-3))))
    dt = run(S)
    return {"value": S / dt, "unit": "prefill tokens/s per layer", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "first %d of %d tokens of the prefill stack (one sequence's positions), all %d heads, "
                      "both axes, in %.2f s" % (S, x_dev[0].shape[0], w.H, dt)}


def measure(args, w, steps, layers, dist_on, rank, world, device, legs=True):
    """Time ``steps`` steps of workload ``w`` (``layers`` layers per step) after
    ``args.warmup`` warm-up steps; the result line's measured fields.  ``legs`` runs
    the optional legs the arguments ask for (window, eviction, prefill)."""
    step = DecodeStep(w, 20260000 + 1 + 1000 * rank, device, window=args.window, decoupled=args.decoupled,
                      paged=args.paged, layers=layers, prefill=legs and args.prefill)
    T = w.T
    LT = T * layers
    # Decode-call timing: events around each layer's T consecutive calls (one call's
    # time = the group's / T; no event between calls, so back-to-back calls run as
    # they would untimed), or around every call when the window call follows each one
    group = not (legs and args.window > 0)
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(LT)] for _ in range(3)]
          for _ in range(steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        clk.wait_live()
        for _ in range(args.warmup):
            step.run()
        torch.cuda.synchronize()
        st = lla.device_status(step.ws)
        if st != lla.LLA_OK:
            raise RuntimeError("device status after warm-up: " + lla.status_string(st))
        barrier(dist_on)
        torch.cuda.synchronize()
        h0 = time.perf_counter()
        start.record()
        for k in range(steps):
            step.run(ev[k], group)
        stop.record()
        torch.cuda.synchronize()
        h1 = time.perf_counter()
        clocks = clk.summary(h0, h1)
        if clocks["samples"] < 3:
            # a timed region shorter than three samples: the same step, untimed, right
            # after it for about 0.4 s, and the clock record taken over those repeats
            h2 = time.perf_counter()
            while time.perf_counter() - h2 < 0.4:
                for _ in range(max(1, min(steps, 50))):
                    step.run()
                torch.cuda.synchronize()
            clocks = clk.summary(h2, time.perf_counter())
            clocks["window"] = "untimed repeats of the step right after the timed region (%.0f ms, shorter " \
                               "than three %d ms samples)" % ((h1 - h0) * 1e3, clk.PERIOD_MS)
        barrier(dist_on)
    elapsed = start.elapsed_time(stop) / 1e3
    st = lla.device_status(step.ws)
    if st != lla.LLA_OK:
        raise RuntimeError("device status after timing: " + lla.status_string(st))
    t_max = max_over_ranks(elapsed, dist_on, device)
    tokens_all = sum_over_ranks(float(step.tokens * LT * steps), dist_on, device)
    value = tokens_all / t_max

    # dominant kernel: the decode call (main kernel + its small combine), timed per launch
    if group:
        durs = [ev[k][0][l * T].elapsed_time(ev[k][1][l * T + T - 1]) / 1e3 / T
                for k in range(steps) for l in range(layers)]
    else:
        durs = [ev[k][0][t].elapsed_time(ev[k][1][t]) / 1e3 for k in range(steps) for t in range(LT)]
    t_call = float(np.mean(durs))
    hbm, tflops, src = peaks()
    if args.decoupled:
        # latent K and V rows plus the rotary key of every token-head, bf16
        lat_bytes = step.tokens * w.H * (w.r_k + w.r_v + D_ROPE) * 2
        achieved = lat_bytes / t_call / 1e9
        import hashlib
        small = lla.decoupled_kernel(step.dm, D_ROPE) == "small-rank"
        src_file, sha, per_th = ((DECOUPLED_SMALL_SRC, TRAFFIC_DEC_SMALL_SRC_SHA, TRAFFIC_DEC_SMALL_PER_TOKEN_HEAD)
                                 if small else (DECOUPLED_SMALL_SRC, TRAFFIC_DEC_TILE_SRC_SHA,
                                                TRAFFIC_DEC_TILE_PER_TOKEN_HEAD))
        with open(src_file, "rb") as f:
            same_src = sha is not None and hashlib.sha256(f.read()).hexdigest().startswith(sha)
        traffic = per_th * step.tokens * w.H if same_src else None
        main = "decoupled_small_kernel" if small else "decoupled_tile_kernel"
        query = "decoupled_small_z_kernel"
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic, "traffic_kernel": main,
                "kernel": "lla_decode_attn_decoupled (%s + %s + decode_combine_kernel)" % (query, main),
                "algorithmic_bytes_per_launch": lat_bytes, "launch_ms": t_call * 1e3,
                "peak_source": src}
    elif w.variant == 0:
        lat_bytes = step.tokens * w.H * (w.r_k + w.r_v) * 2
        achieved = lat_bytes / t_call / 1e9
        import hashlib
        small = lla.decode_kernel(step.dm) == "small-rank"
        per_tile = TRAFFIC_PER_TOKEN_HEAD[min(TRAFFIC_PER_TOKEN_HEAD, key=lambda L: abs(L - w.L_max))]
        src_file, sha, per_th = ((DECODE_SMALL_SRC, TRAFFIC_SMALL_SRC_SHA, TRAFFIC_SMALL_PER_TOKEN_HEAD)
                                 if small else (DECODE_SRC, TRAFFIC_SRC_SHA, per_tile))
        with open(src_file, "rb") as f:
            same_src = sha is not None and hashlib.sha256(f.read()).hexdigest().startswith(sha)
        # (the counters were taken on the dense cache; a paged run reports none)
        traffic = per_th * step.tokens * w.H if same_src and not args.paged else None
        kern = "decode_small_kernel" if small else "decode_bf16_kernel"
        zk = "decode_small_z_kernel" if small else "decode_z_kernel"
        kname = "lla_decode_attn (%s + %s + decode_combine_kernel)" % (zk, kern)
        if step.gathers_rows():
            kern, kname = "decode_paged_generic_kernel", "lla_decode_attn_paged (decode_paged_generic_kernel)"
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic, "traffic_kernel": kern,
                "kernel": kname,
                "algorithmic_bytes_per_launch": lat_bytes, "launch_ms": t_call * 1e3,
                "peak_source": src}
    else:
        # LLA-2D: K reconstruction of every head (2 d r_k) + absorbed V (2 r_v) per
        # latent token-head; latents are shared by the heads, so the call is bound by
        # the tensor pipe (about 700 flop per latent byte at H = 16, r = (128, 256))
        flops = step.tokens * w.H * (2 * w.d * w.r_k + 2 * w.r_v)
        achieved = flops / t_call / 1e12
        import hashlib
        with open(DECODE2D_SRC, "rb") as f:
            same_src = hashlib.sha256(f.read()).hexdigest().startswith(TRAFFIC2D_SRC_SHA)
        traffic = TRAFFIC2D_PER_TOKEN * step.tokens if same_src else None
        roof = {"bound": "tensor", "achieved": achieved, "peak": tflops, "unit": "TFLOP/s",
                "frac": achieved / tflops, "traffic": traffic, "traffic_kernel": "decode2d_score_kernel",
                "kernel": "lla_decode_attn (decode2d_z_kernel + decode2d_score_kernel + "
                          "decode2d_value_kernel + decode2d_combine_kernel)",
                "algorithmic_flops_per_launch": flops,
                "latent_bytes_per_launch": step.tokens * (w.r_k + w.r_v) * 2,
                "launch_ms": t_call * 1e3, "peak_source": src + " (bf16 sustained)"}

    roof["launch_timing"] = ("CUDA events around each layer's %d back-to-back decode calls in the timed steps; "
                             "launch_ms = group time / %d" % (T, T)) if group else \
        "CUDA events around every decode call in the timed steps"

    win = None
    if legs and args.window > 0:
        # exact-window call: window K/V + query read, out / lse read and written
        wdur = float(np.mean([ev[k][1][t].elapsed_time(ev[k][2][t]) / 1e3
                              for k in range(steps) for t in range(T)]))
        esz = 2 if w.dtype == "bf16" else 4
        wtok = int(step.win["win_len"].sum().item())
        wbytes = wtok * w.H * 2 * w.d * esz + w.B * w.H * (w.d * esz + 2 * (w.d + 1) * 4)
        wach = wbytes / wdur / 1e9
        win = {"W": args.window, "window_tokens_per_call": wtok * w.H, "call_ms": wdur * 1e3,
               "roofline": {"bound": "hbm", "achieved": wach, "peak": hbm, "unit": "GB/s", "frac": wach / hbm,
                            "traffic": None, "kernel": "lla_window_attn (window_attn_kernel)",
                            "algorithmic_bytes_per_launch": wbytes, "peak_source": src}}

    evi = None
    if legs and args.evict:
        # token eviction composed with LLA (sink + window budget): lla_evict_window on the
        # layer (lengths restored before each call, outside the events), then one decode
        # call per loop over the kept budget
        sink, window = (int(x) for x in args.evict.split(","))
        i = step.inp
        saved = i["seq_lens"].clone()
        ews = torch.zeros(256, dtype=torch.uint8, device=device)
        esize = 2 if w.dtype == "bf16" else 4
        over = [L for L in saved.cpu().tolist() if L > sink + window]
        units = w.H if w.variant == 0 else 1
        moved = len(over) * units * window * (w.r_k + w.r_v) * esize * 2
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(3, min(args.steps, 100))
        etimes = []
        for k in range(reps + 3):
            i["seq_lens"].copy_(saved)
            e0.record()
            lla.evict_window(step.dm, i["cache_k"], i["cache_v"], i["seq_lens"], sink, window, ews)
            e1.record()
            torch.cuda.synchronize()
            if k >= 3:
                etimes.append(e0.elapsed_time(e1) / 1e3)
        if lla.device_status(ews) != lla.LLA_OK:
            raise RuntimeError("device status after eviction")
        t_ev = float(np.mean(etimes))
        kept = int(i["seq_lens"].sum().item())
        q_pos_kept = (i["seq_lens"] - 1).clamp(min=0).to(torch.int32)
        dtimes = []
        for k in range(reps + 3):
            e0.record()
            for t in range(T):
                lla.decode_attn(step.dm, t, step.q[t], i["cache_k"], i["cache_v"], i["seq_lens"], q_pos_kept,
                                i["w_up_k"], i["w_up_v"], i["mu_k"], i["mu_v"], step.cos, step.sin, step.out[t],
                                step.lse[t], step.ws)
            e1.record()
            torch.cuda.synchronize()
            if k >= 3:
                dtimes.append(e0.elapsed_time(e1) / 1e3 / T)
        i["seq_lens"].copy_(saved)
        t_dec = float(np.mean(dtimes))
        evi = {"sink": sink, "window": window, "sequences_evicted": len(over), "evict_ms": t_ev * 1e3,
               "roofline": {"bound": "hbm", "achieved": moved / t_ev / 1e9, "peak": hbm, "unit": "GB/s",
                            "frac": moved / t_ev / 1e9 / hbm, "traffic": None,
                            "kernel": "lla_evict_window (evict_move_kernel + evict_lens_kernel)",
                            "algorithmic_bytes_per_launch": moved, "peak_source": src},
               "decode_over_budget": {"latent_tokens_per_call": kept, "call_ms": t_dec * 1e3,
                                      "value": kept / t_dec, "unit": UNIT}}

    pre = None
    if legs and args.prefill:
        with ClockSampler(torch.cuda.current_device()) as pclk:
            pclk.wait_live()
            pre = prefill_run(step, max(3, min(args.steps, 10)), hbm, src)
        pre["clocks"] = pclk.summary()
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            pre["cpu_baseline"] = oracle_prefill_sample(w, step.inp, step.prefill_x)

    e2e_steps = max(3, min(steps, 200))
    e2e_dt, h2d, d2h = e2e_run(step, e2e_steps)
    e2e_dt = max_over_ranks(e2e_dt, dist_on, device)
    e2e_val = sum_over_ranks(float(step.tokens * LT * e2e_steps), dist_on, device) / e2e_dt

    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": t_max / steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": arm_config(w, args, step.tokens, world, layers),
        **({"layer_buffers": len(step.bufs)} if layers > 1 else {}),
        "roofline": roof,
        **({"window": win} if win else {}),
        **({"evict": evi} if evi else {}),
        **({"prefill": pre} if pre else {}),
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": step.launches() * steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = oracle_sample(w, step.inp, step.q,
                                            k_rope=step.k_rope if args.decoupled else None,
                                            dense=step.dense_view)
    del step
    torch.cuda.empty_cache()
    return res


# the second Ouro-1.4B 4k-context workload, measured beside the headline in the default run
SECOND = "ouro1.4b_rho21_b768_4k"
SECOND_MAX_STEPS = 40


def step_layers(args, w):
    """Layers per step: --layers, else the workload's stack (one layer when an optional
    leg that works on a single layer is asked for)."""
    if args.layers:
        return args.layers
    if args.window or args.decoupled or args.paged or args.evict or args.prefill:
        return 1
    return w.layers


def run_ours(args, dist_on, rank, world, device):
    w = WORKLOADS[args.workload]
    lla_build.build()
    lla.lib()
    res = measure(args, w, args.steps, step_layers(args, w), dist_on, rank, world, device)
    if (args.workload == DEFAULT_WORKLOAD and not args.no_second and not
            (args.window or args.decoupled or args.paged or args.evict or args.prefill or args.layers)):
        # rho = 21.3 at serving batch (768 x 4096), the full step of its 24-layer stack:
        # 24 new-token encodes and 96 decode calls (the other Ouro-1.4B 4k workload)
        w2 = WORKLOADS[SECOND]
        n2 = min(args.steps, SECOND_MAX_STEPS)
        sub = measure(args, w2, n2, w2.layers, dist_on, rank, world, device, legs=False)
        res[SECOND.split("_", 1)[1].rsplit("_", 1)[0]] = {
            k: sub[k] for k in ("value", "unit", "steps", "warmup", "ms_per_step", "config", "layer_buffers",
                                "roofline", "e2e", "gpu_launches", "clocks", "cpu_baseline") if k in sub}
    return res


# ----------------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle as it stands, on the host cores, on a bounded sample of the same
    workload per step (first sequence, all heads, one loop per step, cycling t)."""
    import oracle
    w = WORKLOADS[args.workload]
    # drawn exactly as the GPU arm's step draws it (with the new-token stacks), so the
    # lengths, and hence the config, are the same
    inp = make_decode_inputs(dataclasses.replace(w, N_encode=min(w.N_encode, w.B)), 20260000 + 1,
                             device="cuda" if torch.cuda.is_available() else "cpu", with_encode=True)
    odm = oracle.dims(w.T, w.H, w.d, w.r_k, w.r_v, w.variant, w.rope_base)
    S = 1
    ck, cv, q = widen(inp["cache_k"][:S]), widen(inp["cache_v"][:S]), widen(inp["q"][:S])
    wk, wv, mk, mv = (widen(inp[k]) for k in ("w_up_k", "w_up_v", "mu_k", "mu_v"))
    lens = inp["seq_lens"][:S].cpu().numpy()
    for i in range(args.warmup):
        oracle.decode(odm, i % w.T, q, ck, cv, lens, lens - 1, wk, wv, mk, mv)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.decode(odm, i % w.T, q, ck, cv, lens, lens - 1, wk, wv, mk, mv)
    dt = time.perf_counter() - t0
    value = float(lens.sum()) * args.steps / dt
    sample = "sequence 0 of %d (%d tokens), all %d heads, one loop per step" % (w.B, int(lens.sum()), w.H)
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": arm_config(w, args, int(inp["seq_lens"].sum().item()),
                                 int(os.environ.get("WORLD_SIZE", "1")), step_layers(args, w)),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="layers per step (default: the workload's stack; buffers cycle when it exceeds HBM)")
    ap.add_argument("--no-second", action="store_true",
                    help="skip the second Ouro-1.4B 4k workload the default run measures (rho = 21.3, 768 x 4096)")
    ap.add_argument("--window", type=int, default=0,
                    help="also run lla_window_attn over an exact window of this many newest tokens")
    ap.add_argument("--evict", default="",
                    help="SINK,WINDOW: also time lla_evict_window to that budget and decode over it")
    ap.add_argument("--paged", type=int, default=0,
                    help="keep the cache in shuffled pages of this many tokens (lla_decode_attn_paged)")
    ap.add_argument("--decoupled", action="store_true",
                    help="decode with lla_decode_attn_decoupled (64 rotary dimensions per token-head)")
    ap.add_argument("--prefill", action="store_true",
                    help="also time lla_encode of the workload's whole prefill stack (ouro_rho4_b64_16k)")
    args = ap.parse_args()
    if args.prefill:
        pw = WORKLOADS[args.workload]
        if pw.N_encode != pw.B * pw.L_max or args.paged:
            ap.error("--prefill needs a workload with a prefill stack (ouro_rho4_b64_16k) and the dense cache")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.paged and (args.decoupled or WORKLOADS[args.workload].variant != 0):
        ap.error("--paged takes the per-head decode only")
    if args.evict and (args.paged or args.decoupled):
        ap.error("--evict runs on the dense cache")
    if args.decoupled and args.window > 0:
        ap.error("--decoupled and --window do not combine (the window call takes d-wide queries)")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    dist_on = world > 1
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if dist_on:
        init_dist("nccl", device)
    try:
        res = run_ours(args, dist_on, rank, world, device)
        if rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        if dist_on:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
