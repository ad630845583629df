#!/usr/bin/env python
"""Benchmark of the absorbed-MLA decode step on GB300.

One step = the whole decode path for one batch: mla_append_latent (the new
token of every sequence) -> mla_absorb_q -> mla_decode_attn (attention +
split-KV combine) -> mla_expand_v, all through the C ABI, inputs resident in HBM.

Default workload: B=64 sequences, H=16 heads, one query token, L=4096 cached
tokens each (contiguous cache, 302 MB of latent rows: larger than the 129 MB
L2, so every step streams the cache from HBM). The other decode workloads
(H=128 paged, ragged, two query tokens), prompt chunks in the absorbed form and
in the expanded (MHA) form (mla_prefill_mha), the FP8 cache and the one-launch
short step are measured too and reported under "workloads"; the projections
around the attention under "extras".

Prints ONE JSON line on rank 0. `value` is latent-cache GB/s of the whole job
(cache bytes of all ranks per step / step time); `ms_per_step` gives the step
time. `--impl reference` times the float64 CPU oracle on a bounded sample
instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "absorbed-MLA decode µs/step and latent-cache HBM GB/s vs GB300 roofline"
ROW_BYTES = 1152
ROW8_BYTES = 656      # FP8 cache row: e4m3 latent | bf16 RoPE key | fp32 scale | padding


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def reduce_max_over_ranks(x: float, dist, device) -> float:
    """Max of a per-rank float over all ranks (identity without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbps(cache_bytes_per_rank: int, world: int, step_s: float) -> float:
    """Whole-job latent-cache throughput: every rank streams its own batch's cache
    once per step (weak scaling), timed by the slowest rank."""
    return world * cache_bytes_per_rank / step_s / 1e9


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class Clocks:
    """nvidia-smi sampler for the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _kernel_hash():
    h = hashlib.sha256()
    for f in ["decode_attn.cu", "decode_attn_pair.cu", "attn_sched.cuh", "mla_ptx.cuh", "mla_kernels.cuh"]:
        with open(os.path.join(ROOT, "mla_absorbed_latent_02_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic_per_token(workload: str):
    """DRAM bytes per cached token of the attention kernel on `workload` from the
    committed ncu summary, or None when it is missing, covers another workload,
    or was taken on other kernel sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "decode_attn_traffic.json")) as f:
            d = json.load(f)
        if d.get("kernel_hash") != _kernel_hash():
            return None
        return float(d["workloads"][workload]["dram_bytes_per_token"])
    except Exception:
        return None


# --------------------------------------------------------------------------- GPU arm
class Bench:
    """One decode workload: cache prefilled with tokens 0..L-Hq-1 of every
    sequence, the step's new tokens L-Hq..L-1 and the queries loaded into a
    DecodeStep (the library's public step object)."""

    def __init__(self, m, S, torch, ctx, wl, device, fp8=False, small=False):
        self.m, self.S, self.torch, self.ctx, self.wl = m, S, torch, ctx, wl
        self.fp8 = fp8
        self.small = small
        self.name = wl.name + ("_fp8" if fp8 else "") + ("_one_launch" if small else "")
        dev = torch.device(device)
        self.dev = dev
        B, H, Hq = wl.B, wl.H, wl.Hq
        w_uk, w_uv = S.weights(wl, device=dev)
        if wl.paged:
            bt = torch.full((B, wl.max_blocks), -1, dtype=torch.int32)
            for b, row in enumerate(wl.block_table):
                bt[b, :len(row)] = torch.tensor(row, dtype=torch.int32)
            cache = m.Cache.paged_pool(wl.num_blocks, bt, device=dev, fp8=fp8)
        else:
            cache = m.Cache.contiguous(B, wl.capacity, device=dev, fp8=fp8)
        # prefill the cache with tokens 0 .. L-Hq-1 (outside any timing)
        for b in range(B):
            n = wl.seq_lens[b] - Hq
            if n <= 0:
                continue
            c, k = S.token_inputs(wl, b, device=dev, t0=0, t1=n)
            ctx.append_latent(cache, c, k, torch.full((n,), b, dtype=torch.int32, device=dev),
                              torch.arange(0, n, dtype=torch.int32, device=dev))
        # the step's new tokens: positions L-Hq .. L-1 of every sequence
        cs, ks, seq, pos = [], [], [], []
        for b in range(B):
            L = wl.seq_lens[b]
            t0 = max(0, L - Hq)
            c, k = S.token_inputs(wl, b, device=dev, t0=t0, t1=L)
            cs.append(c)
            ks.append(k)
            seq += [b] * (L - t0)
            pos += list(range(t0, L))
        self.step = m.DecodeStep(ctx, cache, w_uk, w_uv, B, Hq, n_new=len(seq), small=small)
        st = self.step
        st.c_kv.copy_(torch.cat(cs))
        st.k_rope.copy_(torch.cat(ks))
        st.seq_idx.copy_(torch.tensor(seq, dtype=torch.int32))
        st.pos.copy_(torch.tensor(pos, dtype=torch.int32))
        qn, qr = S.query_inputs(wl, device=dev)
        st.q_nope.copy_(qn)
        st.q_rope.copy_(qr)
        st.q_pos.copy_(torch.tensor(S.query_positions(wl), dtype=torch.int32))
        st.seq_lens.copy_(torch.tensor(wl.seq_lens, dtype=torch.int32))
        torch.cuda.synchronize()
        self.tokens = wl.total_tokens
        self.cache_bytes = self.tokens * (ROW8_BYTES if fp8 else ROW_BYTES)
        # append + absorb_q (one launch), attention, combine, expand_v; or the one-launch step
        self.launches_per_step = 1 if small else 4

    def first_output(self):
        """The last step's output of the first sequence with a query, [Hq, H, 128]
        as float64 on the host (every step rewrites the same rows, so it is the
        output of any step)."""
        self.torch.cuda.synchronize()
        b = next(i for i, L in enumerate(self.wl.seq_lens) if L >= self.wl.Hq)
        return self.step.out[b].double().cpu().numpy()

    def algorithmic(self):
        wl = self.wl
        B, H, Hq = wl.B, wl.H, wl.Hq
        attn_bytes = self.cache_bytes + B * Hq * H * (576 * 2 + 512 * 4 + 4)
        # query j of sequence b attends L_b - Hq + 1 + j tokens (bottom-right causal)
        pairs = sum(Hq * (L - Hq + 1) + Hq * (Hq - 1) // 2 for L in wl.seq_lens if L >= Hq)
        attn_flops = 2 * H * (576 + 512) * pairs
        step_bytes = (self.cache_bytes + 2 * H * 128 * 512 * 2 + B * Hq * H * (128 + 64 + 128) * 2
                      + B * Hq * 1152 + 2 * B * Hq * H * (576 * 2 + 512 * 4))
        return attn_bytes, attn_flops, step_bytes

    def time_steps(self, steps, warmup, dist=None):
        """W direct warm-up steps, then K steps captured as one CUDA graph and
        replayed once untimed and once timed (barrier + synchronize on both
        sides). The attention launch durations come from a second K-step graph
        with an event pair around every attention call (event nodes between the
        kernels would otherwise break their programmatic overlap)."""
        torch = self.torch
        for _ in range(warmup):
            self.step.run()
        torch.cuda.synchronize()
        self.step.capture(steps)
        self.step.replay()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t0.record()
        self.step.replay()
        t1.record()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        total_ms = t0.elapsed_time(t1)
        try:
            evs = [(torch.cuda.Event(enable_timing=True, external=True),
                    torch.cuda.Event(enable_timing=True, external=True)) for _ in range(steps)]
            self.step.capture(steps, evs)
            self.step.replay()
            torch.cuda.synchronize()
            self.step.replay()
            torch.cuda.synchronize()
            attn_ms = [a.elapsed_time(b) for a, b in evs]
        except Exception:
            attn_ms = self.time_attention_direct(steps)
        return total_ms, attn_ms

    def time_direct(self, steps):
        """The same step as plain launches (no graph): K direct steps between
        CUDA events on the launching stream; mean us per step."""
        torch = self.torch
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            self.step.run()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / steps

    def time_attention_direct(self, steps):
        """Fallback: back-to-back direct attention calls with an event pair each."""
        torch = self.torch
        st = self.step
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            a.record()
            self.ctx.decode_attn(st.cache, st.q_abs, st.seq_lens, st.scale, st.workspace, st.o_lat, st.lse)
            b.record()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def time_e2e(self, steps, warmup):
        """The step through the public API with host buffers: every step copies
        the pinned host input arena to the device (one copy kernel), runs the step
        and copies the output back to pinned host memory (one graph replay),
        then waits for it on the host. Wall-clock time per step."""
        torch = self.torch
        st = self.step
        host = st.host_inputs()
        for k, v in host.items():
            v.copy_(getattr(st, k))
        h2d = st.input_bytes
        d2h = st.out_host.numel() * st.out_host.element_size()
        st.capture(1, host_io=True)

        def one():
            st.replay()
            torch.cuda.current_stream().synchronize()

        for _ in range(warmup):
            one()
        t = time.perf_counter()
        for _ in range(steps):
            one()
        dt = (time.perf_counter() - t) / steps
        return dt, h2d, d2h


def time_out_proj(m, S, torch, ctx, M, H, d_model, steps, peaks):
    """The attention block's output projection (mla_out_proj) on its own: a graph
    of `steps` back-to-back calls with inputs resident. Consecutive calls use
    different copies of W_O, together larger than L2, so every call reads its
    weight from HBM."""
    hbm = peaks[0]
    dev = torch.device("cuda")
    w0 = S.normal_bf16(0, f"bench/w_o/{H}/{d_model}", (d_model, H * 128), std=0.02, device=dev)
    copies = max(1, -(-200_000_000 // (w0.numel() * 2)))
    ws = [w0] + [w0.clone() for _ in range(copies - 1)]
    w = w0
    o = S.normal_bf16(0, f"bench/o/{M}/{H}", (M, H, 128), device=dev)
    y = torch.empty(M, d_model, dtype=torch.float32, device=dev)
    for i in range(3):
        ctx.out_proj(ws[i % copies], o, y=y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ctx.out_proj(w, o, y=y)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        for i in range(steps):
            ctx.out_proj(ws[i % copies], o, y=y)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / steps
    nbytes = w.numel() * 2 + o.numel() * 2 + y.numel() * 4
    return {"op": "out_proj", "M": M, "H": H, "d_model": d_model, "us_per_call": round(t * 1e6, 2),
            "GBps": round(nbytes / t / 1e9, 1), "bound": "hbm", "roofline_frac": round(nbytes / t / 1e9 / hbm, 3),
            "weight_MB": round(w.numel() * 2 / 1e6, 1),
            "l2": f"{copies} weight copies rotated ({round(copies * w.numel() * 2 / 1e6)} MB, larger than L2)"}


def time_expand_out_proj(m, S, torch, ctx, M, H, d_model, steps, peaks):
    """The attention's latent output to the block's hidden output, both ways:
    expand_v then out_proj (two calls), and out_proj_latent over W_OV (W_UV folded
    into W_O, one call). Each a graph of `steps` back-to-back steps rotating weight
    copies that together exceed L2."""
    hbm = peaks[0]
    dev = torch.device("cuda")
    w_o = S.normal_bf16(0, f"bench/w_o/{H}/{d_model}", (d_model, H * 128), std=0.02, device=dev)
    w_uv = S.normal_bf16(0, f"bench/w_uv/{H}", (H, 128, 512), std=0.02, device=dev)
    w_ov = ctx.absorb_w_o(w_o, w_uv)
    o_lat = (0.3 * S.normal_bf16(0, f"bench/o_lat/{M}/{H}", (M, H, 512), device=dev).float()).contiguous()
    o = torch.empty(M, H, 128, dtype=torch.bfloat16, device=dev)
    y = torch.empty(M, d_model, dtype=torch.float32, device=dev)

    def timed(weights, call):
        copies = max(1, -(-200_000_000 // sum(w.numel() * 2 for w in weights[0])))
        sets = [weights[0]] + [[w.clone() for w in weights[0]] for _ in range(copies - 1)]
        for i in range(3):
            call(*sets[i % copies])
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            call(*sets[0])
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(steps):
                call(*sets[i % copies])
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        nbytes = sum(w.numel() * 2 for w in weights[0])
        del sets
        return e0.elapsed_time(e1) / 1e3 / steps, nbytes, copies

    o_lat4 = o_lat.view(M, 1, H, 512)
    t2, b2, c2 = timed([[w_uv, w_o]], lambda wu, wo: (ctx.expand_v(wu, o_lat4, out=o), ctx.out_proj(wo, o, y=y)))
    t1, b1, c1 = timed([[w_ov]], lambda wov: ctx.out_proj_latent(wov, o_lat, y=y))
    act = o_lat.numel() * 4 + y.numel() * 4
    rec = {"op": "latent_to_hidden", "M": M, "H": H, "d_model": d_model,
           "two_calls_us": round(t2 * 1e6, 2), "two_calls_weight_MB": round(b2 / 1e6, 1),
           "two_calls_roofline_frac": round((b2 + act) / t2 / 1e9 / hbm, 3),
           "one_call_w_ov_us": round(t1 * 1e6, 2), "one_call_weight_MB": round(b1 / 1e6, 1),
           "one_call_roofline_frac": round((b1 + act) / t1 / 1e9 / hbm, 3),
           "faster": "one_call_w_ov" if t1 < t2 else "two_calls", "bound": "hbm",
           "l2": f"weights rotated over {c2} / {c1} copies (more than L2)"}
    del w_ov
    torch.cuda.empty_cache()
    return rec


def time_project_latent(m, S, torch, ctx, n, d_model, steps, peaks):
    """The latent producer (mla_project_latent: projection, kv_norm, RoPE, cache
    write) for n new tokens, a graph of `steps` calls rotating weight copies that
    together exceed L2."""
    hbm = peaks[0]
    dev = torch.device("cuda")
    w0 = S.normal_bf16(0, f"bench/w_kv_a/{d_model}", (576, d_model), std=0.02, device=dev)
    copies = max(1, -(-200_000_000 // (w0.numel() * 2)))
    ws = [w0] + [w0.clone() for _ in range(copies - 1)]
    h = S.normal_bf16(0, f"bench/h/{n}/{d_model}", (n, d_model), device=dev)
    g = (1.0 + 0.1 * S.normal_bf16(0, "bench/kv_norm", (512,), device=dev).float()).to(torch.bfloat16)
    cache = m.Cache.contiguous(n, 8, device=dev)
    seq = torch.arange(n, dtype=torch.int32, device=dev)
    pos = torch.full((n,), 5, dtype=torch.int32, device=dev)
    work = torch.empty((ctx.lib.mla_project_latent_workspace_size(n) + 3) // 4, dtype=torch.float32, device=dev)
    for i in range(3):
        ctx.project_latent(cache, ws[i % copies], h, seq, pos, kv_norm=g, workspace=work)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ctx.project_latent(cache, w0, h, seq, pos, kv_norm=g, workspace=work)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        for i in range(steps):
            ctx.project_latent(cache, ws[i % copies], h, seq, pos, kv_norm=g, workspace=work)
    gr.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    gr.replay()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / steps
    nbytes = w0.numel() * 2 + h.numel() * 2 + n * 1152
    return {"op": "project_latent", "n": n, "d_model": d_model, "us_per_call": round(t * 1e6, 2),
            "GBps": round(nbytes / t / 1e9, 1), "bound": "hbm", "roofline_frac": round(nbytes / t / 1e9 / hbm, 3),
            "weight_MB": round(w0.numel() * 2 / 1e6, 2),
            "l2": f"{copies} weight copies rotated ({round(copies * w0.numel() * 2 / 1e6)} MB, larger than L2)"}


def time_prefill_mha(m, S, torch, ctx, wl, steps, warmup, peaks, check=True):
    """A prompt chunk in the expanded (MHA) form, mla_prefill_mha: the cache
    holds each sequence's prefix (tokens 0 .. L-T-1) beforehand; every step
    appends the chunk's T rows (mla_append_latent), expands K and V of every
    cached token and runs the causal attention. `warmup` untimed steps, then
    `steps` back-to-back steps between CUDA events, and the mla_prefill_mha call
    alone the same way. Algorithmic FLOPs: 2*H*256*512 per cached token (the
    expansion) plus 2*H*(192+128) per attended (query, key) pair."""
    import math
    hbm, tf, tfs, kind = peaks
    dev = torch.device("cuda")
    B, H, T = wl.B, wl.H, wl.Hq
    w_uk, w_uv = S.weights(wl, device=dev)
    cache = m.Cache.contiguous(B, wl.capacity, device=dev)
    cs, ks, seq, pos = [], [], [], []
    for b in range(B):
        L = wl.seq_lens[b]
        if L - T > 0:
            c, k = S.token_inputs(wl, b, device=dev, t0=0, t1=L - T)
            ctx.append_latent(cache, c, k, torch.full((L - T,), b, dtype=torch.int32, device=dev),
                              torch.arange(0, L - T, dtype=torch.int32, device=dev))
        c, k = S.token_inputs(wl, b, device=dev, t0=L - T, t1=L)
        cs.append(c)
        ks.append(k)
        seq += [b] * T
        pos += list(range(L - T, L))
    c_new, k_new = torch.cat(cs).contiguous(), torch.cat(ks).contiguous()
    seq_t = torch.tensor(seq, dtype=torch.int32, device=dev)
    pos_t = torch.tensor(pos, dtype=torch.int32, device=dev)
    qn, qr = S.query_inputs(wl, device=dev)
    q_pos = torch.tensor(S.query_positions(wl), dtype=torch.int32, device=dev)
    seq_lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=dev)
    max_len = max(wl.seq_lens)
    n = ctx.prefill_mha_workspace_size(H, B, T, max_len)
    ws = torch.empty(((n + 15) // 16, 16), dtype=torch.uint8, device=dev)
    out = torch.empty(B, T, H, 128, dtype=torch.bfloat16, device=dev)
    scale = 1.0 / math.sqrt(192.0)

    def mha():
        ctx.prefill_mha(cache, w_uk, w_uv, qn, qr, q_pos, seq_lens, max_len, scale, workspace=ws, out=out)

    def step():
        ctx.append_latent(cache, c_new, k_new, seq_t, pos_t)
        mha()

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / steps

    step_s = timed(step)
    mha_s = timed(mha)
    pairs = sum(T * (L - T + 1) + T * (T - 1) // 2 for L in wl.seq_lens)
    flops = sum(wl.seq_lens) * 2 * H * 256 * 512 + 2 * H * 320 * pairs
    rec = {"workload": wl.name + "_mha", "path": "MHA form (mla_prefill_mha): append, K/V expansion, causal attention",
           "cache": "bf16", "B": B, "H": H, "Hq": T, "tokens": sum(wl.seq_lens), "paged": wl.paged,
           "us_per_step": round(step_s * 1e6, 2), "prefill_mha_us": round(mha_s * 1e6, 2),
           "prefill_mha_tflops": round(flops / mha_s / 1e12, 1), "prefill_mha_bound": "tensor",
           "prefill_mha_roofline_frac": round(flops / mha_s / 1e12 / tf, 3),
           "flops_per_call": flops,
           "chosen_form": m.prefill_choose_form(H, T, wl.seq_lens)[0],
           "status": ctx.device_status()}
    if check:
        torch.cuda.synchronize()
        rec["cpu_baseline"] = _cpu_workload_baseline(wl, gpu_out=out[0].double().cpu().numpy(), timing=False)
    del cache, ws, out
    torch.cuda.empty_cache()
    return rec


def _workload_record(b, total_ms, attn_ms, steps, peaks, n_gpus):
    hbm, tf, tfs, kind = peaks
    attn_bytes, attn_flops, step_bytes = b.algorithmic()
    step_s = total_ms / 1e3 / steps
    attn_s = statistics.mean(attn_ms) / 1e3
    t_hbm = attn_bytes / (hbm * 1e9)
    t_tc = attn_flops / (tf * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    return {
        "workload": b.name, "cache": "fp8" if b.fp8 else "bf16", "B": b.wl.B, "H": b.wl.H, "Hq": b.wl.Hq, "tokens": b.tokens,
        "paged": b.wl.paged,
        "us_per_step": round(step_s * 1e6, 2),
        "cache_GBps_step": round(n_gpus * b.cache_bytes / step_s / 1e9, 1),
        "decode_attn_us": round(attn_s * 1e6, 2),
        "decode_attn_us_median": round(statistics.median(attn_ms) * 1e3, 2),
        "decode_attn_cache_GBps": round(b.cache_bytes / attn_s / 1e9, 1),
        "decode_attn_bound": bound,
        "decode_attn_roofline_frac": round(max(t_hbm, t_tc) / attn_s, 3),
        "decode_attn_tflops": round(attn_flops / attn_s / 1e12, 1),
        # DRAM bytes of one attention launch from the committed ncu capture (null
        # when none covers this workload and these kernel sources)
        "decode_attn_traffic": (round(_traffic_per_token(b.name) * b.tokens)
                                if _traffic_per_token(b.name) else None),
    }


def run_gpu(args):
    import torch
    rank, world, local = _dist()
    _check_world(args, world)
    if torch.cuda.device_count() <= local:
        raise SystemExit(f"bench.py: rank {rank} needs GPU {local} but {torch.cuda.device_count()} are visible")
    dist = None
    if world > 1:
        import torch.distributed as td
        td.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        dist = td
    torch.cuda.set_device(local)
    import mla_absorbed_latent_02_gb300 as m
    import mla_synth as S
    m.build()
    ctx = m.Context(local, max_pos=131072)
    peaks = _peaks()
    hbm, tf, tfs, kind = peaks

    wl = S.make_config(1)
    b = Bench(m, S, torch, ctx, wl, f"cuda:{local}")
    clocks = Clocks(local)
    clocks.start()
    total_ms, attn_ms = b.time_steps(args.steps, args.warmup, dist)
    clk = clocks.stop()
    total_ms = reduce_max_over_ranks(total_ms, dist, f"cuda:{local}")
    step_s = total_ms / 1e3 / args.steps
    rec = _workload_record(b, total_ms, attn_ms, args.steps, peaks, world)
    attn_bytes, attn_flops, _ = b.algorithmic()
    attn_s = statistics.mean(attn_ms) / 1e3
    achieved = attn_bytes / attn_s / 1e9
    tpt = _traffic_per_token(b.name)
    e2e_s, h2d, d2h = b.time_e2e(max(10, args.steps), 3)
    try:
        direct_us = round(b.time_direct(args.steps), 2)   # this rank's, plain launches
    except Exception:
        direct_us = None

    if rank == 0 and not args.no_cpu:
        rec["cpu_baseline"] = _cpu_workload_baseline(wl, gpu_out=b.first_output())
    workloads = [rec]
    if not args.only_main and rank == 0:
        for wl2 in ([S.make_config(i) for i in (0, 2, 3, 4)]
                    + [S.make_prefill(4, 16, 64, 4096), S.make_prefill(1, 128, 1024, 1024)]):
            b2 = Bench(m, S, torch, ctx, wl2, f"cuda:{local}")
            tm, am = b2.time_steps(args.steps, args.warmup)
            rec2 = _workload_record(b2, tm, am, args.steps, peaks, 1)
            if wl2.Hq > 1:   # a prefill chunk: the form mla_prefill_choose_form picks for it
                rec2["chosen_form"] = m.prefill_choose_form(wl2.H, wl2.Hq, wl2.seq_lens)[0]
            if not args.no_cpu:
                rec2["cpu_baseline"] = _cpu_workload_baseline(wl2, gpu_out=b2.first_output())
            workloads.append(rec2)
            del b2
            torch.cuda.empty_cache()
        # the 1,024-token prompt again in the expanded (MHA) form, and 1,024-token
        # chunks of four sequences over 3,072 cached tokens each at H=16
        for wl2 in (S.make_prefill(1, 128, 1024, 1024), S.make_prefill(4, 16, 1024, 4096)):
            workloads.append(time_prefill_mha(m, S, torch, ctx, wl2, args.steps, args.warmup, peaks,
                                              check=not args.no_cpu))
        # the short single step also as one launch (mla_decode_step_small)
        wl2 = S.make_config(0)
        b2 = Bench(m, S, torch, ctx, wl2, f"cuda:{local}", small=True)
        tm, am = b2.time_steps(args.steps, args.warmup)
        rec2 = _workload_record(b2, tm, am, args.steps, peaks, 1)
        rec2["path"] = "one launch: append, absorb_q, attention and expand_v (decode_attn_us = the whole step)"
        if not args.no_cpu:
            rec2["cpu_baseline"] = _cpu_workload_baseline(wl2, gpu_out=b2.first_output(), timing=False)
        workloads.append(rec2)
        del b2
        # the same decode steps over the FP8 latent cache (656 bytes per token)
        for wl2 in [S.make_config(i) for i in (1, 2, 3)]:
            b2 = Bench(m, S, torch, ctx, wl2, f"cuda:{local}", fp8=True)
            tm, am = b2.time_steps(args.steps, args.warmup)
            rec2 = _workload_record(b2, tm, am, args.steps, peaks, 1)
            if not args.no_cpu:
                rec2["cpu_baseline"] = _cpu_workload_baseline(wl2, gpu_out=b2.first_output(), timing=False)
            workloads.append(rec2)
            del b2
            torch.cuda.empty_cache()
    extras = []
    if not args.only_main and rank == 0:
        extras.append(time_out_proj(m, S, torch, ctx, 64, 16, 2048, args.steps, peaks))
        extras.append(time_out_proj(m, S, torch, ctx, 32, 128, 7168, args.steps, peaks))
        extras.append(time_expand_out_proj(m, S, torch, ctx, 64, 16, 2048, args.steps, peaks))
        extras.append(time_expand_out_proj(m, S, torch, ctx, 32, 128, 7168, args.steps, peaks))
        extras.append(time_project_latent(m, S, torch, ctx, 64, 2048, args.steps, peaks))
        extras.append(time_project_latent(m, S, torch, ctx, 32, 7168, args.steps, peaks))
    status = ctx.device_status()

    if rank == 0:
        cpu = _cpu_baseline(args, wl, sample_seqs=args.cpu_seqs) if not args.no_cpu else None
        line = {
            "metric": METRIC,
            "value": round(job_gbps(b.cache_bytes, world, step_s), 1),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(step_s * 1e3, 5),
            "us_per_step": round(step_s * 1e6, 2),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
            "config": {"workload": "V2-Lite batched decode: B=64, H=16, Hq=1, L=4096, contiguous latent cache",
                       "B": wl.B, "H": wl.H, "Hq": wl.Hq, "L": 4096, "cache_MB": round(b.cache_bytes / 1e6, 1),
                       "l2": "inputs larger than L2 (302 MB latent cache streamed every step)",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"kernel": "decode_attn (attention + split-KV combine)", "bound": "hbm",
                         "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(achieved / hbm, 3), "peak_kind": kind,
                         "algorithmic_bytes_per_launch": attn_bytes,
                         "traffic": (round(tpt * b.tokens) if tpt else None)},
            "e2e": {"value": round(job_gbps(b.cache_bytes, world, reduce_max_over_ranks(e2e_s, dist, f"cuda:{local}")), 1),
                    "unit": "GB/s",
                    "us_per_step": round(e2e_s * 1e6, 2), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": b.launches_per_step * args.steps,
            "us_per_step_direct_launches": direct_us,
            "clocks": clk,
            "device_status": status,
            "workloads": workloads,
            "extras": extras,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line))
    ctx.close()
    if dist is not None:
        dist.destroy_process_group()


def _free_port() -> int:
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        return so.getsockname()[1]


def _launch_ranks(args) -> int:
    """`--gpus N` (N > 1) without a launcher: start N ranks of this script on
    this node, one per GPU, with the same arguments (torch.distributed.run,
    rendezvous on 127.0.0.1); returns the launcher's exit code. Refuses when
    fewer than N GPUs are visible."""
    if not args.dry and args.impl == "ours":
        import torch
        n = torch.cuda.device_count()
        if n < args.gpus:
            print(f"bench.py: --gpus {args.gpus} but {n} GPU(s) visible", file=sys.stderr)
            return 2
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def _check_world(args, world):
    if world != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but the launcher started {world} rank(s)")


def run_dry(args):
    """The multi-rank bookkeeping of run_gpu without a GPU: gloo process group,
    a made-up per-rank time ((rank + 1) ms per step), barrier, max over ranks, one
    line from rank 0. Nothing is measured; the line says so."""
    rank, world, local = _dist()
    _check_world(args, world)
    dist = None
    if world > 1:
        import torch.distributed as td
        td.init_process_group("gloo")
        dist = td
        dist.barrier()
    step_ms = reduce_max_over_ranks(float(rank + 1), dist, "cpu")
    if rank == 0:
        print(json.dumps({"dry_run": True, "measured": False, "n_gpus": world, "steps": args.steps,
                          "warmup": args.warmup, "max_rank_ms_per_step": step_ms,
                          "value_if_measured": round(job_gbps(301989888, world, step_ms / 1e3), 1)}))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def run_profile(args):
    """W untimed and K timed direct steps of one configuration (launches that a
    profiler attributes one by one)."""
    import torch
    import mla_absorbed_latent_02_gb300 as m
    import mla_synth as S
    m.build()
    ctx = m.Context(0, max_pos=131072)
    wl = S.make_config(args.profile_config)
    b = Bench(m, S, torch, ctx, wl, "cuda:0", fp8=args.fp8)
    for _ in range(args.warmup):
        b.step.run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        b.step.run()
    e1.record()
    torch.cuda.synchronize()
    status = ctx.device_status()
    print(json.dumps({"profile_config": args.profile_config, "workload": b.name, "steps": args.steps,
                      "us_per_step_direct": round(e0.elapsed_time(e1) * 1e3 / args.steps, 2),
                      "device_status": status}))
    ctx.close()
    if status != 0:
        sys.exit(1)


def run_profile_mha(args):
    """W untimed and K timed steps of the 1,024-token H=128 prompt through the
    MHA-form prefill (direct launches), then the call alone the same way."""
    import torch
    import mla_absorbed_latent_02_gb300 as m
    import mla_synth as S
    m.build()
    ctx = m.Context(0, max_pos=131072)
    rec = time_prefill_mha(m, S, torch, ctx, S.make_prefill(1, 128, 1024, 1024), args.steps, args.warmup, _peaks(),
                           check=False)
    status = ctx.device_status()
    print(json.dumps({"profile_mha": rec["workload"], "steps": args.steps, "us_per_step": rec["us_per_step"],
                      "prefill_mha_us": rec["prefill_mha_us"], "device_status": status}))
    ctx.close()
    if status != 0:
        sys.exit(1)


def run_profile_proj(args):
    """One projection on its own (the cases the bench's extras time): 0 and 1
    mla_out_proj at M=64, H=16, d_model=2048 and M=32, H=128, d_model=7168; 2 and
    3 mla_project_latent for 64 tokens at d_model=2048 and 32 at 7168. Three
    direct warm-up calls, one on a side stream, then a graph of K calls replayed
    twice."""
    import torch
    import mla_absorbed_latent_02_gb300 as m
    import mla_synth as S
    m.build()
    ctx = m.Context(0, max_pos=131072)
    peaks = _peaks()
    case = args.profile_proj
    if case in (0, 1):
        M, H, d = ((64, 16, 2048), (32, 128, 7168))[case]
        rec = time_out_proj(m, S, torch, ctx, M, H, d, args.steps, peaks)
    else:
        n, d = ((64, 2048), (32, 7168))[case - 2]
        rec = time_project_latent(m, S, torch, ctx, n, d, args.steps, peaks)
    status = ctx.device_status()
    rec["device_status"] = status
    print(json.dumps({"profile_proj": case, **rec}))
    ctx.close()
    if status != 0:
        sys.exit(1)


# --------------------------------------------------------------------------- oracle arm
def _cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _oracle_sequence(S, O, wl, b, inputs):
    import numpy as np
    import torch
    w_uk, w_uv, qn, qr = inputs
    c, k = S.token_inputs(wl, b, device="cpu")
    f = lambda t: O.bf16_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))
    qpos = [wl.seq_lens[b] - wl.Hq + j for j in range(wl.Hq)]
    t = time.perf_counter()
    O.naive_decode(f(c), f(k), qn[b], qr[b], w_uk, w_uv, 1.0 / math.sqrt(192.0), qpos)
    return time.perf_counter() - t, wl.seq_lens[b] * ROW_BYTES


def _cpu_baseline(args, wl, sample_seqs=4):
    """The float64 naive oracle (the oracle of record) on a bounded sample:
    `sample_seqs` sequences of the workload, every head."""
    import numpy as np
    import torch
    import mla_synth as S
    import oracle as O
    f = lambda t: O.bf16_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))
    w_uk, w_uv = [f(w) for w in S.weights(wl)]
    qn, qr = [f(q) for q in S.query_inputs(wl)]
    tot_t = tot_b = 0.0
    for b in range(sample_seqs):
        dt, nb = _oracle_sequence(S, O, wl, b, (w_uk, w_uv, qn, qr))
        tot_t += dt
        tot_b += nb
    return {"value": round(tot_b / tot_t / 1e9, 6), "unit": "GB/s", "cores": _cpu_cores(), "kind": "oracle",
            "sample": f"float64 naive MLA decode (expand K,V per head, then softmax attention) of {sample_seqs} "
                      f"of the {wl.B} sequences, all {wl.H} heads, L={wl.seq_lens[0]}; {tot_t:.1f} s of CPU time",
            "us_per_step_extrapolated": round(tot_t / sample_seqs * wl.B * 1e6, 1)}


def _cpu_workload_baseline(wl, budget_s=2.0, gpu_out=None, timing=True):
    """The oracle on the host cores for one decode workload (float64, the same
    seeded inputs as the GPU run), bounded in time:
      absorbed: ``absorbed_decode`` over every (b, j, h) of the first sequences
        of the batch, in order, until ``budget_s`` of oracle time (or all of them);
      naive: ``naive_decode`` (K and V expanded per head, then softmax
        attention) on the first sequence for as many heads as ~2e9 multiply-adds
        of expansion allow.
    Each is scaled to the whole step by its share of the work (attended
    (query, token) pairs x heads) and labelled "extrapolated" when sampled.
    Input generation is not timed. ``gpu_out``: the GPU step's output of the
    first sequence ([Hq, H, 128], float64), checked against the float64
    absorbed oracle on the same bf16 inputs (max-abs and relative L2 error;
    for an FP8 cache this includes the format's rounding of the latent).
    ``timing=False``: the check only."""
    import numpy as np
    import torch
    import mla_synth as S
    import oracle as O
    f = lambda t: O.bf16_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))
    w_uk, w_uv = [f(w) for w in S.weights(wl)]
    qn, qr = [f(q) for q in S.query_inputs(wl)]
    scale = 1.0 / math.sqrt(192.0)
    pairs = lambda L: (wl.Hq * (L - wl.Hq + 1) + wl.Hq * (wl.Hq - 1) // 2) if L >= wl.Hq else 0
    total = sum(pairs(L) for L in wl.seq_lens)
    t_abs, done, nseq = 0.0, 0, 0
    first = None
    check = None
    for b in range(wl.B):
        L = wl.seq_lens[b]
        if L < wl.Hq:
            continue
        c, k = S.token_inputs(wl, b, device="cpu")
        c, k = f(c), f(k)
        qpos = [L - wl.Hq + j for j in range(wl.Hq)]
        t = time.perf_counter()
        o_ref, _, _ = O.absorbed_decode(c, k, qn[b], qr[b], w_uk, w_uv, scale, qpos)
        t_abs += time.perf_counter() - t
        done += pairs(L)
        nseq += 1
        if first is None:
            first = (b, L, c, k, qpos)
            if gpu_out is not None:
                d = np.asarray(gpu_out, np.float64) - o_ref
                check = {"seq": b, "max_abs": float(f"{np.max(np.abs(d)):.3e}"),
                         "rel_l2": float(f"{np.linalg.norm(d) / np.linalg.norm(o_ref):.3e}"),
                         "vs": "float64 absorbed oracle on the bf16 inputs"}
            if not timing:
                return {"kind": "oracle", "check_vs_bf16_oracle": check}
        if t_abs >= budget_s:
            break
    b, L, c, k, qpos = first
    nh = max(1, min(wl.H, int(2e9 // (2 * 128 * 512 * L))))
    t = time.perf_counter()
    O.naive_decode(c, k, qn[b], qr[b], w_uk, w_uv, scale, qpos, heads=list(range(nh)))
    t_naive = time.perf_counter() - t
    naive_step = t_naive * (total / pairs(L)) * (wl.H / nh)
    return {"kind": "oracle", "cores": _cpu_cores(), "check_vs_bf16_oracle": check,
            "absorbed_us_per_step": round(t_abs * total / done * 1e6, 1),
            "absorbed_sample": f"absorbed_decode, {nseq} of {wl.B} sequences, all {wl.Hq}x{wl.H} query rows; "
                               f"{t_abs:.2f} s" + (", extrapolated to the step" if nseq < wl.B else ""),
            "naive_us_per_step": round(naive_step * 1e6, 1),
            "naive_sample": f"naive_decode, sequence {b} (L={L}), {nh} of {wl.H} heads; {t_naive:.2f} s, "
                            f"extrapolated to the step" if (nh < wl.H or wl.B > 1) else
                            f"naive_decode, the whole step; {t_naive:.2f} s"}


def run_reference(args):
    rank, world, local = _dist()
    if rank != 0:
        return
    import mla_synth as S
    wl = S.make_config(1)
    import numpy as np
    import torch
    import oracle as O
    f = lambda t: O.bf16_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))
    w_uk, w_uv = [f(w) for w in S.weights(wl)]
    qn, qr = [f(q) for q in S.query_inputs(wl)]
    inputs = (w_uk, w_uv, qn, qr)
    for i in range(args.warmup):
        _oracle_sequence(S, O, wl, i % wl.B, inputs)
    ts, nbytes = [], 0
    for i in range(args.steps):
        dt, nb = _oracle_sequence(S, O, wl, i % wl.B, inputs)
        ts.append(dt)
        nbytes += nb
    tot = sum(ts)
    value = nbytes / tot / 1e9
    sample = (f"each step: float64 naive MLA decode of one of the {wl.B} sequences (all {wl.H} heads, "
              f"L={wl.seq_lens[0]}) on the host CPU")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
        "config": {"workload": "V2-Lite batched decode: B=64, H=16, Hq=1, L=4096, contiguous latent cache",
                   "B": wl.B, "H": wl.H, "Hq": wl.Hq, "L": 4096, "sample": "one sequence per step"},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": _cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--only-main", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--cpu-seqs", type=int, default=64,
                    help="sequences of the workload the oracle baseline runs (64 = the whole step)")
    ap.add_argument("--profile-config", type=int, default=None,
                    help="profiling aid: run W+K direct (non-graph) steps of configuration N and print "
                         "their mean time; no contract line")
    ap.add_argument("--fp8", action="store_true", help="with --profile-config: use the FP8 latent cache")
    ap.add_argument("--profile-mha", action="store_true",
                    help="profiling aid: W+K direct steps of the 1,024-token H=128 prompt through the MHA-form "
                         "prefill, then the call alone; no contract line")
    ap.add_argument("--profile-proj", type=int, default=None, choices=[0, 1, 2, 3],
                    help="profiling aid: one projection on its own (0/1: mla_out_proj at V2-Lite / V3 width, "
                         "2/3: mla_project_latent); no contract line")
    ap.add_argument("--dry", action="store_true",
                    help="host-only check of the multi-rank plumbing (gloo, no GPU, no timing): each rank "
                         "reports a made-up time, rank 0 prints one line with n_gpus and the max over ranks")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(_launch_ranks(args))
    if args.dry:
        run_dry(args)
    elif args.profile_config is not None:
        run_profile(args)
    elif args.profile_mha:
        run_profile_mha(args)
    elif args.profile_proj is not None:
        run_profile_proj(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
