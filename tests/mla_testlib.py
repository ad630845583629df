"""Helpers shared by the GPU parity tests: seeded inputs, the CUDA path through
the C ABI, and the oracle on the same input bits."""
from __future__ import annotations

import math

import numpy as np
import torch

import mla_synth as S
import oracle as O

SCALE = 1.0 / math.sqrt(192.0)
# GPU vs oracle bars for floating-point outputs (bf16 inputs, fp32 accumulation)
MAX_ABS = 1e-2
REL_L2 = 5e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (CPU)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return O.bf16_to_f64(bits(t))
    return t.detach().cpu().double().numpy()


def rel_l2(got, want) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def assert_close(got, want, max_abs=MAX_ABS, rel=REL_L2, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    ma = float(np.max(np.abs(got - want))) if got.size else 0.0
    r = rel_l2(got, want) if got.size else 0.0
    assert ma <= max_abs and r <= rel, f"{what}: max_abs={ma:.3e} (<= {max_abs}), rel_l2={r:.3e} (<= {rel})"
    return ma, r


class Problem:
    """One workload's inputs on the GPU plus host copies for the oracle."""

    def __init__(self, wl: S.Workload, device="cuda", keep_host=True, gen_device=None):
        self.wl = wl
        dev = torch.device(device)
        gen = gen_device or device
        self.gen_device = gen
        B, H, Hq = wl.B, wl.H, wl.Hq
        self.w_uk, self.w_uv = [w.to(dev) for w in S.weights(wl, device=gen)]
        qn, qr = S.query_inputs(wl, device=gen)
        self.q_nope, self.q_rope = qn.to(dev), qr.to(dev)
        self.q_pos = torch.tensor(S.query_positions(wl), dtype=torch.int32, device=dev)
        self.seq_lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=dev)
        self.host = {}
        if keep_host:
            self.host["w_uk"] = f64(self.w_uk)
            self.host["w_uv"] = f64(self.w_uv)
            self.host["q_nope"] = f64(self.q_nope)
            self.host["q_rope"] = f64(self.q_rope)

    def token_inputs(self, b, t0=0, t1=None):
        """Raw (c_kv, k_rope) of sequence b, drawn on the generating device and
        returned on the CPU: the same bits the cache was filled with."""
        c, k = S.token_inputs(self.wl, b, device=self.gen_device, t0=t0, t1=t1)
        return c.cpu(), k.cpu()


def make_cache(ctx_mod, wl: S.Workload, device="cuda", fp8=False):
    if wl.paged:
        bt = torch.full((wl.B, wl.max_blocks), -1, dtype=torch.int32)
        for b, row in enumerate(wl.block_table):
            bt[b, :len(row)] = torch.tensor(row, dtype=torch.int32)
        return ctx_mod.Cache.paged_pool(wl.num_blocks, bt, device=device, fp8=fp8)
    return ctx_mod.Cache.contiguous(wl.B, wl.capacity, device=device, fp8=fp8)


def fill_cache(ctx, cache, prob: Problem, chunk_tokens=1 << 20):
    """Append every token of every sequence through mla_append_latent."""
    wl = prob.wl
    dev = cache.storage.device
    for b in range(wl.B):
        L = wl.seq_lens[b]
        for t0 in range(0, L, chunk_tokens):
            t1 = min(L, t0 + chunk_tokens)
            c, k = S.token_inputs(wl, b, device=prob.gen_device, t0=t0, t1=t1)
            n = t1 - t0
            seq = torch.full((n,), b, dtype=torch.int32, device=dev)
            pos = torch.arange(t0, t1, dtype=torch.int32, device=dev)
            ctx.append_latent(cache, c.to(dev).contiguous(), k.to(dev).contiguous(), seq, pos)


def gpu_step(ctx, cache, prob: Problem, scale=SCALE):
    out, o_lat, lse = ctx.decode_step(cache, prob.w_uk, prob.w_uv, prob.q_nope, prob.q_rope, prob.q_pos,
                                      prob.seq_lens, scale)
    torch.cuda.synchronize()
    return out, o_lat, lse


def oracle_absorbed(prob: Problem, b: int, scale=SCALE):
    """(o [Hq,H,128], o_lat [Hq,H,512], lse [Hq,H]) of sequence b from the raw inputs."""
    wl, h = prob.wl, prob.host
    c, k = prob.token_inputs(b)
    qpos = [wl.seq_lens[b] - wl.Hq + j for j in range(wl.Hq)]
    return O.absorbed_decode(f64(c), f64(k), h["q_nope"][b], h["q_rope"][b], h["w_uk"], h["w_uv"], scale, qpos)


def oracle_absorbed_fp8(prob: Problem, b: int, scale=SCALE):
    """oracle_absorbed over the FP8 cache: the latent each token's FP8 row stands
    for (codes * sigma, written by the oracle's FP8 row writer) in place of c_kv."""
    wl, h = prob.wl, prob.host
    c, k = prob.token_inputs(b)
    L = wl.seq_lens[b]
    c_deq = O.fp8_rows_dequantize(O.fp8_cache_rows(bits(c), bits(k), np.arange(L)))[:, :512]
    qpos = [L - wl.Hq + j for j in range(wl.Hq)]
    return O.absorbed_decode(c_deq, f64(k), h["q_nope"][b], h["q_rope"][b], h["w_uk"], h["w_uv"], scale, qpos)


def oracle_naive(prob: Problem, b: int, heads, scale=SCALE):
    wl, h = prob.wl, prob.host
    c, k = prob.token_inputs(b)
    qpos = [wl.seq_lens[b] - wl.Hq + j for j in range(wl.Hq)]
    o, _ = O.naive_decode(f64(c), f64(k), h["q_nope"][b], h["q_rope"][b], h["w_uk"], h["w_uv"], scale, qpos,
                          heads=heads)
    return o
