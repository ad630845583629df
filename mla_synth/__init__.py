"""Seeded synthetic inputs for the absorbed-MLA decode path.

This module only draws numbers. It holds none of the method's arithmetic and is
shared by the tests, the benchmark and the oracle checks, so that the CUDA path
and the oracle always see the same input bits.

Generator (counter based, so any slice can be drawn on its own and on any
device): element ``i`` of stream ``k`` uses two 64-bit words
``splitmix64(k + 2*i)`` and ``splitmix64(k + 2*i + 1)`` (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", 2014). Their top 53 bits give
``u1, u2`` in [0, 1); one standard normal is ``sqrt(-2 ln(1-u1)) * cos(2 pi u2)``
(Box and Muller, 1958), computed in float64, scaled by ``std``, rounded to float32
and then to bfloat16 with round-to-nearest-even. The stream key ``k`` is a
splitmix64 hash of the seed and the tensor's name.

Integer draws (lengths, permutations) use the same words: ``1 + (w >> 11) % n``
for a uniform integer in [1, n] and a Fisher-Yates shuffle for permutations.

Workload recipes (``make_config``) follow the five decode configurations of the
absorbed-MLA study: V2-Lite (H=16) and DeepSeek-V2/V3-size (H=128) heads,
d_nope=128, d_rope=64, d_c=512, d_v=128, activations N(0,1), weights N(0,0.02),
RoPE base 10000, softmax scale 1/sqrt(192), seed 0.
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field

import torch

_MASK64 = (1 << 64) - 1


def _s64(v: int) -> int:
    """Unsigned 64-bit constant as the signed int64 torch stores."""
    v &= _MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


_GOLDEN = _s64(0x9E3779B97F4A7C15)
_M1 = _s64(0xBF58476D1CE4E5B9)
_M2 = _s64(0x94D049BB133111EB)


def _lsr(x: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (x >> k) & ((1 << (64 - k)) - 1)


def splitmix64(x: torch.Tensor) -> torch.Tensor:
    """splitmix64 finaliser on int64 tensors (wrapping arithmetic)."""
    z = x + _GOLDEN
    z = (z ^ _lsr(z, 30)) * _M1
    z = (z ^ _lsr(z, 27)) * _M2
    return z ^ _lsr(z, 31)


def _splitmix64_int(x: int) -> int:
    z = (x + 0x9E3779B97F4A7C15) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, name: str) -> int:
    """Key of the named stream (a python int, used as a signed int64)."""
    return _s64(_splitmix64_int((seed * 0x100000001B3) ^ zlib.crc32(name.encode())))


def _words(key: int, start: int, count: int, device) -> torch.Tensor:
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)
    return splitmix64(idx + key)


def f32_to_bf16_bits_rne(x: torch.Tensor) -> torch.Tensor:
    """float32 -> bfloat16 bit pattern (int16 view), round to nearest even."""
    u = x.contiguous().view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    r = torch.where(torch.isnan(x), torch.full_like(r, 0x7FC0), r)
    return (r & 0xFFFF).to(torch.int32).to(torch.int16)


def normal_bf16(seed: int, name: str, shape, std: float = 1.0, device="cpu",
                offset: int = 0) -> torch.Tensor:
    """bfloat16 tensor of N(0, std^2) draws, elements ``offset ..`` of the stream."""
    n = 1
    for s in shape:
        n *= int(s)
    key = stream_key(seed, name)
    w = _words(key, 2 * offset, 2 * n, device).view(n, 2)
    u1 = _lsr(w[:, 0], 11).to(torch.float64) * (1.0 / 9007199254740992.0)
    u2 = _lsr(w[:, 1], 11).to(torch.float64) * (1.0 / 9007199254740992.0)
    z = torch.sqrt(-2.0 * torch.log1p(-u1)) * torch.cos((2.0 * math.pi) * u2)
    z = (z * std).to(torch.float32)
    return f32_to_bf16_bits_rne(z).view(torch.bfloat16).view(*shape)


def normal_bf16_chunked(seed, name, shape, std=1.0, device="cpu", chunk=1 << 24):
    """Same values as ``normal_bf16`` but drawn in chunks to bound temporaries."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for o in range(0, n, chunk):
        c = min(chunk, n - o)
        out[o:o + c] = normal_bf16(seed, name, (c,), std, device, offset=o)
    return out.view(*shape)


def uniform_ints(seed: int, name: str, n: int, lo: int, hi: int) -> list:
    """n integers uniform on [lo, hi] (inclusive)."""
    key = stream_key(seed, name)
    span = hi - lo + 1
    out = []
    for i in range(n):
        w = _splitmix64_int((key + i) & _MASK64)
        out.append(lo + (w >> 11) % span)
    return out


def permutation(seed: int, name: str, n: int) -> list:
    """Fisher-Yates permutation of 0..n-1."""
    key = stream_key(seed, name)
    p = list(range(n))
    for i in range(n - 1, 0, -1):
        w = _splitmix64_int((key + i) & _MASK64)
        j = (w >> 11) % (i + 1)
        p[i], p[j] = p[j], p[i]
    return p


# ---------------------------------------------------------------------------
# Workload recipes
# ---------------------------------------------------------------------------

D_NOPE, D_ROPE, D_C, D_V = 128, 64, 512, 128
ROW = D_C + D_ROPE  # 576 elements per cached token
BLOCK = 64          # paged-cache block size (tokens)
ROPE_BASE = 10000.0
SCALE = 1.0 / math.sqrt(D_NOPE + D_ROPE)


@dataclass
class Workload:
    """Shape and cache layout of one decode workload (no tensors)."""
    name: str
    B: int
    H: int
    Hq: int
    seq_lens: list
    paged: bool
    capacity: int = 0            # contiguous: rows per sequence
    block_table: list = field(default_factory=list)  # paged: per sequence block ids
    num_blocks: int = 0
    max_blocks: int = 0
    seed: int = 0

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seq_lens))


def _paged_tables(seed, name, seq_lens):
    nblk = [(L + BLOCK - 1) // BLOCK for L in seq_lens]
    total = sum(nblk)
    perm = permutation(seed, name + "/block_perm", total)
    tables, o = [], 0
    for n in nblk:
        tables.append(perm[o:o + n])
        o += n
    return tables, total, max(nblk)


def make_config(idx: int, seed: int = 0, scale_down: int = 1) -> Workload:
    """The five decode workloads; ``scale_down`` divides lengths (for quick tests)."""
    if idx == 0:
        return Workload("v2lite_b1_h16_l26", 1, 16, 1, [26], False, capacity=32, seed=seed)
    if idx == 1:
        L = max(1, 4096 // scale_down)
        return Workload("v2lite_b64_h16_l4096", 64, 16, 1, [L] * 64, False, capacity=L, seed=seed)
    if idx == 2:
        L = max(1, 8192 // scale_down)
        lens = [L] * 32
        tbl, nb, mb = _paged_tables(seed, "cfg2", lens)
        return Workload("v3_b32_h128_l8192_paged", 32, 128, 1, lens, True,
                        block_table=tbl, num_blocks=nb, max_blocks=mb, seed=seed)
    if idx == 3:
        lens = uniform_ints(seed, "cfg3/seq_lens", 128, 1, max(1, 32768 // scale_down))
        tbl, nb, mb = _paged_tables(seed, "cfg3", lens)
        return Workload("v3_b128_h128_ragged32k_paged", 128, 128, 1, lens, True,
                        block_table=tbl, num_blocks=nb, max_blocks=mb, seed=seed)
    if idx == 4:
        L = max(2, 131072 // scale_down)
        lens = [L] * 4
        tbl, nb, mb = _paged_tables(seed, "cfg4", lens)
        return Workload("v3_b4_hq2_h128_l131072_paged", 4, 128, 2, lens, True,
                        block_table=tbl, num_blocks=nb, max_blocks=mb, seed=seed)
    raise ValueError(idx)


def make_prefill(B: int = 4, H: int = 16, chunk: int = 64, L: int = 4096, seed: int = 0) -> Workload:
    """A chunked-prefill step: ``chunk`` new tokens at the end of each of B
    sequences of length L (contiguous cache), every one of them a query."""
    return Workload(f"prefill{chunk}_b{B}_h{H}_l{L}", B, H, chunk, [L] * B, False, capacity=L, seed=seed)


def token_inputs(wl: Workload, b: int, device="cpu", t0: int = 0, t1=None):
    """Pre-RoPE latent rows of sequence ``b`` for tokens [t0, t1): (c_kv, k_rope)."""
    L = wl.seq_lens[b]
    t1 = L if t1 is None else t1
    n = t1 - t0
    c = normal_bf16(wl.seed, f"c_kv/{b}", (n, D_C), device=device, offset=t0 * D_C)
    k = normal_bf16(wl.seed, f"k_rope/{b}", (n, D_ROPE), device=device, offset=t0 * D_ROPE)
    return c, k


def query_inputs(wl: Workload, device="cpu"):
    """(q_nope [B,Hq,H,128], q_rope [B,Hq,H,64]) pre-RoPE queries."""
    qn = normal_bf16(wl.seed, "q_nope", (wl.B, wl.Hq, wl.H, D_NOPE), device=device)
    qr = normal_bf16(wl.seed, "q_rope", (wl.B, wl.Hq, wl.H, D_ROPE), device=device)
    return qn, qr


def weights(wl: Workload, device="cpu"):
    """(W_UK, W_UV), each [H, 128, 512] ~ N(0, 0.02^2)."""
    wuk = normal_bf16(wl.seed, f"W_UK/H{wl.H}", (wl.H, D_NOPE, D_C), std=0.02, device=device)
    wuv = normal_bf16(wl.seed, f"W_UV/H{wl.H}", (wl.H, D_V, D_C), std=0.02, device=device)
    return wuk, wuv


def query_positions(wl: Workload):
    """Absolute position of query j of sequence b: L_b - Hq + j."""
    return [[wl.seq_lens[b] - wl.Hq + j for j in range(wl.Hq)] for b in range(wl.B)]
