"""Reference oracle for absorbed-latent MLA decode -- TEST INFRASTRUCTURE ONLY.

Plain, slow, float64 numpy. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module; the library never does, and this module
imports nothing from the library. Both sides share only the seeded input
generator (``mla_synth``), which holds none of the method's arithmetic.

Sources (cited by page title and section):
  * "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" (llm-atlas,
    DEEPSEEK_MLA_ABSORB_AUDIT) -- below "MLA absorb audit".
  * "80 行 PyTorch 从零写 DeepSeek 的 MLA" (CSDN) -- below "80-line PyTorch MLA".
  * "DeepSeek-V2-Lite 真实权重执行审计" (llm-atlas, DEEPSEEK_V2_LITE_TRACE) --
    below "V2-Lite trace audit".

What is computed, per sequence, query token j and head h:
  naive form (MLA absorb audit §2.1; 80-line PyTorch MLA §2 and Appendix A):
      k_t = [W_UK[h] c_t ; RoPE_t(k_rope_t)],  v_t = W_UV[h] c_t,
      s_t = scale * (q_nope . k_t[:128] + RoPE_pos(q_rope) . k_t[128:]),
      p = softmax(s over t <= pos_j),  o = sum_t p_t v_t.
  absorbed form (MLA absorb audit §2.2-§2.4; 80-line PyTorch MLA §4-§5):
      q_lat = W_UK[h]^T q_nope,  s_t = scale * (q_lat . c_t + q_rope' . k_rope'_t),
      o_lat = sum_t p_t c_t,  o = W_UV[h] o_lat.

Every function here is pinned by the not-gpu tests against values the pages
print, closed forms, invariants, special cases and brute force; see the pins in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import math

import numpy as np

D_NOPE = 128
D_ROPE = 64
D_C = 512
D_V = 128
ROW = D_C + D_ROPE


# ---------------------------------------------------------------------------
# bfloat16 <-> float
# ---------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bfloat16 bit patterns (uint16) as float64."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def f32_to_bf16(x) -> np.ndarray:
    """float32 -> bfloat16 bits, round to nearest, ties to even (NaN -> 0x7FC0)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    r = np.where(np.isnan(x), np.uint64(0x7FC0), r)
    return r.astype(np.uint16)


# ---------------------------------------------------------------------------
# RoPE: interleaved pairs (x[2i], x[2i+1]), inverse frequency 1/base^(2i/d)
# (80-line PyTorch MLA, Appendix A: rotate_half / apply_rope / build_rope;
#  the decoupled 64-dim RoPE key, MLA absorb audit §2.4)
# ---------------------------------------------------------------------------

def rope_inv_freq(d_r: int = D_ROPE, base: float = 10000.0) -> np.ndarray:
    """theta_i = 1 / base^(2i/d_r), i = 0 .. d_r/2-1, in float64 (libm pow)."""
    return np.array([1.0 / (base ** ((2 * i) / d_r)) for i in range(d_r // 2)],
                    dtype=np.float64)


def rope_angles(pos, d_r: int = D_ROPE, base: float = 10000.0) -> np.ndarray:
    """phi[n, i] = pos[n] * theta_i in float64."""
    inv = rope_inv_freq(d_r, base)
    pos = np.asarray(pos, dtype=np.float64).reshape(-1)
    return pos[:, None] * inv[None, :]


def rope_f64(x, pos, base: float = 10000.0) -> np.ndarray:
    """Exact-arithmetic RoPE of rows x[n, :] at positions pos[n].

    Pair i of row n turns (a, b) = (x[2i], x[2i+1]) into
    (a cos phi - b sin phi, b cos phi + a sin phi), phi = pos[n] * theta_i.
    ``x`` may carry extra leading axes after n (e.g. [n, heads, d_r]).
    """
    x = np.asarray(x, dtype=np.float64)
    d_r = x.shape[-1]
    phi = rope_angles(pos, d_r, base)                     # [n, d_r/2]
    shp = (phi.shape[0],) + (1,) * (x.ndim - 2) + (d_r // 2,)
    c = np.vectorize(math.cos)(phi).reshape(shp)
    s = np.vectorize(math.sin)(phi).reshape(shp)
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = b * c + a * s
    return out


def rope_cos_sin_f32(pos, d_r: int = D_ROPE, base: float = 10000.0):
    """The cache-write contract's float32 table: RNE(cos(phi)), RNE(sin(phi)).

    cos/sin are libm's double-precision functions of the float64 angle; each is
    rounded once to float32.
    """
    phi = rope_angles(pos, d_r, base)
    c = np.vectorize(math.cos)(phi).astype(np.float32)
    s = np.vectorize(math.sin)(phi).astype(np.float32)
    return c, s


def rope_f32_contract(x_bits, pos, base: float = 10000.0) -> np.ndarray:
    """Bit-exact RoPE of bfloat16 rows: the bytes the cache writer must store.

    With the float32 table (c, s) and float32 operands a, b taken exactly from
    bf16: y0 = f32(f32(a*c) - f32(b*s)), y1 = f32(f32(b*c) + f32(a*s)), each a
    separately rounded IEEE operation (no fused multiply-add), then RNE to bf16.
    ``x_bits`` is uint16 [n, ..., d_r]; positions index the first axis.
    """
    x32 = bf16_to_f64(x_bits).astype(np.float32)
    d_r = x32.shape[-1]
    c, s = rope_cos_sin_f32(pos, d_r, base)
    shp = (c.shape[0],) + (1,) * (x32.ndim - 2) + (d_r // 2,)
    c, s = c.reshape(shp), s.reshape(shp)
    a, b = x32[..., 0::2], x32[..., 1::2]
    y = np.empty_like(x32)
    y[..., 0::2] = np.subtract(np.multiply(a, c, dtype=np.float32),
                               np.multiply(b, s, dtype=np.float32), dtype=np.float32)
    y[..., 1::2] = np.add(np.multiply(b, c, dtype=np.float32),
                          np.multiply(a, s, dtype=np.float32), dtype=np.float32)
    return f32_to_bf16(y)


# ---------------------------------------------------------------------------
# Cache writer: one 576-element row per token = [c_kv (512) | RoPE(k_rope) (64)]
# (MLA absorb audit §2.4 and §4.1; V2-Lite trace audit §3.1-§3.2)
# ---------------------------------------------------------------------------

def cache_rows(c_kv_bits, k_rope_bits, pos, base: float = 10000.0) -> np.ndarray:
    """uint16 [n, 576]: the latent copied verbatim, the rope key rotated at pos."""
    c = np.asarray(c_kv_bits).astype(np.uint16)
    kr = rope_f32_contract(k_rope_bits, pos, base)
    return np.concatenate([c, kr], axis=1)


def contiguous_row(seq: int, pos: int, capacity: int) -> int:
    """Row of (seq, pos) in a contiguous [B, capacity, 576] cache."""
    return seq * capacity + pos


def paged_row(seq: int, pos: int, block_table, block: int = 64) -> int:
    """Row of (seq, pos) in a paged pool [num_blocks, block, 576]."""
    return int(block_table[seq][pos // block]) * block + pos % block


# ---------------------------------------------------------------------------
# Byte accounting (MLA absorb audit §0 and §4; V2-Lite trace audit §3.2;
# 80-line PyTorch MLA §1)
# ---------------------------------------------------------------------------

def latent_cache_bytes(L: int, d_c: int = D_C, d_r: int = D_ROPE, elem: int = 2) -> int:
    """Shared latent plus shared rope key: L * (d_c + d_r) elements."""
    return L * (d_c + d_r) * elem


def expanded_cache_bytes(L: int, H: int, d_nope: int = D_NOPE, d_r: int = D_ROPE,
                         d_v: int = D_V, elem: int = 2):
    """Naive per-head cache: key H*(d_nope+d_r) and value H*d_v elements per token.

    Returns (key_bytes, value_bytes, total_bytes).
    """
    k = L * H * (d_nope + d_r) * elem
    v = L * H * d_v * elem
    return k, v, k + v


def kv_bytes_per_token(kind: str, n_h: int = 128, d_h: int = 128, n_kv: int = 8,
                       d_c: int = D_C, d_r: int = D_ROPE, elem: int = 2) -> int:
    """Per-layer, per-token cache bytes for MHA, GQA and MLA (80-line PyTorch MLA §1)."""
    if kind == "mha":
        return 2 * n_h * d_h * elem
    if kind == "gqa":
        return 2 * n_kv * d_h * elem
    if kind == "mla":
        return (d_c + d_r) * elem
    raise ValueError(kind)


# ---------------------------------------------------------------------------
# Attention forms
# ---------------------------------------------------------------------------

def _softmax(s: np.ndarray) -> np.ndarray:
    m = np.max(s)
    e = np.exp(s - m)
    return e / np.sum(e)


def naive_decode(c_kv, k_rope_raw, q_nope, q_rope_raw, W_UK, W_UV, scale, q_pos,
                 heads=None, base: float = 10000.0):
    """Naive MLA decode of one sequence in float64 (the oracle of record).

    c_kv [L, 512] and k_rope_raw [L, 64] are the cached latent and the pre-RoPE
    rope key of tokens 0..L-1 (token t sits at position t). q_nope [Hq, H, 128] and
    q_rope_raw [Hq, H, 64] are the pre-RoPE queries; query j sits at q_pos[j] and
    attends tokens t <= q_pos[j]. W_UK, W_UV are [H, 128, 512] (nn.Linear weight of
    d_c -> H*128, viewed per head).

    Per head, keys and values are expanded from the latent first
    (MLA absorb audit §2.1; 80-line PyTorch MLA §2 and §3):
        k_t = [W_UK[h] c_t ; RoPE_t(k_rope_t)], v_t = W_UV[h] c_t,
    then plain softmax attention.

    Returns (o [Hq, nh, 128], probs) with probs[j][i] the softmax row of head
    heads[i].
    """
    c = np.asarray(c_kv, dtype=np.float64)
    L = c.shape[0]
    kr = rope_f64(k_rope_raw, np.arange(L), base)          # [L, 64]
    qn = np.asarray(q_nope, dtype=np.float64)
    Hq, H = qn.shape[0], qn.shape[1]
    qr = rope_f64(np.asarray(q_rope_raw, dtype=np.float64), np.asarray(q_pos), base)
    heads = list(range(H)) if heads is None else list(heads)
    o = np.zeros((Hq, len(heads), W_UV.shape[1]))
    probs = [[None] * len(heads) for _ in range(Hq)]
    for hi, h in enumerate(heads):
        k_nope = c @ np.asarray(W_UK[h], dtype=np.float64).T   # [L, 128]
        v = c @ np.asarray(W_UV[h], dtype=np.float64).T        # [L, 128]
        k = np.concatenate([k_nope, kr], axis=1)              # [L, 192]
        for j in range(Hq):
            n = int(q_pos[j]) + 1
            q = np.concatenate([qn[j, h], qr[j, h]])
            s = scale * (k[:n] @ q)
            p = _softmax(s)
            probs[j][hi] = p
            o[j, hi] = p @ v[:n]
    return o, probs


def naive_prefill_causal(c_kv, k_rope_raw, q_nope, q_rope_raw, W_UK, W_UV, scale,
                         base: float = 10000.0):
    """One-shot causal forward over L tokens with queries at positions 0..L-1.

    Matrix form of the naive path with a causal mask: the one-shot side of the
    prefill+decode equivalence check (80-line PyTorch MLA §2, cache equivalence
    test; MLA absorb audit §3.4). q_nope [L, H, 128], q_rope_raw [L, H, 64].
    Returns o [L, H, 128].
    """
    c = np.asarray(c_kv, dtype=np.float64)
    L = c.shape[0]
    kr = rope_f64(k_rope_raw, np.arange(L), base)
    qr = rope_f64(np.asarray(q_rope_raw, dtype=np.float64), np.arange(L), base)
    qn = np.asarray(q_nope, dtype=np.float64)
    H = qn.shape[1]
    o = np.zeros((L, H, W_UV.shape[1]))
    mask = np.tril(np.ones((L, L), dtype=bool))
    for h in range(H):
        K = np.concatenate([c @ np.asarray(W_UK[h], np.float64).T, kr], axis=1)
        V = c @ np.asarray(W_UV[h], np.float64).T
        Q = np.concatenate([qn[:, h], qr[:, h]], axis=1)
        S = scale * (Q @ K.T)
        S = np.where(mask, S, -np.inf)
        S = S - S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P = P / P.sum(axis=1, keepdims=True)
        o[:, h] = P @ V
    return o


def absorb_query(q_nope, W_UK) -> np.ndarray:
    """q_lat[..., h, :] = W_UK[h]^T q_nope[..., h, :]  (512 <- 128).

    Key absorption: q^T (W c) = (W^T q)^T c (MLA absorb audit §2.2; 80-line
    PyTorch MLA §4, path B).
    """
    qn = np.asarray(q_nope, dtype=np.float64)
    W = np.asarray(W_UK, dtype=np.float64)
    return np.einsum("...hd,hdc->...hc", qn, W)


def latent_attention(q_abs, rows, scale, limits, d_c: int = D_C):
    """Attention of G queries over the 576-wide latent rows (MQA form).

    q_abs [G, 576] = [q_lat | RoPE'd q_rope]; rows [L, 576] = [c_kv | RoPE'd k_rope];
    query g attends rows t < limits[g]. Every query shares the one cached row per
    token, as a multi-query attention with a 576-wide key and a 512-wide value
    (MLA absorb audit §6.1, head_dim_k=576 / head_dim_v=512).

    The value is the first ``d_c`` elements of each row.

    Returns (o_lat [G, d_c], lse [G], probs list). lse is the natural-log
    log-sum-exp of the scaled scores.
    """
    q = np.asarray(q_abs, dtype=np.float64)
    R = np.asarray(rows, dtype=np.float64)
    G = q.shape[0]
    o = np.zeros((G, d_c))
    lse = np.zeros(G)
    probs = []
    for g in range(G):
        n = int(limits[g])
        s = scale * (R[:n] @ q[g])
        m = np.max(s)
        e = np.exp(s - m)
        z = np.sum(e)
        p = e / z
        probs.append(p)
        o[g] = p @ R[:n, :d_c]
        lse[g] = m + math.log(z)
    return o, lse, probs


def absorbed_decode(c_kv, k_rope_raw, q_nope, q_rope_raw, W_UK, W_UV, scale, q_pos,
                    base: float = 10000.0):
    """Absorbed MLA decode of one sequence in float64.

    Same inputs as ``naive_decode``. The query is folded into latent space, the
    scores and the value aggregation run against the shared 576-wide rows, and
    the latent result is expanded last (MLA absorb audit §2.2-§2.3; 80-line
    PyTorch MLA §5).

    Returns (o [Hq, H, 128], o_lat [Hq, H, 512], lse [Hq, H]).
    """
    c = np.asarray(c_kv, dtype=np.float64)
    L = c.shape[0]
    kr = rope_f64(k_rope_raw, np.arange(L), base)
    rows = np.concatenate([c, kr], axis=1)
    qn = np.asarray(q_nope, dtype=np.float64)
    Hq, H = qn.shape[0], qn.shape[1]
    q_lat = absorb_query(qn, W_UK)                         # [Hq, H, 512]
    qr = rope_f64(np.asarray(q_rope_raw, dtype=np.float64), np.asarray(q_pos), base)
    d_c = c.shape[1]
    q_abs = np.concatenate([q_lat, qr], axis=2).reshape(Hq * H, rows.shape[1])
    limits = np.repeat(np.asarray(q_pos) + 1, H)
    o_lat, lse, _ = latent_attention(q_abs, rows, scale, limits, d_c)
    o_lat = o_lat.reshape(Hq, H, d_c)
    W = np.asarray(W_UV, dtype=np.float64)
    o = np.einsum("hvc,jhc->jhv", W, o_lat)
    return o, o_lat, lse.reshape(Hq, H)


def expand_values(o_lat, W_UV) -> np.ndarray:
    """o[..., h, :] = W_UV[h] o_lat[..., h, :]  (128 <- 512).

    Value absorption applied after aggregation: sum_t p_t W c_t = W sum_t p_t c_t
    (MLA absorb audit §2.3).
    """
    return np.einsum("hvc,...hc->...hv", np.asarray(W_UV, np.float64),
                     np.asarray(o_lat, np.float64))


def latent_projection(h, W_KV_A, kv_norm=None, eps: float = 1e-6):
    """The token's cached latent before rounding: (c_kv [n, 512], k_rope_raw [n, 64]).

    h [n, d_model] is the hidden state of the new tokens and W_KV_A [576, d_model]
    the combined down-projection (V2-Lite's kv_a_proj_with_mqa: the first 512
    outputs are the KV latent c_kv = W_DKV h, the last 64 the shared RoPE key
    k_R = W_KR h; 80-line PyTorch MLA §2, Wdkv / Wkr; V2-Lite trace audit §3.3).
    With ``kv_norm`` (the kv_a_layernorm weight, [512]) the latent is
    RMS-normalised: c / sqrt(mean(c^2) + eps) * kv_norm (MLA absorb audit §3.3
    names the norm; its definition is the RMSNorm one).
    """
    y = np.asarray(h, np.float64) @ np.asarray(W_KV_A, np.float64).T
    c, k = y[..., :D_C], y[..., D_C:D_C + D_ROPE]
    if kv_norm is not None:
        rms = np.sqrt(np.mean(c * c, axis=-1, keepdims=True) + eps)
        c = c / rms * np.asarray(kv_norm, np.float64)
    return c, k


def output_projection(o, W_O) -> np.ndarray:
    """y = W_O concat_h(o[..., h, :]): the attention block's output projection.

    o [..., H, d_v] is the per-head attention output, W_O [d_model, H * d_v] the
    nn.Linear(n_h * d_h -> d_model) weight. The heads are concatenated head-major
    (head h's d_v values at columns h*d_v .. h*d_v + d_v - 1), the order the
    module's o.transpose(1, 2).contiguous().view(B, L, n_h * d_h) produces
    (80-line PyTorch MLA §2, the forward's last line; V2-Lite trace audit §3.3,
    o_proj / wo).
    """
    o = np.asarray(o, np.float64)
    flat = o.reshape(o.shape[:-2] + (o.shape[-2] * o.shape[-1],))
    return flat @ np.asarray(W_O, np.float64).T


def absorb_output_weight(W_O, W_UV) -> np.ndarray:
    """W_OV [d_model, H * 512]: the value up-projection folded into the output
    projection, W_OV[:, h*512 + c] = sum_v W_O[:, h*d_v + v] W_UV[h][v, c].

    The value absorption of MLA absorb audit §2.3 (sum_t p_t W_UV c_t =
    W_UV sum_t p_t c_t) carried one matrix further, into the module's output
    projection (80-line PyTorch MLA §2, the forward's last line): y = W_O
    concat_h(W_UV[h] o_lat[h]) = W_OV concat_h(o_lat[h]), the heads' latents
    concatenated head-major. Not a step the pages take; a regrouping of the
    same products.
    """
    W_O = np.asarray(W_O, np.float64)
    W_UV = np.asarray(W_UV, np.float64)
    H, dv, dc = W_UV.shape
    return np.einsum("dhv,hvc->dhc", W_O.reshape(W_O.shape[0], H, dv), W_UV).reshape(W_O.shape[0], H * dc)


def combine_partials(o_parts, lse_parts):
    """Merge attention results of disjoint token ranges of one query row.

    o_parts [k, D] are the normalised per-range outputs, lse_parts [k] their
    log-sum-exp. The merged row is sum_k w_k o_k with w_k = exp(lse_k - lse),
    lse = log sum_k exp(lse_k): the softmax over the union of the ranges.
    """
    lp = np.asarray(lse_parts, dtype=np.float64)
    m = np.max(lp)
    w = np.exp(lp - m)
    z = np.sum(w)
    return (w[:, None] * np.asarray(o_parts, np.float64)).sum(0) / z, m + math.log(z)


# ---------------------------------------------------------------------------
# FP8 latent cache (MLA absorb audit §6.1: FlashMLA's decoding kernels read an
# FP8 KV cache in MQA mode, head_dim_k = 576, head_dim_v = 512). The pages name
# the variant only; the row format below is this library's reading of it:
#   bytes   0..511  e4m3 codes of c_kv / sigma (one code per latent element)
#   bytes 512..639  the RoPE'd key, bf16, the same bits the bf16 cache stores
#   bytes 640..643  sigma, float32: the token's power-of-two latent scale
#   bytes 644..655  zero
# ---------------------------------------------------------------------------

FP8_ROW_BYTES = 656
FP8_ROPE_OFF = 512
FP8_SCALE_OFF = 640
E4M3_MAX = 448.0


def e4m3_value(code) -> np.ndarray:
    """float64 value of e4m3 codes (OCP 8-bit floating point, E4M3: sign bit,
    4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
    subnormals m/8 * 2^-6; S.1111.111 is NaN; there are no infinities, so the
    largest finite magnitude is 1.75 * 2^8 = 448)."""
    c = np.asarray(code).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """uint8 e4m3 code of the value nearest to each x, ties to the even code
    (round to nearest even), magnitudes above 448 saturating to 448. The sign bit
    is the sign of x, zeros included (-0.0 -> 0x80)."""
    x = np.asarray(x, dtype=np.float64)
    table = e4m3_value(np.arange(0x7F))          # the 127 finite magnitudes, increasing
    a = np.minimum(np.abs(x), E4M3_MAX)
    i = np.clip(np.searchsorted(table, a, side="left"), 1, 0x7E)
    below, above = table[i - 1], table[i]
    d_lo, d_hi = a - below, above - a
    tie_pick = np.where((i - 1) % 2 == 0, i - 1, i)
    code = np.where(d_lo < d_hi, i - 1, np.where(d_hi < d_lo, i, tie_pick))
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


FP8_SCALE_EXP_MIN = -64


def fp8_scale_exponent(amax: float) -> int:
    """Exponent e of the token's scale sigma = 2^e: the smallest power of two
    with amax / sigma <= 448, but at least 2^-64 (amax = 0 gives 2^-64; the
    floor keeps 1/sigma, which the attention's softmax sum multiplies by, well
    inside float32). With amax = m * 2^k, 1 <= m < 2, and 448 = 1.75 * 2^8 this
    is e = k - 8 when m <= 1.75, else k - 7."""
    if amax == 0.0:
        return FP8_SCALE_EXP_MIN
    f, k1 = math.frexp(float(amax))     # amax = f * 2^k1, 0.5 <= f < 1
    m, k = 2.0 * f, k1 - 1
    e = k - 8 + (1 if m > 1.75 else 0)
    return max(e, FP8_SCALE_EXP_MIN)


def fp8_cache_rows(c_kv_bits, k_rope_bits, pos, base: float = 10000.0) -> np.ndarray:
    """uint8 [n, 656]: the FP8 cache rows of n tokens (format above).

    The latent of each token is scaled by its sigma (exact: a power of two) and
    rounded to e4m3; the RoPE key is the bf16 cache writer's, at pos."""
    c = bf16_to_f64(c_kv_bits)
    n = c.shape[0]
    out = np.zeros((n, FP8_ROW_BYTES), dtype=np.uint8)
    kr = rope_f32_contract(k_rope_bits, pos, base).astype("<u2")
    for i in range(n):
        e = fp8_scale_exponent(float(np.max(np.abs(c[i]))))
        out[i, :D_C] = e4m3_encode(c[i] * 2.0 ** -e)
        out[i, FP8_ROPE_OFF:FP8_SCALE_OFF] = np.frombuffer(kr[i].tobytes(), dtype=np.uint8)
        out[i, FP8_SCALE_OFF:FP8_SCALE_OFF + 4] = np.frombuffer(np.float32(2.0 ** e).astype("<f4").tobytes(),
                                                               dtype=np.uint8)
    return out


def fp8_rows_dequantize(rows) -> np.ndarray:
    """float64 [n, 576] = [e4m3 value * sigma (512) | RoPE'd key (64)] of FP8
    cache rows: the 576-wide rows the FP8 cache stands for."""
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.uint8))
    sigma = r[:, FP8_SCALE_OFF:FP8_SCALE_OFF + 4].copy().view("<f4").astype(np.float64)   # [n, 1]
    lat = e4m3_value(r[:, :D_C]) * sigma
    key = bf16_to_f64(r[:, FP8_ROPE_OFF:FP8_SCALE_OFF].copy().view("<u2"))
    return np.concatenate([lat, key], axis=1)
