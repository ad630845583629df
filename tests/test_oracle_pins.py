"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each test ties one oracle function to something other than itself: a value a
page prints for a worked example (tests/golden), a closed form, an invariant, a
special case that reduces to a textbook routine, or brute force written out
with scalar loops. CPU only.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SCALE = 1.0 / math.sqrt(192.0)


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand_bf16(rng, shape, std=1.0):
    """Random values that are exactly representable in bf16 (as float64)."""
    x = (rng.standard_normal(shape) * std).astype(np.float32)
    return O.bf16_to_f64(O.f32_to_bf16(x))


# ---------------------------------------------------------------------------
# byte accounting: the pages' printed sizes
# ---------------------------------------------------------------------------

def test_cache_bytes_v2lite_26_tokens():
    g = _load("cache_bytes.json")["v2lite_26_tokens_active"]
    L, H = g["L"], g["H"]
    assert O.latent_cache_bytes(L, g["d_c"], 0) == g["latent_c_kv_bytes"]
    assert O.latent_cache_bytes(L, 0, g["d_r"]) == g["latent_rope_bytes"]
    assert O.latent_cache_bytes(L) == g["latent_total_bytes"]
    k, v, tot = O.expanded_cache_bytes(L, H)
    assert (k, v, tot) == (g["naive_key_bytes"], g["naive_value_bytes"], g["naive_total_bytes"])
    assert tot / O.latent_cache_bytes(L) == pytest.approx(g["ratio"], rel=1e-15)
    assert 100.0 * (1 - O.latent_cache_bytes(L) / tot) == pytest.approx(g["reduction_percent"], abs=1e-12)


def test_cache_bytes_32_slot_allocated():
    g = _load("cache_bytes.json")["v2lite_32_slot_allocated"]
    assert O.latent_cache_bytes(g["L"], 512, 0) == g["latent_c_kv_bytes"]
    assert O.latent_cache_bytes(g["L"], 0, 64) == g["latent_rope_bytes"]
    assert O.latent_cache_bytes(g["L"]) == g["latent_total_bytes"]
    assert O.expanded_cache_bytes(g["L"], g["H"]) == (
        g["naive_key_bytes"], g["naive_value_bytes"], g["naive_total_bytes"])


def test_per_token_bytes_deepseek_v2_dims():
    g = _load("cache_bytes.json")["per_token_deepseek_v2"]
    mla = O.kv_bytes_per_token("mla")
    mha = O.kv_bytes_per_token("mha", n_h=128, d_h=128)
    gqa = O.kv_bytes_per_token("gqa", n_kv=8, d_h=128)
    assert (mla, mha, gqa) == (g["mla_bytes"], g["mha_bytes"], g["gqa8_bytes"])
    assert round(mha / mla, 1) == g["ratio_rounded"]
    gib = 1 << 30
    n = g["layers"] * g["tokens"]
    assert round(mla * n / gib, 2) == g["mla_total_gib_rounded"]
    assert mha * n / gib == g["mha_total_gib"]
    assert gqa * n / gib == g["gqa8_total_gib"]


def test_per_token_v2lite_eager_vs_latent():
    g = _load("cache_bytes.json")["per_token_v2lite_eager"]
    _, _, tot = O.expanded_cache_bytes(1, 16)
    assert tot == g["expanded_bytes"]
    assert O.latent_cache_bytes(1) == g["latent_bytes"]
    assert round(tot / O.latent_cache_bytes(1), 4) == g["ratio_rounded"]


# ---------------------------------------------------------------------------
# bfloat16 helpers
# ---------------------------------------------------------------------------

def test_bf16_roundtrip_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = O.bf16_to_f64(bits)
    ok = ~np.isnan(v)
    assert np.array_equal(O.f32_to_bf16(v[ok].astype(np.float32)), bits[ok])


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, 1.0 + 2.0**-8 + 2.0**-20,
                  -2.0, np.inf, 3.4e38, 0.0, -0.0], dtype=np.float32)
    want = [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC000, 0x7F80, 0x7F80, 0x0000, 0x8000]
    assert O.f32_to_bf16(x).tolist() == want
    assert O.f32_to_bf16(np.array([np.nan], np.float32)).tolist() == [0x7FC0]


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def test_rope_inverse_frequencies_closed_form():
    # base 10000, d=64: 10000^(-2i/64) = 10^(-i/8)
    inv = O.rope_inv_freq(64, 10000.0)
    want = np.array([10.0 ** (-i / 8.0) for i in range(32)])
    assert np.allclose(inv, want, rtol=1e-15, atol=0)
    assert inv[0] == 1.0


def test_rope_rotation_direction_matches_rotate_half():
    # 80-line PyTorch MLA, Appendix A: out = x*cos + rotate_half(x)*sin with
    # rotate_half(x) = (-x[2i+1], x[2i]) interleaved. At position 1 pair 0 turns
    # by exactly 1 radian: e0 -> (cos 1, sin 1), e1 -> (-sin 1, cos 1).
    c1, s1 = 0.5403023058681398, 0.8414709848078965
    e0 = np.zeros((1, 64)); e0[0, 0] = 1.0
    e1 = np.zeros((1, 64)); e1[0, 1] = 1.0
    y0, y1 = O.rope_f64(e0, [1]), O.rope_f64(e1, [1])
    assert y0[0, :2] == pytest.approx([c1, s1], abs=1e-16)
    assert y1[0, :2] == pytest.approx([-s1, c1], abs=1e-16)
    assert not y0[0, 2:].any() and not y1[0, 2:].any()
    # pair 1 turns by 10^(-1/8) radians at position 1
    e2 = np.zeros((1, 64)); e2[0, 2] = 1.0
    t = 10.0 ** (-1 / 8)
    assert O.rope_f64(e2, [1])[0, 2:4] == pytest.approx([math.cos(t), math.sin(t)], abs=1e-16)


def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 64))
    assert np.array_equal(O.rope_f64(x, [0, 0, 0]), x)
    bits = O.f32_to_bf16(x.astype(np.float32))
    assert np.array_equal(O.rope_f32_contract(bits, [0, 0, 0]), bits)


def test_rope_preserves_pair_norms_and_is_relative():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 64))
    k = rng.standard_normal((1, 64))
    for m, n in [(5, 3), (100, 37), (4095, 4000), (131071, 131000)]:
        qm, kn = O.rope_f64(q, [m]), O.rope_f64(k, [n])
        # per-pair norms preserved
        assert np.allclose(qm[0, 0::2]**2 + qm[0, 1::2]**2, q[0, 0::2]**2 + q[0, 1::2]**2,
                           rtol=1e-13)
        # (R_m q).(R_n k) depends only on m - n; the float64 angle m*theta carries
        # an absolute error of about m * 2^-53, hence the position-scaled bound
        lhs = float((qm @ kn.T)[0, 0])
        rhs = float((O.rope_f64(q, [m - n]) @ k.T)[0, 0])
        tol = 2.0**-50 * (m + 1) * np.linalg.norm(q) * np.linalg.norm(k)
        assert abs(lhs - rhs) <= tol


def test_rope_table_values():
    c, s = O.rope_cos_sin_f32([0, 1, 2])
    assert c.dtype == np.float32 and s.dtype == np.float32
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)
    assert c[1, 0] == np.float32(0.5403023058681398)   # cos 1
    assert s[2, 0] == np.float32(0.9092974268256817)   # sin 2
    cc, ss = O.rope_cos_sin_f32(np.arange(0, 131072, 997))
    r = cc.astype(np.float64)**2 + ss.astype(np.float64)**2
    assert np.all(np.abs(r - 1.0) < 4 * 2.0**-24)


def test_rope_contract_within_one_bf16_ulp_of_exact():
    rng = np.random.default_rng(3)
    n = 512
    pos = rng.integers(0, 131072, size=n)
    bits = O.f32_to_bf16(rng.standard_normal((n, 64)).astype(np.float32))
    got = O.bf16_to_f64(O.rope_f32_contract(bits, pos))
    x = O.bf16_to_f64(bits)
    exact = O.rope_f64(x, pos)
    # ulp of bf16 at |exact|, plus the float32 intermediate error
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(exact), 2.0**-126))) - 7)
    pair = np.repeat(np.abs(x[:, 0::2]) + np.abs(x[:, 1::2]), 2, axis=1)
    assert np.all(np.abs(got - exact) <= ulp + 8 * 2.0**-24 * pair)


def test_cache_row_layout_and_addressing():
    rng = np.random.default_rng(4)
    c = O.f32_to_bf16(rng.standard_normal((2, 512)).astype(np.float32))
    k = O.f32_to_bf16(rng.standard_normal((2, 64)).astype(np.float32))
    rows = O.cache_rows(c, k, [7, 8])
    assert rows.shape == (2, 576)
    assert np.array_equal(rows[:, :512], c)
    assert np.array_equal(rows[:, 512:], O.rope_f32_contract(k, [7, 8]))
    assert O.contiguous_row(3, 5, 32) == 101
    table = [[9, 2], [4, 0]]
    assert O.paged_row(0, 0, table) == 576 and O.paged_row(0, 70, table) == 134
    assert O.paged_row(1, 63, table) == 319 and O.paged_row(1, 64, table) == 0


# ---------------------------------------------------------------------------
# attention: brute force, special cases, invariants
# ---------------------------------------------------------------------------

def _brute_naive(c, kr_raw, qn, qr_raw, wuk, wuv, scale, qpos):
    """Scalar-loop naive MLA with one RoPE pair (d_r = 2, theta = 1)."""
    L, Dc = len(c), len(c[0])
    H, Dn, Dv = len(wuk), len(wuk[0]), len(wuv[0])
    out = []
    for h in range(H):
        keys, vals = [], []
        for t in range(L):
            kn = [sum(wuk[h][d][e] * c[t][e] for e in range(Dc)) for d in range(Dn)]
            a, b = kr_raw[t]
            kr = [a * math.cos(t) - b * math.sin(t), b * math.cos(t) + a * math.sin(t)]
            keys.append(kn + kr)
            vals.append([sum(wuv[h][d][e] * c[t][e] for e in range(Dc)) for d in range(Dv)])
        a, b = qr_raw[h]
        q = list(qn[h]) + [a * math.cos(qpos) - b * math.sin(qpos),
                           b * math.cos(qpos) + a * math.sin(qpos)]
        s = [scale * sum(q[i] * keys[t][i] for i in range(len(q))) for t in range(qpos + 1)]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        z = sum(e)
        out.append([sum(e[t] / z * vals[t][d] for t in range(qpos + 1)) for d in range(Dv)])
    return np.array(out)


@pytest.mark.parametrize("L", [1, 2, 3])
def test_brute_force_tiny(L):
    rng = np.random.default_rng(10 + L)
    H, Dn, Dc, Dv = 2, 3, 4, 3
    c = rng.standard_normal((L, Dc))
    kr = rng.standard_normal((L, 2))
    qn = rng.standard_normal((1, H, Dn))
    qr = rng.standard_normal((1, H, 2))
    wuk = rng.standard_normal((H, Dn, Dc))
    wuv = rng.standard_normal((H, Dv, Dc))
    scale = 1.0 / math.sqrt(Dn + 2)
    want = _brute_naive(c.tolist(), kr.tolist(), qn[0].tolist(), qr[0].tolist(),
                        wuk.tolist(), wuv.tolist(), scale, L - 1)
    got_n, _ = O.naive_decode(c, kr, qn, qr, wuk, wuv, scale, [L - 1])
    got_a, _, _ = O.absorbed_decode(c, kr, qn, qr, wuk, wuv, scale, [L - 1])
    assert np.allclose(got_n[0], want, rtol=0, atol=1e-14)
    assert np.allclose(got_a[0], want, rtol=0, atol=1e-14)


def _config0(rng, Hq=1, L=26, H=16):
    c = _rand_bf16(rng, (L, 512))
    kr = _rand_bf16(rng, (L, 64))
    qn = _rand_bf16(rng, (Hq, H, 128))
    qr = _rand_bf16(rng, (Hq, H, 64))
    wuk = _rand_bf16(rng, (H, 128, 512), 0.02)
    wuv = _rand_bf16(rng, (H, 128, 512), 0.02)
    return c, kr, qn, qr, wuk, wuv


@pytest.mark.parametrize("Hq", [1, 2])
def test_naive_equals_absorbed(Hq):
    rng = np.random.default_rng(20 + Hq)
    c, kr, qn, qr, wuk, wuv = _config0(rng, Hq)
    qpos = [26 - Hq + j for j in range(Hq)]
    on, probs = O.naive_decode(c, kr, qn, qr, wuk, wuv, SCALE, qpos)
    oa, olat, lse = O.absorbed_decode(c, kr, qn, qr, wuk, wuv, SCALE, qpos)
    assert np.max(np.abs(on - oa)) <= 1e-10
    # softmax rows sum to one
    for j in range(Hq):
        for p in probs[j]:
            assert abs(p.sum() - 1.0) <= 1e-14
            assert len(p) == qpos[j] + 1


def test_single_token_output_is_value_projection():
    rng = np.random.default_rng(30)
    c, kr, qn, qr, wuk, wuv = _config0(rng, 1, L=1)
    on, probs = O.naive_decode(c, kr, qn, qr, wuk, wuv, SCALE, [0])
    assert all(p.tolist() == [1.0] for p in probs[0])
    for h in range(16):
        assert np.array_equal(on[0, h], c[0] @ wuv[h].T)


def test_prefill_plus_decode_equals_one_shot():
    rng = np.random.default_rng(40)
    L, H = 26, 16
    c = _rand_bf16(rng, (L, 512))
    kr = _rand_bf16(rng, (L, 64))
    qn = _rand_bf16(rng, (L, H, 128))
    qr = _rand_bf16(rng, (L, H, 64))
    wuk = _rand_bf16(rng, (H, 128, 512), 0.02)
    wuv = _rand_bf16(rng, (H, 128, 512), 0.02)
    one_shot = O.naive_prefill_causal(c, kr, qn, qr, wuk, wuv, SCALE)
    for i in [0, 1, 12, 24, 25]:
        # cache holds tokens 0..i, the query of token i decodes over it
        inc, _ = O.naive_decode(c[:i + 1], kr[:i + 1], qn[i:i + 1], qr[i:i + 1],
                                wuk, wuv, SCALE, [i])
        assert np.max(np.abs(inc[0] - one_shot[i])) <= 1e-12


def test_mqa_reduction_identity_weights():
    # With W_UK = W_UV = I (d_nope = d_v = d_c) MLA decode is single-head attention
    # with key [c ; RoPE(k_rope)] and value c (MLA absorb audit §6.1, MQA mode).
    rng = np.random.default_rng(50)
    L, H, D = 9, 3, 8
    c = rng.standard_normal((L, D))
    kr = rng.standard_normal((L, 4))
    qn = rng.standard_normal((1, H, D))
    qr = rng.standard_normal((1, H, 4))
    eye = np.stack([np.eye(D)] * H)
    scale = 0.3
    got, _ = O.naive_decode(c, kr, qn, qr, eye, eye, scale, [L - 1])
    got_a, _, _ = O.absorbed_decode(c, kr, qn, qr, eye, eye, scale, [L - 1])
    theta = [1.0, 0.01]
    for h in range(H):
        keys = []
        for t in range(L):
            k = list(c[t])
            for i in range(2):
                a, b = kr[t][2 * i], kr[t][2 * i + 1]
                k += [a * math.cos(t * theta[i]) - b * math.sin(t * theta[i]),
                      b * math.cos(t * theta[i]) + a * math.sin(t * theta[i])]
            keys.append(k)
        q = list(qn[0, h])
        for i in range(2):
            a, b = qr[0, h, 2 * i], qr[0, h, 2 * i + 1]
            p = L - 1
            q += [a * math.cos(p * theta[i]) - b * math.sin(p * theta[i]),
                  b * math.cos(p * theta[i]) + a * math.sin(p * theta[i])]
        s = [scale * sum(x * y for x, y in zip(q, keys[t])) for t in range(L)]
        m = max(s)
        w = [math.exp(x - m) for x in s]
        z = sum(w)
        o = [sum(w[t] / z * c[t][d] for t in range(L)) for d in range(D)]
        assert np.allclose(got[0, h], o, atol=1e-12, rtol=0)
        assert np.allclose(got_a[0, h], o, atol=1e-12, rtol=0)


def test_rope_on_content_key_breaks_absorption():
    # Rotating the per-head content key W_UK c_t by its position cannot be folded
    # into the query: the absorbed scores then disagree (80-line PyTorch MLA §4).
    rng = np.random.default_rng(60)
    L = 26
    c = _rand_bf16(rng, (L, 512))
    qn = _rand_bf16(rng, (1, 1, 128))
    wuk = _rand_bf16(rng, (1, 128, 512), 0.02)
    k_c = c @ wuk[0].T                                  # [L, 128]
    k_c_rot = O.rope_f64(k_c, np.arange(L))            # RoPE on the content key
    q_rot = O.rope_f64(qn[0], [L - 1])[0]
    s_rope = k_c_rot @ q_rot
    q_lat = O.absorb_query(qn, wuk)[0, 0]
    s_abs = c @ q_lat
    s_plain = k_c @ qn[0, 0]
    assert np.max(np.abs(s_abs - s_plain)) <= 1e-12   # absorption itself holds
    assert np.max(np.abs(s_abs - s_rope)) > 1e-2      # but not with RoPE'd K_C


def test_latent_attention_causal_limits_and_lse():
    rng = np.random.default_rng(70)
    L = 17
    rows = rng.standard_normal((L, 576))
    q = rng.standard_normal((3, 576))
    lim = [17, 16, 1]
    o, lse, probs = O.latent_attention(q, rows, 0.05, lim)
    for g in range(3):
        s = 0.05 * rows[:lim[g]] @ q[g]
        assert lse[g] == pytest.approx(math.log(np.sum(np.exp(s))), abs=1e-12)
        assert len(probs[g]) == lim[g]
    assert np.array_equal(o[2], rows[0, :512])


@pytest.mark.parametrize("cuts", [[5], [1, 2, 40], [63, 64, 65]])
def test_split_and_combine_equals_unsplit(cuts):
    rng = np.random.default_rng(80)
    L = 100
    rows = rng.standard_normal((L, 576))
    q = rng.standard_normal((1, 576)) * 3
    full_o, full_lse, _ = O.latent_attention(q, rows, SCALE, [L])
    edges = [0] + cuts + [L]
    parts_o, parts_lse = [], []
    for a, b in zip(edges[:-1], edges[1:]):
        o, lse, _ = O.latent_attention(q, rows[a:b], SCALE, [b - a])
        parts_o.append(o[0])
        parts_lse.append(lse[0])
    o, lse = O.combine_partials(parts_o, parts_lse)
    assert np.max(np.abs(o - full_o[0])) <= 1e-12
    assert lse == pytest.approx(full_lse[0], abs=1e-12)


def test_absorb_and_expand_one_hot():
    rng = np.random.default_rng(90)
    W = rng.standard_normal((2, 128, 512))
    q = np.zeros((1, 2, 128)); q[0, 1, 7] = 1.0
    assert np.array_equal(O.absorb_query(q, W)[0, 1], W[1, 7, :])
    o = np.zeros((1, 2, 512)); o[0, 0, 300] = 1.0
    assert np.array_equal(O.expand_values(o, W)[0, 0], W[0, :, 300])


def test_output_projection_brute_force_and_head_order():
    # scalar loops over the definition y[m, d] = sum_h sum_v W_O[d, h*dv + v] o[m, h, v]
    rng = np.random.default_rng(21)
    M, H, dv, Dm = 3, 2, 3, 4
    o = rng.standard_normal((M, H, dv))
    w = rng.standard_normal((Dm, H * dv))
    want = np.zeros((M, Dm))
    for m in range(M):
        for d in range(Dm):
            acc = 0.0
            for h in range(H):
                for v in range(dv):
                    acc += w[d, h * dv + v] * o[m, h, v]
            want[m, d] = acc
    assert np.allclose(O.output_projection(o, w), want, rtol=0, atol=1e-12)
    # one-hot rows pick single (head, dim) entries: head-major concatenation
    w1 = np.zeros((H * dv, H * dv))
    for i in range(H * dv):
        w1[i, i] = 1.0
    y = O.output_projection(o, w1)
    assert np.array_equal(y[:, 1 * dv + 2], o[:, 1, 2])
    assert np.array_equal(y[:, 0 * dv + 1], o[:, 0, 1])


def test_output_projection_of_the_naive_block():
    # the whole attention block of the pages' module in matrix form (per-head
    # outputs of naive_decode, then W_O) equals the absorbed path followed by the
    # same projection, to 1e-10
    rng = np.random.default_rng(22)
    L, H = 9, 2
    c = rng.standard_normal((L, 512))
    k = rng.standard_normal((L, 64))
    qn = rng.standard_normal((1, H, 128))
    qr = rng.standard_normal((1, H, 64))
    wuk = rng.standard_normal((H, 128, 512)) * 0.02
    wuv = rng.standard_normal((H, 128, 512)) * 0.02
    wo = rng.standard_normal((256, H * 128)) * 0.02
    o_naive, _ = O.naive_decode(c, k, qn, qr, wuk, wuv, SCALE, [L - 1])
    o_abs, _, _ = O.absorbed_decode(c, k, qn, qr, wuk, wuv, SCALE, [L - 1])
    y1 = O.output_projection(o_naive, wo)
    y2 = O.output_projection(o_abs, wo)
    assert y1.shape == (1, 256)
    assert np.max(np.abs(y1 - y2)) <= 1e-10


def test_absorbed_output_weight_brute_force_and_two_step_form():
    # scalar loops over the definition W_OV[d, h*dc + c] = sum_v W_O[d, h*dv + v] W_UV[h, v, c]
    rng = np.random.default_rng(23)
    Dm, H, dv, dc = 3, 2, 2, 3
    wo = rng.standard_normal((Dm, H * dv))
    wuv = rng.standard_normal((H, dv, dc))
    want = np.zeros((Dm, H * dc))
    for d in range(Dm):
        for h in range(H):
            for c in range(dc):
                acc = 0.0
                for v in range(dv):
                    acc += wo[d, h * dv + v] * wuv[h, v, c]
                want[d, h * dc + c] = acc
    assert np.allclose(O.absorb_output_weight(wo, wuv), want, rtol=0, atol=1e-12)
    # at the library's dimensions: one projection of the concatenated latents
    # equals expand_values then output_projection, to 1e-10
    H = 4
    wo = rng.standard_normal((256, H * 128)) * 0.02
    wuv = rng.standard_normal((H, 128, 512)) * 0.02
    o_lat = rng.standard_normal((3, H, 512))
    y_two = O.output_projection(O.expand_values(o_lat, wuv), wo)
    y_one = o_lat.reshape(3, H * 512) @ O.absorb_output_weight(wo, wuv).T
    assert np.max(np.abs(y_two - y_one)) <= 1e-10
    # a one-hot W_UV row maps a latent column onto one value column of its head
    wuv1 = np.zeros((H, 128, 512))
    wuv1[2, 5, 300] = 1.0
    w_ov = O.absorb_output_weight(wo, wuv1)
    assert np.array_equal(w_ov[:, 2 * 512 + 300], wo[:, 2 * 128 + 5])
    assert np.count_nonzero(w_ov) == np.count_nonzero(wo[:, 2 * 128 + 5])


def test_latent_projection_brute_force_and_norm():
    rng = np.random.default_rng(31)
    n, D = 2, 5
    h = rng.standard_normal((n, D))
    w = rng.standard_normal((576, D))
    g = rng.standard_normal(512)
    c, k = O.latent_projection(h, w)
    # plain projection: scalar loops
    for t in range(n):
        for j in (0, 511):
            assert abs(c[t, j] - sum(w[j, d] * h[t, d] for d in range(D))) <= 1e-12
        for j in (0, 63):
            assert abs(k[t, j] - sum(w[512 + j, d] * h[t, d] for d in range(D))) <= 1e-12
    # RMSNorm: scalar loops over the definition, and unit RMS with a unit weight
    cn, kn = O.latent_projection(h, w, kv_norm=g, eps=1e-6)
    assert np.array_equal(kn, k)                      # the RoPE key is not normalised
    for t in range(n):
        ms = sum(c[t, j] ** 2 for j in range(512)) / 512
        r = math.sqrt(ms + 1e-6)
        assert abs(cn[t, 7] - c[t, 7] / r * g[7]) <= 1e-12
    c1, _ = O.latent_projection(h, w, kv_norm=np.ones(512), eps=0.0)
    assert np.allclose(np.sqrt(np.mean(c1 * c1, axis=-1)), 1.0, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# FP8 latent cache: e4m3 coding, the per-token scale, the 656-byte row
# ---------------------------------------------------------------------------

def test_e4m3_value_format_points():
    # points the E4M3 definition fixes: bias 7, 3 mantissa bits, subnormals
    # m/8 * 2^-6, S.1111.111 = NaN, largest finite 1.75 * 2^8
    v = O.e4m3_value
    assert v(0x00) == 0.0 and v(0x01) == 2.0 ** -9 and v(0x07) == 7 * 2.0 ** -9
    assert v(0x08) == 2.0 ** -6 and v(0x38) == 1.0 and v(0x39) == 1.125
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0 and v(0xB8) == -1.0
    assert math.isnan(v(0x7F)) and math.isnan(v(0xFF))
    finite = v(np.arange(0x7F))
    assert np.all(np.diff(finite) > 0)                       # increasing with the code
    assert np.sum(np.isfinite(v(np.arange(256)))) == 254


def test_e4m3_encode_ties_and_round_trip():
    e = O.e4m3_encode
    # midpoints go to the even code
    assert e(1.0625) == 0x38 and e(1.1875) == 0x3A          # 1 | 1.125 | 1.25
    assert e(2.0 ** -10) == 0x00 and e(3 * 2.0 ** -10) == 0x02
    assert e(-1.0625) == 0xB8 and e(-0.0) == 0x80 and e(0.0) == 0x00
    # just off a midpoint goes to the nearer code
    assert e(1.0625 + 1e-12) == 0x39 and e(1.0625 - 1e-12) == 0x38
    # saturation and exact values
    assert e(1000.0) == 0x7E and e(-449.0) == 0xFE
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F])
    assert np.array_equal(e(O.e4m3_value(codes)), codes.astype(np.uint8))


def test_e4m3_encode_matches_library_on_float32():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = np.concatenate([np.linspace(-448, 448, 100001), rng.standard_normal(50000) * 4,
                        rng.standard_normal(50000) * 0.005,
                        (O.e4m3_value(np.arange(0x7E)) + O.e4m3_value(np.arange(1, 0x7F))) / 2]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x), ref)


def test_fp8_scale_exponent_brute_force():
    rng = np.random.default_rng(3)
    cases = [0.0, 448.0, 448.0 * (1 + 2 ** -20), 3.5, 3.5 * (1 + 2 ** -7), 1.0, 2.0 ** -130, 1e30]
    cases += list(np.abs(_rand_bf16(rng, 200, 10.0)))
    for a in cases:
        e = O.fp8_scale_exponent(a)
        assert e >= -64
        # the smallest e from -64 up with a / 2^e <= 448
        want = next(k for k in range(-64, 200) if a / 2.0 ** k <= 448.0)
        assert e == want, (a, e, want)


def test_fp8_rows_bytes_and_error_bound():
    rng = np.random.default_rng(11)
    n = 40
    c = _rand_bf16(rng, (n, 512), 1.0)
    c[3] = 0.0                                     # all-zero latent
    c[4] *= 2.0 ** -70                             # tiny latent: the scale floor, subnormal codes
    c[5, 7] = 448.0 * 2 ** 3                       # amax exactly 448 * 2^3
    kr_bits = O.f32_to_bf16(rng.standard_normal((n, 64)).astype(np.float32))
    pos = np.arange(n) * 37
    rows = O.fp8_cache_rows(O.f32_to_bf16(c.astype(np.float32)), kr_bits, pos)
    assert rows.shape == (n, 656) and rows.dtype == np.uint8
    assert np.all(rows[:, 644:] == 0)
    # RoPE key bytes: the bf16 cache writer's
    bf_rows = O.cache_rows(O.f32_to_bf16(c.astype(np.float32)), kr_bits, pos)
    assert np.array_equal(rows[:, 512:640].copy().view("<u2"), bf_rows[:, 512:])
    sigma = rows[:, 640:644].copy().view("<f4")[:, 0].astype(np.float64)
    assert sigma[5] == 2.0 ** 3                   # amax 448 * 2^3 codes as 448 with sigma 2^3
    assert sigma[3] == 2.0 ** -64 and sigma[4] == 2.0 ** -64
    assert np.any((rows[4, :512] & 0x78) == 0) and np.any(rows[4, :512] & 0x07)
    assert np.all(np.frexp(sigma)[0] == 0.5)      # powers of two
    deq = O.fp8_rows_dequantize(rows)
    assert deq[5, 7] == 3584.0 and rows[5, 7] == 0x7E
    # no code saturates: |c / sigma| <= 448 everywhere
    assert np.all(np.abs(c) / sigma[:, None] <= 448.0)
    # nearest-code error bound: half a step of e4m3 at the value's binade
    # (2^-4 relative for normal codes, 2^-10 * sigma absolute below 2^-6 * sigma)
    err = np.abs(deq[:, :512] - c)
    bound = np.maximum(np.abs(c) * 2.0 ** -4, sigma[:, None] * 2.0 ** -10)
    assert np.all(err <= bound)
    assert np.array_equal(deq[:, 512:], O.bf16_to_f64(bf_rows[:, 512:]))


def test_fp8_rows_exact_latent_gives_the_bf16_result():
    # a latent whose values are e4m3 codes times the token's scale (with the
    # largest at 448 * sigma) is stored exactly, so attention over the FP8 rows
    # equals attention over the bf16 rows
    rng = np.random.default_rng(5)
    n = 50
    e = rng.integers(-12, 4, size=n)
    codes = rng.integers(0, 0x7F, size=(n, 512))
    codes[:, 0] = 0x7E
    sign = np.where(rng.random((n, 512)) < 0.5, -1.0, 1.0)
    c = sign * O.e4m3_value(codes) * np.exp2(e.astype(np.float64))[:, None]
    c_bits = O.f32_to_bf16(c.astype(np.float32))
    assert np.array_equal(O.bf16_to_f64(c_bits), c)          # exact in bf16 too
    kr_bits = O.f32_to_bf16(rng.standard_normal((n, 64)).astype(np.float32))
    pos = np.arange(n)
    deq = O.fp8_rows_dequantize(O.fp8_cache_rows(c_bits, kr_bits, pos))
    ref = O.bf16_to_f64(O.cache_rows(c_bits, kr_bits, pos))
    assert np.array_equal(deq, ref)
    q = rng.standard_normal((4, 576))
    a = O.latent_attention(q, deq, SCALE, [n, 10, 1, 33])
    b = O.latent_attention(q, ref, SCALE, [n, 10, 1, 33])
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
