"""Per-call parity of the CUDA path (through the C ABI) against the oracle."""
import math

import numpy as np
import pytest
import torch

import mla_synth as S
import oracle as O
from mla_testlib import SCALE, assert_close, bits, f64

pytestmark = pytest.mark.gpu


def _normal(name, shape, std=1.0, seed=7):
    return S.normal_bf16(seed, name, shape, std=std, device="cuda")


# ----------------------------------------------------------------- append
@pytest.mark.parametrize("paged", [False, True])
def test_append_latent_bit_exact(mla, ctx, paged):
    B, n = 3, 200
    c = _normal(f"app/c/{paged}", (n, 512))
    k = _normal(f"app/k/{paged}", (n, 64))
    seq = torch.tensor(S.uniform_ints(1, f"app/seq/{paged}", n, 0, B - 1), dtype=torch.int32)
    if paged:
        max_blocks = 2048                      # positions up to 131071
        nb = B * 4
        table = torch.full((B, max_blocks), -1, dtype=torch.int32)
        perm = S.permutation(1, "app/perm", nb)
        for b in range(B):
            for j in range(4):
                table[b, [0, 1, 700, 2047][j]] = perm[4 * b + j]
        # positions inside the four mapped blocks, including 131071
        blocks = torch.tensor([0, 1, 700, 2047])
        sel = torch.tensor(S.uniform_ints(2, "app/blk", n, 0, 3))
        off = torch.tensor(S.uniform_ints(3, "app/off", n, 0, 63))
        pos = (blocks[sel] * 64 + off).to(torch.int32)
        pos[0] = 131071
        cache = mla.Cache.paged_pool(nb, table)
    else:
        cap = 1000
        pos = torch.tensor(S.uniform_ints(2, "app/pos", n, 0, cap - 1), dtype=torch.int32)
        pos[0] = cap - 1
        cache = mla.Cache.contiguous(B, cap)
    # distinct slots so that later writes do not overwrite earlier ones
    key = seq.long() * 10**7 + pos.long()
    _, first = np.unique(key.numpy(), return_index=True)
    first = torch.tensor(np.sort(first))
    c, k, seq, pos = c[first.cuda()].contiguous(), k[first.cuda()].contiguous(), seq[first], pos[first]
    ctx.append_latent(cache, c, k, seq.cuda(), pos.cuda())
    assert ctx.device_status() == 0
    got = bits(cache.storage).reshape(-1, 576)
    want = np.zeros_like(got)
    rows = O.cache_rows(bits(c), bits(k), pos.numpy())
    for i in range(len(seq)):
        s, t = int(seq[i]), int(pos[i])
        r = O.paged_row(s, t, table.tolist()) if paged else O.contiguous_row(s, t, 1000)
        want[r] = rows[i]
    assert np.array_equal(got, want)


def test_append_out_of_range_sets_bounds_and_skips(mla, ctx):
    cache = mla.Cache.contiguous(2, 16)
    c = _normal("oob/c", (3, 512))
    k = _normal("oob/k", (3, 64))
    seq = torch.tensor([0, 2, 1], dtype=torch.int32, device="cuda")   # seq 2 does not exist
    pos = torch.tensor([3, 0, 16], dtype=torch.int32, device="cuda")  # pos 16 >= capacity
    ctx.append_latent(cache, c, k, seq, pos)
    st = ctx.device_status()
    assert st & mla.DEVICE_BOUNDS
    got = bits(cache.storage).reshape(-1, 576)
    assert np.array_equal(got[3], O.cache_rows(bits(c[:1]), bits(k[:1]), [3])[0])
    assert np.count_nonzero(np.delete(got, 3, axis=0)) == 0
    assert ctx.device_status() == 0


# ----------------------------------------------------------------- absorb_q
@pytest.mark.parametrize("B,Hq,H", [(5, 2, 16), (3, 1, 128), (130, 1, 32), (2, 2, 64)])
def test_absorb_q(mla, ctx, B, Hq, H):
    w = _normal(f"aq/w/{H}", (H, 128, 512), std=0.02)
    qn = _normal(f"aq/qn/{B}/{H}", (B, Hq, H, 128))
    qr = _normal(f"aq/qr/{B}/{H}", (B, Hq, H, 64))
    qpos = torch.tensor(S.uniform_ints(4, f"aq/pos/{B}", B * Hq, 0, 131071), dtype=torch.int32).view(B, Hq)
    q_abs = ctx.absorb_q(w, qn, qr, qpos.cuda())
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    want = O.absorb_query(f64(qn), f64(w))
    got = f64(q_abs[..., :512])
    err = np.abs(got - want)
    assert np.all(err <= 2.0**-8 * np.abs(want) + 1e-5), float(np.max(err))
    assert_close(got, want, what="q_lat")
    # the rope part follows the cache writer's bit-exact RoPE contract
    rope_want = O.rope_f32_contract(bits(qr).reshape(B * Hq, H, 64), qpos.reshape(-1).numpy())
    assert np.array_equal(bits(q_abs[..., 512:]).reshape(B * Hq, H, 64), rope_want)


# ----------------------------------------------------------------- expand_v
@pytest.mark.parametrize("B,Hq,H", [(5, 1, 16), (3, 2, 128), (129, 1, 16), (130, 1, 64),
                                    (64, 1, 16), (33, 1, 32), (16, 2, 16)])   # <= 64 rows: column-split kernel
def test_expand_v(mla, ctx, B, Hq, H):
    w = _normal(f"ev/w/{H}", (H, 128, 512), std=0.02)
    a = _normal(f"ev/a/{B}/{H}", (B, Hq, H, 512)).float()
    b = _normal(f"ev/b/{B}/{H}", (B, Hq, H, 512)).float()
    o_lat = (a + b * 2.0**-9).contiguous()           # fp32 values with more than 8 mantissa bits
    out = ctx.expand_v(w, o_lat)
    torch.cuda.synchronize()
    want = O.expand_values(f64(o_lat), f64(w))
    got = f64(out)
    err = np.abs(got - want)
    assert np.all(err <= 2.0**-8 * np.abs(want) + 1e-4), float(np.max(err))
    assert_close(got, want, what="expand_v")


# ----------------------------------------------------------------- project_latent
@pytest.mark.parametrize("n,D,paged,norm", [(64, 2048, False, True), (5, 256, True, False),
                                            (300, 512, False, True), (32, 7168, True, True),
                                            (7936, 64, False, True)])
def test_project_latent(mla, ctx, n, D, paged, norm):
    # (7936, 64): 31 blocks of 256 tokens do not fit five times over on 152 SMs,
    # so the call takes the split-K + finish path instead of the one launch
    w = _normal(f"pl/w/{D}", (576, D), std=0.02)
    h = _normal(f"pl/h/{n}/{D}", (n, D))
    g = (1.0 + 0.1 * _normal("pl/g", (512,)).float()).to(torch.bfloat16) if norm else None
    B = 3
    seq = torch.tensor([i % B for i in range(n)], dtype=torch.int32)
    pos = torch.tensor([i // B + 7 for i in range(n)], dtype=torch.int32)
    L = int(pos.max()) + 1
    if paged:
        nblk = (L + 63) // 64
        perm = S.permutation(5, "pl/perm", B * nblk)
        table = torch.tensor(perm, dtype=torch.int32).view(B, nblk)
        cache = mla.Cache.paged_pool(B * nblk, table)
        rows = [O.paged_row(int(s_), int(t_), table.tolist()) for s_, t_ in zip(seq, pos)]
    else:
        cache = mla.Cache.contiguous(B, L)
        rows = [O.contiguous_row(int(s_), int(t_), L) for s_, t_ in zip(seq, pos)]
    ctx.project_latent(cache, w, h, seq.cuda(), pos.cuda(), kv_norm=g, eps=1e-6)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    got = O.bf16_to_f64(bits(cache.storage).reshape(-1, 576)[rows])
    c_want, k_want = O.latent_projection(f64(h), f64(w), None if g is None else f64(g), 1e-6)
    k_rot = O.rope_f64(k_want, pos.numpy())
    assert np.all(np.abs(got[:, :512] - c_want) <= 2.0**-8 * np.abs(c_want) + 1e-4), \
        float(np.max(np.abs(got[:, :512] - c_want)))
    kmax = np.max(np.abs(k_rot), axis=1, keepdims=True)
    assert np.all(np.abs(got[:, 512:] - k_rot) <= 2.0**-7 * kmax + 1e-4), float(np.max(np.abs(got[:, 512:] - k_rot)))


def test_project_latent_one_launch_is_deterministic(mla, ctx):
    """The one-launch producer adds its split partials in a fixed order: two calls
    write the same bytes (the barrier words reset themselves between calls)."""
    n, D = 32, 7168
    w = _normal(f"pl/w/{D}", (576, D), std=0.02)
    h = _normal(f"pl/h/{n}/{D}", (n, D))
    seq = torch.arange(n, dtype=torch.int32, device="cuda")
    pos = torch.full((n,), 3, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(3):
        cache = mla.Cache.contiguous(n, 4)
        ctx.project_latent(cache, w, h, seq, pos)
        torch.cuda.synchronize()
        outs.append(bits(cache.storage))
    assert ctx.device_status() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_project_latent_out_of_range_row_flagged(mla, ctx):
    cache = mla.Cache.contiguous(2, 8)
    w = _normal("pl/w/64", (576, 64), std=0.02)
    h = _normal("pl/h/3/64", (3, 64))
    seq = torch.tensor([0, 1, 5], dtype=torch.int32, device="cuda")      # sequence 5 does not exist
    pos = torch.tensor([0, 3, 0], dtype=torch.int32, device="cuda")
    ctx.project_latent(cache, w, h, seq, pos)
    torch.cuda.synchronize()
    assert ctx.device_status() & mla.DEVICE_BOUNDS


# ----------------------------------------------------------------- out_proj
@pytest.mark.parametrize("M,H,Dm", [(5, 16, 256), (64, 16, 2048), (129, 16, 384), (300, 32, 256),
                                    (32, 128, 1024)])
def test_out_proj(mla, ctx, M, H, Dm):
    w = _normal(f"op/w/{H}/{Dm}", (Dm, H * 128), std=0.02)
    o = _normal(f"op/o/{M}/{H}", (M, H, 128))
    y = ctx.out_proj(w, o)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    want = O.output_projection(f64(o), f64(w))
    got = f64(y)
    # bf16 inputs are exact in fp64; only the fp32 accumulation differs
    assert np.max(np.abs(got - want)) <= 1e-4 * np.max(np.abs(want)) + 1e-5
    assert_close(got, want, what="out_proj")
    # y is overwritten, not accumulated into
    y2 = ctx.out_proj(w, o, y=y)
    torch.cuda.synchronize()
    assert np.max(np.abs(f64(y2) - want)) <= 1e-4 * np.max(np.abs(want)) + 1e-5


@pytest.mark.parametrize("M,H,Dm", [(64, 16, 2048), (300, 32, 256), (1024, 16, 512)])
def test_out_proj_overwrites_and_repeats(mla, ctx, M, H, Dm):
    """y starts as NaN (no zero-fill is needed: the first split of each tile
    stores, the others add after it), and calls queued back to back on one
    stream, with no synchronisation between them, each give the right result
    (the per-tile words reset themselves between calls)."""
    w = _normal(f"op/w/{H}/{Dm}", (Dm, H * 128), std=0.02)
    os_ = [_normal(f"op/o/{M}/{H}/{i}", (M, H, 128)) for i in range(4)]
    ys = [torch.full((M, Dm), float("nan"), dtype=torch.float32, device="cuda") for _ in range(4)]
    for i in range(4):
        ctx.out_proj(w, os_[i], y=ys[i])
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    for i in range(4):
        want = O.output_projection(f64(os_[i]), f64(w))
        got = f64(ys[i])
        assert np.all(np.isfinite(got))
        assert np.max(np.abs(got - want)) <= 1e-4 * np.max(np.abs(want)) + 1e-5


@pytest.mark.parametrize("H,Dm", [(16, 256), (128, 384)])
def test_absorb_w_o(mla, ctx, H, Dm):
    """W_UV folded into W_O: fp32 accumulation of 128 exact bf16 products, then
    one rounding to bf16 (within half a bf16 step of the exact fold)."""
    w_o = _normal(f"ov/wo/{H}/{Dm}", (Dm, H * 128), std=0.02)
    w_uv = _normal(f"ov/wuv/{H}", (H, 128, 512), std=0.02)
    w_ov = ctx.absorb_w_o(w_o, w_uv)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    want = O.absorb_output_weight(f64(w_o), f64(w_uv))
    got = f64(w_ov)
    assert got.shape == (Dm, H * 512)
    assert np.all(np.abs(got - want) <= 2.0**-8 * np.abs(want) + 1e-9), float(np.max(np.abs(got - want)))


@pytest.mark.parametrize("M,H,Dm", [(5, 16, 256), (64, 16, 2048), (129, 16, 384), (300, 32, 256),
                                    (32, 128, 1024)])
def test_out_proj_latent_vs_two_step(mla, ctx, M, H, Dm):
    """y = W_OV concat_h(o_lat) in one GEMM against expand_values then
    output_projection in float64; the two-call GPU path (expand_v, out_proj)
    on the same inputs meets the same bars."""
    w_o = _normal(f"ov/wo/{H}/{Dm}", (Dm, H * 128), std=0.02)
    w_uv = _normal(f"ov/wuv/{H}", (H, 128, 512), std=0.02)
    o_lat = (0.3 * _normal(f"ov/olat/{M}/{H}", (M, H, 512)).float()).contiguous()
    w_ov = ctx.absorb_w_o(w_o, w_uv)
    y = ctx.out_proj_latent(w_ov, o_lat)
    y2 = ctx.out_proj(w_o, ctx.expand_v(w_uv, o_lat.view(M, 1, H, 512)))
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    want = O.output_projection(O.expand_values(f64(o_lat), f64(w_uv)), f64(w_o))
    assert_close(f64(y), want, what="out_proj_latent (one GEMM)")
    assert_close(f64(y2), want, what="expand_v + out_proj")
    # y is overwritten, not accumulated into
    y3 = ctx.out_proj_latent(w_ov, o_lat, y=y)
    torch.cuda.synchronize()
    assert_close(f64(y3), want, what="out_proj_latent, second call")


@pytest.mark.parametrize("M,H,Dm", [(64, 16, 2048), (300, 32, 256)])
def test_out_proj_latent_overwrites_and_repeats(mla, ctx, M, H, Dm):
    """y starts as NaN (the first split of each column group to finish stores,
    the others add after it), and calls queued back to back on one stream each
    give the right result (the per-tile words reset themselves)."""
    w_o = _normal(f"ov/wo/{H}/{Dm}", (Dm, H * 128), std=0.02)
    w_uv = _normal(f"ov/wuv/{H}", (H, 128, 512), std=0.02)
    w_ov = ctx.absorb_w_o(w_o, w_uv)
    o_lats = [(0.3 * _normal(f"ov/olat/{M}/{H}/{i}", (M, H, 512)).float()).contiguous() for i in range(3)]
    ys = [torch.full((M, Dm), float("nan"), dtype=torch.float32, device="cuda") for _ in range(3)]
    for i in range(3):
        ctx.out_proj_latent(w_ov, o_lats[i], y=ys[i])
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    for i in range(3):
        want = O.output_projection(O.expand_values(f64(o_lats[i]), f64(w_uv)), f64(w_o))
        got = f64(ys[i])
        assert np.all(np.isfinite(got))
        assert_close(got, want, what=f"out_proj_latent call {i}")


def test_out_proj_rejects_bad_width(mla, ctx):
    w = torch.zeros(200, 16 * 128, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(4, 16, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError):
        ctx.out_proj(w, o)


# ----------------------------------------------------------------- decode attention
def _attn_case(mla, ctx, H, Hq, lens, paged, q_std=1.0, units=0, seed=11, workspace=None):
    """Oracle rows written straight into the cache, random q_abs, decode_attn vs oracle."""
    B = len(lens)
    G = Hq * H
    rows_b = []
    for b, L in enumerate(lens):
        c = S.normal_bf16(seed, f"at/c/{b}", (L, 512), device="cuda")
        k = S.normal_bf16(seed, f"at/k/{b}", (L, 64), device="cuda")
        rows_b.append(O.cache_rows(bits(c), bits(k), np.arange(L)))
    if paged:
        nblk = [(L + 63) // 64 for L in lens]
        perm = S.permutation(seed, "at/perm", sum(nblk) + 3)   # a few unused blocks
        table = torch.full((B, max(nblk)), -1, dtype=torch.int32)
        o = 0
        for b in range(B):
            table[b, :nblk[b]] = torch.tensor(perm[o:o + nblk[b]], dtype=torch.int32)
            o += nblk[b]
        cache = mla.Cache.paged_pool(sum(nblk) + 3, table)
        # fill every slot with NaN first: rows past a sequence's end must not leak
        cache.storage.view(torch.int16).fill_(0x7FC0)
        host = bits(cache.storage).reshape(-1, 576).copy()
        for b, L in enumerate(lens):
            for t in range(L):
                host[O.paged_row(b, t, table.tolist())] = rows_b[b][t]
    else:
        cap = max(lens) + 5
        cache = mla.Cache.contiguous(B, cap)
        cache.storage.view(torch.int16).fill_(0x7FC0)
        host = bits(cache.storage).reshape(-1, 576).copy()
        for b, L in enumerate(lens):
            host[b * cap:b * cap + L] = rows_b[b]
    cache.storage.view(torch.int16).copy_(torch.from_numpy(host.view(np.int16)).view_as(cache.storage.view(torch.int16)))
    q = S.normal_bf16(seed, "at/q", (B, Hq, H, 576), std=q_std, device="cuda")
    seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ctx.set_decode_units(units)
    try:
        o_lat, lse = ctx.decode_attn(cache, q, seq_lens, SCALE, workspace=workspace)
        torch.cuda.synchronize()
    finally:
        ctx.set_decode_units(0)
    assert ctx.device_status() == 0
    qh = f64(q).reshape(B, G, 576)
    want_o = np.zeros((B, G, 512))
    want_l = np.zeros((B, G))
    for b, L in enumerate(lens):
        lim = [L - Hq + 1 + g // H for g in range(G)]
        o, l, _ = O.latent_attention(qh[b], O.bf16_to_f64(rows_b[b]), SCALE, lim)
        want_o[b], want_l[b] = o, l
    got_o = f64(o_lat).reshape(B, G, 512)
    got_l = f64(lse).reshape(B, G)
    assert_close(got_o, want_o, what="o_lat")
    assert np.max(np.abs(got_l - want_l)) <= 5e-3, float(np.max(np.abs(got_l - want_l)))
    return got_o, got_l


@pytest.mark.parametrize("H,Hq,lens,paged", [
    (16, 1, [1], False),
    (16, 1, [26], False),
    (16, 1, [63, 64, 65, 127, 128, 129, 300], False),
    (16, 2, [2, 130, 257], False),
    (32, 1, [200, 1], True),
    (64, 1, [333, 64], True),
    (128, 1, [1, 64, 129, 700], True),
    (128, 2, [2, 129, 450], True),
    # prefill chunks: many query tokens per sequence, bottom-right causal
    (16, 64, [64, 200], False),
    (16, 128, [128, 131], False),
    (128, 8, [8, 300], True),
    (64, 16, [16, 77, 256], True),
    (128, 16, [16, 40], True),         # 2048 query rows per sequence: 32 CTAs per unit
    # an odd number of 64-row CTAs per unit (single CTAs, not pairs)
    (64, 3, [3, 300], True),
    (16, 20, [20, 141], False),
])
def test_decode_attn_vs_oracle(mla, ctx, H, Hq, lens, paged):
    _attn_case(mla, ctx, H, Hq, lens, paged)


def test_decode_attn_max_batch(mla, ctx):
    # 1024 sequences (the per-call maximum), lengths 0..199 drawn from the seed:
    # the tile prefix over all of them, split-KV across sequences, and the
    # sequences shorter than Hq flagged
    lens = S.uniform_ints(9, "maxb/lens", 1024, 0, 199)
    short = [b for b, L in enumerate(lens) if L < 1]
    lens_ok = [max(L, 1) for L in lens]
    got, _ = _attn_case(mla, ctx, 16, 1, lens_ok, False, seed=9)
    assert got.shape == (1024, 16, 512)
    cache = mla.Cache.contiguous(1024, 200)
    q = torch.zeros(1024, 1, 16, 576, dtype=torch.bfloat16, device="cuda")
    o_lat, lse = ctx.decode_attn(cache, q, torch.tensor(lens, dtype=torch.int32, device="cuda"), SCALE)
    st = ctx.device_status()
    assert bool(st & mla.DEVICE_LENGTH) == bool(short)
    if short:
        assert torch.all(torch.isneginf(lse[short]))


@pytest.mark.parametrize("H", [64, 128])
def test_decode_attn_batch_spanning_every_warp(mla, ctx, H):
    # 600 sequences: one per thread of the 640-thread CTAs (64 rows each), so
    # the last warps of the tile prefix hold sequences too
    lens = [max(L, 1) for L in S.uniform_ints(12, "b600/lens", 600, 0, 150)]
    _attn_case(mla, ctx, H, 1, lens, True, seed=12)


def test_decode_attn_rejects_batch_above_max(mla, ctx):
    cache = mla.Cache.contiguous(1025, 8)
    q = torch.zeros(1025, 1, 16, 576, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError):
        ctx.decode_attn(cache, q, torch.full((1025,), 4, dtype=torch.int32, device="cuda"), SCALE)


def test_decode_attn_rejects_too_many_rows(mla, ctx):
    cache = mla.Cache.contiguous(1, 256)
    q = torch.zeros(1, 129, 16, 576, dtype=torch.bfloat16, device="cuda")   # 129 * 16 rows
    with pytest.raises(RuntimeError):
        ctx.decode_attn(cache, q, torch.tensor([256], dtype=torch.int32, device="cuda"), SCALE)


@pytest.mark.parametrize("H", [16, 128])
def test_decode_attn_peaky_scores_rescale(mla, ctx, H):
    # large queries make the running max jump often (lazy rescale path)
    _attn_case(mla, ctx, H, 1, [1000, 517], True, q_std=6.0)


@pytest.mark.parametrize("H,Hq", [(16, 1), (128, 1), (128, 2)])
def test_decode_attn_split_kv(mla, ctx, H, Hq):
    lens = [900, 31, 1200, 5]
    one, _ = _attn_case(mla, ctx, H, Hq, lens, True, units=1)
    many, _ = _attn_case(mla, ctx, H, Hq, lens, True, units=0)
    seven, _ = _attn_case(mla, ctx, H, Hq, lens, True, units=7)
    assert_close(many, one, what="split vs unsplit")
    assert_close(seven, one, what="7 units vs unsplit")


@pytest.mark.parametrize("H", [16, 128])
def test_decode_attn_reuses_workspace(mla, ctx, H):
    # one workspace serves consecutive calls with different lengths, layouts and
    # unit counts (nothing in it carries over from one call to the next)
    ws = ctx.alloc_workspace(H, 4, 1)
    first, _ = _attn_case(mla, ctx, H, 1, [900, 31, 1200, 5], True, workspace=ws)
    _attn_case(mla, ctx, H, 1, [64, 700, 3, 2000], False, seed=12, workspace=ws)
    _attn_case(mla, ctx, H, 1, [900, 31, 1200, 5], True, units=7, workspace=ws)
    again, _ = _attn_case(mla, ctx, H, 1, [900, 31, 1200, 5], True, workspace=ws)
    assert np.array_equal(first, again)


def test_decode_attn_workspace_across_shapes(mla, ctx):
    # one workspace serves calls of different batch, heads, query tokens and
    # split (nothing in it carries over from one call to the next)
    ws = ctx.alloc_workspace(128, 8, 2)   # the largest shape below
    a, _ = _attn_case(mla, ctx, 16, 1, [900, 31, 1200, 5], True, workspace=ws)
    _attn_case(mla, ctx, 128, 2, [517, 2, 3000], True, seed=13, workspace=ws)
    _attn_case(mla, ctx, 16, 1, [4000] * 8, False, seed=14, workspace=ws)
    _attn_case(mla, ctx, 128, 1, [900, 31, 1200, 5], True, units=7, workspace=ws)
    b, _ = _attn_case(mla, ctx, 16, 1, [900, 31, 1200, 5], True, workspace=ws)
    assert np.array_equal(a, b)


def test_decode_attn_deterministic(mla, ctx):
    a = _attn_case(mla, ctx, 128, 1, [1000, 300, 77], True)
    b = _attn_case(mla, ctx, 128, 1, [1000, 300, 77], True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("H", [16, 128])
def test_decode_attn_bad_block_table_sets_bounds(mla, ctx, H):
    # a block id outside the pool (single-CTA kernel at H=16, CTA pairs at
    # H=128): that page's copies are skipped and the bounds bit is set, with no
    # fault; the other sequence's output is still exact
    lens = [200, 130]
    table = torch.tensor([[0, 1, 2, 3], [4, 5, 99, -1]], dtype=torch.int32)   # block 99 does not exist
    cache = mla.Cache.paged_pool(8, table)
    cache.storage.view(torch.int16).fill_(0x7FC0)
    host = bits(cache.storage).reshape(-1, 576).copy()
    rows = []
    for b, L in enumerate(lens):
        c = S.normal_bf16(44, f"at/bt/c/{b}", (L, 512), device="cuda")
        k = S.normal_bf16(44, f"at/bt/k/{b}", (L, 64), device="cuda")
        rows.append(O.cache_rows(bits(c), bits(k), np.arange(L)))
        for t in range(min(L, 128) if b == 1 else L):   # sequence 1: only its first two blocks exist
            host[O.paged_row(b, t, table.tolist())] = rows[b][t]
    cache.storage.view(torch.int16).copy_(torch.from_numpy(host.view(np.int16)).view_as(cache.storage.view(torch.int16)))
    q = S.normal_bf16(44, "at/bt/q", (2, 1, H, 576), device="cuda")
    o_lat, lse = ctx.decode_attn(cache, q, torch.tensor(lens, dtype=torch.int32, device="cuda"), SCALE)
    torch.cuda.synchronize()
    assert ctx.device_status() & mla.DEVICE_BOUNDS
    want, _, _ = O.latent_attention(f64(q)[0, 0], O.bf16_to_f64(rows[0]), SCALE, [lens[0]] * H)
    assert_close(f64(o_lat)[0, 0], want, what="o_lat of the intact sequence")
    # the context stays usable: a clean call afterwards
    _attn_case(mla, ctx, H, 1, [90, 260], True)


def test_decode_attn_short_length_flagged(mla, ctx):
    cache = mla.Cache.contiguous(2, 8)
    q = S.normal_bf16(1, "short/q", (2, 2, 16, 576), device="cuda")
    seq_lens = torch.tensor([1, 0], dtype=torch.int32, device="cuda")   # below Hq = 2
    o_lat, lse = ctx.decode_attn(cache, q, seq_lens, SCALE)
    st = ctx.device_status()
    assert st & mla.DEVICE_LENGTH
    assert torch.count_nonzero(o_lat).item() == 0
    assert torch.all(torch.isneginf(lse))


def test_bounded_wait_reports_timeout(mla, ctx):
    ctx.debug_wait_timeout(20_000_000)
    st = ctx.device_status()
    assert st & mla.DEVICE_TIMEOUT
    # the context is still usable
    test_expand_v(mla, ctx, 5, 1, 16)
    assert ctx.device_status() == 0


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("B,Hq,H,n", [(64, 1, 16, 64), (5, 2, 128, 7), (3, 1, 32, 0)])
def test_append_absorb_q_matches_the_two_calls(mla, ctx, fp8, B, Hq, H, n):
    # the fused launch writes exactly what append_latent + absorb_q write
    w = _normal(f"aaq/w/{H}", (H, 128, 512), std=0.02)
    qn = _normal(f"aaq/qn/{B}/{H}", (B, Hq, H, 128))
    qr = _normal(f"aaq/qr/{B}/{H}", (B, Hq, H, 64))
    qpos = torch.tensor(S.uniform_ints(6, f"aaq/pos/{B}", B * Hq, 0, 4000), dtype=torch.int32).view(B, Hq).cuda()
    c = _normal(f"aaq/c/{n}", (max(n, 1), 512))[:n].contiguous()
    k = _normal(f"aaq/k/{n}", (max(n, 1), 64))[:n].contiguous()
    seq = torch.tensor([i % 4 for i in range(n)], dtype=torch.int32, device="cuda")
    pos = torch.tensor([i // 4 * 3 for i in range(n)], dtype=torch.int32, device="cuda")
    caches = [mla.Cache.contiguous(4, 64, fp8=fp8) for _ in range(2)]
    ctx.append_latent(caches[0], c, k, seq, pos)
    q0 = ctx.absorb_q(w, qn, qr, qpos)
    q1 = ctx.append_absorb_q(caches[1], c, k, seq, pos, w, qn, qr, qpos)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    assert torch.equal(caches[0].storage, caches[1].storage)
    assert torch.equal(q0, q1)


# ----------------------------------------------------------------- copy kernel
@pytest.mark.parametrize("nbytes", [16, 4096 + 48, 468992, (1 << 22) + 16])
def test_copy_async_between_host_and_device(mla, ctx, nbytes):
    block = np.array(S.uniform_ints(13, "cp/block", 4096, 0, 255), dtype=np.uint8)
    data = np.resize(block, nbytes) ^ (np.arange(nbytes) >> 12).astype(np.uint8)   # no two 4 KB pages alike
    src_host = torch.from_numpy(data).pin_memory()
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ctx.copy_async(dev, src_host)                       # host -> device
    dev2 = torch.empty_like(dev)
    ctx.copy_async(dev2, dev)                           # device -> device
    back = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    ctx.copy_async(back, dev2)                          # device -> host
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), src_host)
    assert torch.equal(back, src_host)


def test_copy_async_rejects_bad_arguments(mla, ctx):
    a = torch.zeros(64, dtype=torch.uint8, device="cuda")
    b = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(RuntimeError):
        ctx.copy_async(a[8:24], b[:16])                 # dst not 16-byte aligned
    with pytest.raises(RuntimeError):
        ctx.copy_async(a[:24], b[:24])                  # not a multiple of 16 bytes
    with pytest.raises(RuntimeError):
        ctx.copy_async(a[16:48], a[:32])                # overlapping ranges
    with pytest.raises(ValueError):
        ctx.copy_async(a[:16], torch.zeros(16, dtype=torch.uint8))   # pageable host memory
