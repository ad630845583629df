"""The FP8 latent cache through the C ABI: the append's bytes against the
oracle's FP8 row writer (bit-exact), the attention against the oracle's
attention over the rows the FP8 cache stands for, and a whole decode step."""
import numpy as np
import pytest
import torch

import mla_synth as S
import oracle as O
from mla_testlib import (MAX_ABS, REL_L2, Problem, SCALE, assert_close, bits, f64, fill_cache, gpu_step, make_cache,
                         oracle_absorbed, oracle_absorbed_fp8, rel_l2)

pytestmark = pytest.mark.gpu


def _u8(t):
    return t.detach().cpu().contiguous().numpy().view(np.uint8)


# ----------------------------------------------------------------- append
@pytest.mark.parametrize("paged", [False, True])
def test_append_fp8_bit_exact(mla, ctx, paged):
    B, n = 3, 160
    c = S.normal_bf16(21, f"a8/c/{paged}", (n, 512), device="cuda")
    k = S.normal_bf16(21, f"a8/k/{paged}", (n, 64), device="cuda")
    # special latents: zero, tiny (scale floor, subnormal codes), amax exactly
    # 448 * 2^3, huge, and a row with one large value among small ones
    c[1] = 0
    c[2] = (c[2].float() * 2.0 ** -70).to(torch.bfloat16)
    c[3, 5] = 448.0 * 8
    c[4] = (c[4].float() * 2.0 ** 100).to(torch.bfloat16)
    c[5] = (c[5].float() * 1e-3).to(torch.bfloat16)
    c[5, 0] = 300.0
    c[6, ::2] = -c[6, ::2]
    seq = torch.tensor([i % B for i in range(n)], dtype=torch.int32)
    pos = torch.tensor([i // B * 3 + 1 for i in range(n)], dtype=torch.int32)
    L = int(pos.max()) + 1
    if paged:
        nblk = (L + 63) // 64
        perm = S.permutation(22, "a8/perm", B * nblk + 2)
        table = torch.tensor(perm[:B * nblk], dtype=torch.int32).view(B, nblk)
        cache = mla.Cache.paged_pool(B * nblk + 2, table, fp8=True)
        rows = [O.paged_row(int(s_), int(t_), table.tolist()) for s_, t_ in zip(seq, pos)]
    else:
        cache = mla.Cache.contiguous(B, L, fp8=True)
        rows = [O.contiguous_row(int(s_), int(t_), L) for s_, t_ in zip(seq, pos)]
    ctx.append_latent(cache, c.contiguous(), k.contiguous(), seq.cuda(), pos.cuda())
    assert ctx.device_status() == 0
    got = _u8(cache.storage).reshape(-1, 656)
    want = np.zeros_like(got)
    want[rows] = O.fp8_cache_rows(bits(c), bits(k), pos.numpy())
    assert np.array_equal(got, want), int(np.count_nonzero(got != want))


def test_append_fp8_out_of_range_sets_bounds(mla, ctx):
    cache = mla.Cache.contiguous(2, 16, fp8=True)
    c = S.normal_bf16(23, "a8/oob/c", (2, 512), device="cuda")
    k = S.normal_bf16(23, "a8/oob/k", (2, 64), device="cuda")
    ctx.append_latent(cache, c, k, torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                      torch.tensor([4, 16], dtype=torch.int32, device="cuda"))
    assert ctx.device_status() & mla.DEVICE_BOUNDS
    got = _u8(cache.storage).reshape(-1, 656)
    assert np.array_equal(got[4], O.fp8_cache_rows(bits(c[:1]), bits(k[:1]), [4])[0])
    assert np.count_nonzero(np.delete(got, 4, axis=0)) == 0


# ----------------------------------------------------------------- attention
def _attn8_case(mla, ctx, H, Hq, lens, paged, q_std=1.0, units=0, seed=31, c_std=1.0):
    """Oracle FP8 rows written straight into the cache (every other slot filled
    with 0xFF bytes: NaN codes and a NaN scale), random q_abs, decode_attn vs the
    oracle's attention over the dequantised rows."""
    B = len(lens)
    G = Hq * H
    rows_b = []
    for b, L in enumerate(lens):
        c = S.normal_bf16(seed, f"a8t/c/{b}", (L, 512), std=c_std, device="cuda")
        k = S.normal_bf16(seed, f"a8t/k/{b}", (L, 64), device="cuda")
        rows_b.append(O.fp8_cache_rows(bits(c), bits(k), np.arange(L)))
    if paged:
        nblk = [(L + 63) // 64 for L in lens]
        perm = S.permutation(seed, "a8t/perm", sum(nblk) + 3)
        table = torch.full((B, max(nblk)), -1, dtype=torch.int32)
        o = 0
        for b in range(B):
            table[b, :nblk[b]] = torch.tensor(perm[o:o + nblk[b]], dtype=torch.int32)
            o += nblk[b]
        cache = mla.Cache.paged_pool(sum(nblk) + 3, table, fp8=True)
        host = np.full((cache.storage.numel() // 656, 656), 0xFF, dtype=np.uint8)
        for b, L in enumerate(lens):
            for t in range(L):
                host[O.paged_row(b, t, table.tolist())] = rows_b[b][t]
    else:
        cap = max(lens) + 5
        cache = mla.Cache.contiguous(B, cap, fp8=True)
        host = np.full((B * cap, 656), 0xFF, dtype=np.uint8)
        for b, L in enumerate(lens):
            host[b * cap:b * cap + L] = rows_b[b]
    cache.storage.copy_(torch.from_numpy(host).view_as(cache.storage))
    q = S.normal_bf16(seed, "a8t/q", (B, Hq, H, 576), std=q_std, device="cuda")
    seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ctx.set_decode_units(units)
    try:
        o_lat, lse = ctx.decode_attn(cache, q, seq_lens, SCALE)
        torch.cuda.synchronize()
    finally:
        ctx.set_decode_units(0)
    assert ctx.device_status() == 0
    qh = f64(q).reshape(B, G, 576)
    want_o = np.zeros((B, G, 512))
    want_l = np.zeros((B, G))
    for b, L in enumerate(lens):
        lim = [L - Hq + 1 + g // H for g in range(G)]
        o, l, _ = O.latent_attention(qh[b], O.fp8_rows_dequantize(rows_b[b]), SCALE, lim)
        want_o[b], want_l[b] = o, l
    got_o = f64(o_lat).reshape(B, G, 512)
    got_l = f64(lse).reshape(B, G)
    # o_lat is a convex combination of latents of size ~c_std: the absolute
    # bar (set for unit-size values) scales with it, the relative one does not
    assert_close(got_o, want_o, max_abs=1e-2 * max(1.0, c_std), what="o_lat (fp8 cache)")
    assert np.max(np.abs(got_l - want_l)) <= 5e-3, float(np.max(np.abs(got_l - want_l)))
    return got_o, got_l


@pytest.mark.parametrize("H,Hq,lens,paged", [
    (16, 1, [1], False),
    (16, 1, [26], False),
    (16, 1, [63, 64, 65, 127, 128, 129, 300], False),
    (16, 2, [2, 130, 257], False),
    (32, 1, [200, 1], True),
    (64, 1, [129, 640], True),
    (128, 1, [300, 64, 1000, 129], True),
    (128, 2, [517, 2], True),
    (16, 64, [64, 700], False),           # prefill chunk: 1024 query rows per sequence
    (128, 16, [16, 40], True),            # 2048 query rows per sequence
    (16, 200, [300, 200], False),         # 3,200 rows: 50 CTAs a unit, split over 3 units
    (16, 640, [700], False),              # 10,240 rows: more CTAs than SMs, one unit in waves
])
def test_decode_attn_fp8_vs_oracle(mla, ctx, H, Hq, lens, paged):
    _attn8_case(mla, ctx, H, Hq, lens, paged)


@pytest.mark.parametrize("H", [16, 128])
def test_decode_attn_fp8_peaky_scores(mla, ctx, H):
    # large queries: the running max moves often and most weights are tiny
    _attn8_case(mla, ctx, H, 1, [1000, 517], True, q_std=6.0)


def test_decode_attn_fp8_latent_scales(mla, ctx):
    # latents far from unit size: the token scales enter the logits and weights
    _attn8_case(mla, ctx, 16, 1, [700, 300], False, c_std=2.0 ** -20)
    _attn8_case(mla, ctx, 16, 1, [700, 300], False, c_std=2.0 ** 12, q_std=2.0 ** -12)


@pytest.mark.parametrize("H,Hq", [(16, 1), (128, 2)])
def test_decode_attn_fp8_split_kv(mla, ctx, H, Hq):
    lens = [900, 31, 1200, 5]
    # each cut passes the oracle bar; between cuts the weights P' are rounded
    # (e4m3 hi + lo, about 2^-8 relative) against different running maxima, so
    # the results agree to that rounding rather than to float32 summation order
    one, _ = _attn8_case(mla, ctx, H, Hq, lens, True, units=1)
    seven, _ = _attn8_case(mla, ctx, H, Hq, lens, True, units=7)
    many, _ = _attn8_case(mla, ctx, H, Hq, lens, True, units=0)
    for other in (seven, many):
        assert np.linalg.norm(other - one) <= 1e-3 * np.linalg.norm(one)
        assert np.max(np.abs(other - one)) <= 5e-3


# ----------------------------------------------------------------- decode step
@pytest.mark.parametrize("idx,scale_down", [(1, 16), (2, 32)])
def test_decode_step_fp8_cache(mla, ctx, idx, scale_down):
    """append (FP8) -> absorb_q -> decode_attn (FP8) -> expand_v against the
    absorbed oracle over the latent the FP8 rows stand for."""
    wl = S.make_config(idx, scale_down=scale_down)
    wl.B = min(wl.B, 8)
    wl.seq_lens = wl.seq_lens[:wl.B]
    if wl.paged:
        wl.block_table = wl.block_table[:wl.B]
    prob = Problem(wl)
    cache = make_cache(mla, wl, fp8=True)
    fill_cache(ctx, cache, prob)
    out, o_lat, lse = gpu_step(ctx, cache, prob)
    assert ctx.device_status() == 0
    for b in range(wl.B):
        o, ol, l = oracle_absorbed_fp8(prob, b)
        assert_close(f64(out)[b], o, what=f"out[b={b}]")
        assert_close(f64(o_lat)[b], ol, what=f"o_lat[b={b}]")
        assert np.max(np.abs(f64(lse)[b] - l)) <= 5e-3


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_decode_step_fp8_full_size_sampled(mla, ctx, idx):
    """The FP8 decode workloads at full size (every sequence through the step,
    sampled sequences checked, all heads): against the oracle over the latent the
    FP8 rows stand for, within the bf16 bars; and against the bf16-input oracle,
    where the gap is the format's own rounding of the latent: the output's
    relative L2 error stays within 1.5x the rows' rms relative rounding error (the
    weights average independent per-element errors) plus the kernel's bar."""
    wl = S.make_config(idx)
    samples = {1: [0, 37, 63], 2: [0, 31], 3: [0, 64, 127]}[idx]
    prob = Problem(wl)
    cache = make_cache(mla, wl, fp8=True)
    fill_cache(ctx, cache, prob)
    out, o_lat, lse = gpu_step(ctx, cache, prob)
    assert ctx.device_status() == 0
    got_out, got_lat, got_lse = f64(out), f64(o_lat), f64(lse)
    for b in samples:
        o, ol, l = oracle_absorbed_fp8(prob, b)
        assert_close(got_out[b], o, what=f"out[b={b}] vs oracle over FP8 rows")
        assert_close(got_lat[b], ol, what=f"o_lat[b={b}] vs oracle over FP8 rows")
        assert np.max(np.abs(got_lse[b] - l)) <= 5e-3
        ob, _, _ = oracle_absorbed(prob, b)
        c, k = prob.token_inputs(b)
        c64 = f64(c)
        deq = O.fp8_rows_dequantize(O.fp8_cache_rows(bits(c), bits(k), np.arange(len(c64))))[:, :512]
        q_rms = float(np.sqrt(np.mean((deq - c64) ** 2) / np.mean(c64 ** 2)))
        r = rel_l2(got_out[b], ob)
        assert r <= 1.5 * q_rms + REL_L2, (r, q_rms)
        assert float(np.max(np.abs(got_out[b] - ob))) <= MAX_ABS


def _tail_case(mla, ctx, H, units):
    """One sequence of 32,768 FP8 rows: token 0 holds the dominant score and the
    other tokens form two interleaved tails whose scores sit 20 and 26 (log2
    units) below it. The query is nonzero only in latent column 0, so a row's
    score is set by its column 0; column 1 is 28 in every row, which gives every
    row the same scale sigma = 2^-4 (the cutoff acts on weight x sigma); columns
    2..511 of a tail are one fixed vector, so a tail's weight shows in the
    output as a whole. Returns the output [H, 512], the dequantised rows and the
    query."""
    L = 32768
    qa = 9.625                                   # scale * log2(e) * qa ~ 1
    k2 = SCALE * qa / np.log(2.0)
    vec = [S.normal_bf16(77, f"tail/vec/{g}", (510,)).float() for g in range(3)]
    c = torch.empty(L, 512, dtype=torch.float32)
    grp = np.zeros(L, dtype=np.int64)
    grp[1:] = 1 + (np.arange(1, L) % 2)          # 1, 2: tails at -20, -26
    off = np.array([0.0, -20.0, -26.0])
    for g in range(3):
        idx = torch.from_numpy(np.nonzero(grp == g)[0])
        c[idx, 0] = float(off[g] / k2)
        c[idx, 1] = 28.0
        c[idx, 2:] = vec[g]
    c = c.to(torch.bfloat16)
    k = S.normal_bf16(77, "tail/k", (L, 64))
    rows = O.fp8_cache_rows(bits(c), bits(k), np.arange(L))
    cache = mla.Cache.contiguous(1, L, fp8=True)
    cache.storage.copy_(torch.from_numpy(rows).view_as(cache.storage))
    q = torch.zeros(1, 1, H, 576, dtype=torch.float32)
    q[..., 0] = qa
    q = q.to(torch.bfloat16).cuda()
    ctx.set_decode_units(units)
    try:
        o_lat, lse = ctx.decode_attn(cache, q, torch.tensor([L], dtype=torch.int32, device="cuda"), SCALE)
        torch.cuda.synchronize()
    finally:
        ctx.set_decode_units(0)
    assert ctx.device_status() == 0
    deq = O.fp8_rows_dequantize(rows)
    sig = rows[:, 640:644].copy().view(np.float32)[:, 0]
    assert np.all(sig == 2.0 ** -4)
    return f64(o_lat)[0, 0], deq, f64(q)[0, 0, 0]


def _attention_with_cutoff(rows, q, cutoff):
    """Softmax attention of one query over the rows (float64), weights below
    `cutoff` times the largest weight set to zero (cutoff 0: the exact attention)."""
    s = SCALE * (rows @ q)
    w = np.exp(s - s.max())
    w[w < cutoff] = 0.0
    return (w @ rows[:, :512]) / w.sum()


def _per_head_close(got, want, what):
    # every head sees the same query; compare the content columns 2..511
    for h in range(got.shape[0]):
        assert_close(got[h, 2:], want[2:], what=f"{what}, head {h}")


@pytest.mark.parametrize("H", [16, 32, 128])
def test_decode_attn_fp8_long_tail_near_cutoff(mla, ctx, H):
    """The documented weight cutoff of the FP8 attention, pinned on 32k tokens.
    One unit walks the whole sequence, so the running max is token 0's from the
    first tile on: with Hq*H <= 32 the cutoff is 2^-22, so the tail at 2^-20 is
    carried and the one at 2^-26 dropped (11k x 2^-26 of the mass, which the
    exact attention cannot tell apart); with Hq*H = 128 the cutoff is 2^-18, so
    the 2^-20 tail (1 % of the mass, one direction) is dropped as well and the
    output moves measurably away from the exact attention. With the default
    split over all SMs every unit has its own running max, the 2^-20 tail stays
    above every unit's cutoff, and the output is the exact attention."""
    got, rows, q = _tail_case(mla, ctx, H, units=1)
    exact = _attention_with_cutoff(rows, q, 0.0)
    if H <= 32:
        _per_head_close(got, exact, f"H={H}, one unit")
    else:
        _per_head_close(got, _attention_with_cutoff(rows, q, 2.0 ** -18),
                        f"H={H}, one unit, weights below 2^-18 dropped")
        assert rel_l2(got[0, 2:], exact[2:]) > REL_L2          # the drop is real and documented
    got_split, _, _ = _tail_case(mla, ctx, H, units=0)
    _per_head_close(got_split, exact, f"H={H}, split over all units")


# ----------------------------------------------------------------- edge cases
def test_decode_attn_fp8_max_batch_and_short_sequences(mla, ctx):
    # 1024 sequences (the per-call maximum) with lengths 1..120 drawn from the
    # seed (one unit holds many sequences), then lengths below Hq flagged
    lens = [max(1, L) for L in S.uniform_ints(41, "a8/maxb/lens", 1024, 0, 120)]
    got, _ = _attn8_case(mla, ctx, 16, 1, lens, False, seed=41)
    assert got.shape == (1024, 16, 512)
    cache = mla.Cache.contiguous(8, 64, fp8=True)
    q = torch.zeros(8, 2, 16, 576, dtype=torch.bfloat16, device="cuda")
    o_lat, lse = ctx.decode_attn(cache, q, torch.tensor([5, 1, 3, 0, 2, 64, 1, 7], dtype=torch.int32,
                                                         device="cuda"), SCALE)
    assert ctx.device_status() & mla.DEVICE_LENGTH
    short = [1, 3, 6]                       # lengths 1, 0, 1 are below Hq = 2
    assert torch.all(torch.isneginf(lse[short]))
    assert torch.all(o_lat[short] == 0)


def test_decode_attn_fp8_bad_block_table_sets_bounds(mla, ctx):
    # a block id outside the pool: the tile's copy is skipped and the bounds
    # bit is set (no fault); the other sequence's output is still exact
    lens = [200, 130]
    table = torch.tensor([[0, 1, 2, 3], [4, 5, 99, -1]], dtype=torch.int32)   # block 99 does not exist
    cache = mla.Cache.paged_pool(8, table, fp8=True)
    rows = []
    for b, L in enumerate(lens):
        c = S.normal_bf16(43, f"a8/bt/c/{b}", (L, 512), device="cuda")
        k = S.normal_bf16(43, f"a8/bt/k/{b}", (L, 64), device="cuda")
        rows.append(O.fp8_cache_rows(bits(c), bits(k), np.arange(L)))
    host = np.zeros((8 * 64, 656), dtype=np.uint8)
    for t in range(lens[0]):
        host[O.paged_row(0, t, table.tolist())] = rows[0][t]
    for t in range(128):                    # sequence 1: only its first two blocks exist
        host[O.paged_row(1, t, table.tolist())] = rows[1][t]
    cache.storage.copy_(torch.from_numpy(host).view_as(cache.storage))
    q = S.normal_bf16(43, "a8/bt/q", (2, 1, 16, 576), device="cuda")
    o_lat, lse = ctx.decode_attn(cache, q, torch.tensor(lens, dtype=torch.int32, device="cuda"), SCALE)
    torch.cuda.synchronize()
    assert ctx.device_status() & mla.DEVICE_BOUNDS
    want, _, _ = O.latent_attention(f64(q)[0, 0], O.fp8_rows_dequantize(rows[0]), SCALE, [lens[0]] * 16)
    assert_close(f64(o_lat)[0, 0], want, what="o_lat of the intact sequence")


# ----------------------------------------------------------------- random shapes
@pytest.mark.parametrize("case", range(8))
def test_decode_attn_random_shapes(mla, ctx, case):
    # seeded draws of heads, query tokens, batch, lengths, layout, unit count
    # and cache format, each against the oracle
    r = S.uniform_ints(70 + case, "rand/shape", 6, 0, 1 << 20)
    H = [16, 32, 64, 128][r[0] % 4]
    Hq = 1 + r[1] % 2
    B = 1 + r[2] % 6
    lens = [max(Hq, L) for L in S.uniform_ints(80 + case, "rand/lens", B, 1, 2500)]
    paged = bool(r[3] % 2)
    units = [0, 3, 17][r[4] % 3]
    fp8 = bool(r[5] % 2)
    if fp8:
        _attn8_case(mla, ctx, H, Hq, lens, paged, units=units, seed=90 + case)
    else:
        from test_gpu_kernels import _attn_case
        _attn_case(mla, ctx, H, Hq, lens, paged, units=units, seed=90 + case)
