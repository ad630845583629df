"""The one-launch decode step for short sequences (mla_decode_step_small)
through the C ABI: against the float64 oracle on the same raw inputs, against
the four-call path, the new token's cache row against the oracle's writer
(bit-exact), out-of-range lengths, and graph replay of the step object."""
import numpy as np
import pytest
import torch

import mla_synth as S
import oracle as O
from mla_testlib import (Problem, SCALE, assert_close, bits, f64, make_cache, oracle_absorbed, oracle_naive)

pytestmark = pytest.mark.gpu


def _prefill_all_but_last(ctx, cache, prob):
    """Tokens 0 .. L-2 of every sequence through mla_append_latent; returns the
    last tokens' (c_kv [B, 512], k_rope [B, 64])."""
    wl = prob.wl
    cs, ks = [], []
    for b, L in enumerate(wl.seq_lens):
        c, k = S.token_inputs(wl, b, device="cuda")
        if L > 1:
            ctx.append_latent(cache, c[:L - 1].contiguous(), k[:L - 1].contiguous(),
                              torch.full((L - 1,), b, dtype=torch.int32, device="cuda"),
                              torch.arange(L - 1, dtype=torch.int32, device="cuda"))
        cs.append(c[L - 1])
        ks.append(k[L - 1])
    return torch.stack(cs).contiguous(), torch.stack(ks).contiguous()


def _run_small(mla, ctx, wl):
    prob = Problem(wl)
    cache = make_cache(mla, wl)
    c_new, k_new = _prefill_all_but_last(ctx, cache, prob)
    out, o_lat, lse = ctx.decode_step_small(cache, c_new, k_new, prob.w_uk, prob.w_uv, prob.q_nope, prob.q_rope,
                                            prob.seq_lens, SCALE)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    return prob, cache, out, o_lat, lse


def _check(prob, out, o_lat, lse, naive_heads=(0,)):
    for b in range(prob.wl.B):
        o, ol, l = oracle_absorbed(prob, b)
        assert_close(f64(out)[b], o, what=f"out[b={b}]")
        assert_close(f64(o_lat)[b], ol, what=f"o_lat[b={b}]")
        assert np.max(np.abs(f64(lse)[b] - l)) <= 5e-3
        if naive_heads:
            on = oracle_naive(prob, b, list(naive_heads))
            assert_close(f64(out)[b][:, list(naive_heads)], on, what=f"out vs naive[b={b}]")


def test_small_step_v2lite_single_step(mla, ctx):
    """B=1, H=16, L=26 (25 cached + the step's token): outputs against the
    oracle (all heads, naive and absorbed) and the new row bit-exact."""
    wl = S.make_config(0)
    prob, cache, out, o_lat, lse = _run_small(mla, ctx, wl)
    _check(prob, out, o_lat, lse, naive_heads=range(16))
    c, k = prob.token_inputs(0)
    want_rows = O.cache_rows(bits(c), bits(k), np.arange(26))
    got = bits(cache.storage).reshape(-1, 576)[:26]
    assert np.array_equal(got, want_rows)


@pytest.mark.parametrize("H,lens,paged", [(16, [1, 2, 63, 130, 700], True), (128, [5, 129, 300], False),
                                          (32, [4096, 17], True)])
def test_small_step_ragged_batches(mla, ctx, H, lens, paged):
    if paged:
        tbl, nb, mb = S._paged_tables(9, "small", lens)
        wl = S.Workload(f"small_h{H}", len(lens), H, 1, lens, True, block_table=tbl, num_blocks=nb, max_blocks=mb,
                        seed=9)
    else:
        wl = S.Workload(f"small_h{H}", len(lens), H, 1, lens, False, capacity=max(lens) + 3, seed=9)
    prob, cache, out, o_lat, lse = _run_small(mla, ctx, wl)
    _check(prob, out, o_lat, lse, naive_heads=(1,))


def test_small_step_matches_four_call_path(mla, ctx):
    lens = [26, 200, 513]
    wl = S.Workload("small_vs_four", 3, 16, 1, lens, False, capacity=600, seed=10)
    prob = Problem(wl)
    cache_a = make_cache(mla, wl)
    cache_b = make_cache(mla, wl)
    c_new, k_new = _prefill_all_but_last(ctx, cache_a, prob)
    _prefill_all_but_last(ctx, cache_b, prob)
    out_s, lat_s, lse_s = ctx.decode_step_small(cache_a, c_new, k_new, prob.w_uk, prob.w_uv, prob.q_nope,
                                                prob.q_rope, prob.seq_lens, SCALE)
    ctx.append_latent(cache_b, c_new, k_new, torch.arange(3, dtype=torch.int32, device="cuda"),
                      (prob.seq_lens - 1).contiguous())
    out_f, lat_f, lse_f = ctx.decode_step(cache_b, prob.w_uk, prob.w_uv, prob.q_nope, prob.q_rope, prob.q_pos,
                                          prob.seq_lens, SCALE)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    assert torch.equal(cache_a.storage, cache_b.storage)     # the same rows written
    assert_close(f64(out_s), f64(out_f), what="one launch vs four calls: out")
    assert_close(f64(lat_s), f64(lat_f), what="one launch vs four calls: o_lat")


def test_small_step_length_out_of_range(mla, ctx):
    wl = S.Workload("small_len", 2, 16, 1, [3, 3], False, capacity=8, seed=11)
    prob = Problem(wl)
    cache = make_cache(mla, wl)
    c_new, k_new = _prefill_all_but_last(ctx, cache, prob)
    for bad in (0, ctx.lib.mla_small_step_max_len() + 1):
        lens = torch.tensor([3, bad], dtype=torch.int32, device="cuda")
        out, o_lat, lse = ctx.decode_step_small(cache, c_new, k_new, prob.w_uk, prob.w_uv, prob.q_nope, prob.q_rope,
                                                lens, SCALE)
        torch.cuda.synchronize()
        assert ctx.device_status() & mla.DEVICE_LENGTH
        assert float(f64(out)[1].max()) == 0.0 and float(f64(out)[1].min()) == 0.0
        assert np.all(np.isneginf(f64(lse)[1]))
        o, _, _ = oracle_absorbed(prob, 0)
        assert_close(f64(out)[0], o, what="the valid sequence beside it")


def test_small_step_object_graph_replay(mla, ctx):
    wl = S.make_config(0)
    prob = Problem(wl)
    cache = make_cache(mla, wl)
    c_new, k_new = _prefill_all_but_last(ctx, cache, prob)
    st = mla.DecodeStep(ctx, cache, prob.w_uk, prob.w_uv, 1, 1, small=True)
    st.c_kv.copy_(c_new)
    st.k_rope.copy_(k_new)
    st.q_nope.copy_(prob.q_nope)
    st.q_rope.copy_(prob.q_rope)
    st.seq_lens.copy_(prob.seq_lens)
    st.run()
    torch.cuda.synchronize()
    direct = st.out.clone()
    st.capture(3)
    st.out.zero_()
    st.replay()
    torch.cuda.synchronize()
    assert torch.equal(st.out, direct)
    assert ctx.device_status() == 0
    _check(prob, st.out, st.o_lat, st.lse, naive_heads=(0,))
