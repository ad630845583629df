"""End-to-end decode step (append -> absorb_q -> decode_attn -> expand_v) through
the C ABI, against the float64 oracle on the same raw bf16 inputs.

Small cases span several 128-token tiles and ragged tails and are checked on
every output; the full-size workloads are checked on sampled sequences (all
heads, absorbed oracle) plus a sampled head against the naive oracle.
"""
import numpy as np
import pytest
import torch

import mla_synth as S
from mla_testlib import (Problem, SCALE, assert_close, f64, fill_cache, gpu_step, make_cache,
                         oracle_absorbed, oracle_naive)

pytestmark = pytest.mark.gpu


def _check_sequences(prob, out, o_lat, lse, seqs, naive_heads=(0,)):
    wl = prob.wl
    got_out = f64(out)
    got_lat = f64(o_lat)
    got_lse = f64(lse)
    for b in seqs:
        o, ol, l = oracle_absorbed(prob, b)
        assert_close(got_out[b], o, what=f"out[b={b}]")
        assert_close(got_lat[b], ol, what=f"o_lat[b={b}]")
        assert np.max(np.abs(got_lse[b] - l)) <= 5e-3
        if naive_heads:
            on = oracle_naive(prob, b, list(naive_heads))
            assert_close(got_out[b][:, list(naive_heads)], on, what=f"out vs naive[b={b}]")


def _run(mla, ctx, wl, seqs=None, naive_heads=(0,)):
    prob = Problem(wl)
    cache = make_cache(mla, wl)
    fill_cache(ctx, cache, prob)
    out, o_lat, lse = gpu_step(ctx, cache, prob)
    assert ctx.device_status() == 0
    _check_sequences(prob, out, o_lat, lse, range(wl.B) if seqs is None else seqs, naive_heads)
    return prob, cache, out


def test_config0_v2lite_single_step(mla, ctx):
    """B=1, H=16, L=26 (25 prefill + 1 decode), contiguous cache of 32 slots."""
    wl = S.make_config(0)
    prob = Problem(wl)
    cache = make_cache(mla, wl)
    # prefill the first 25 tokens, then append the decode token on its own
    c, k = S.token_inputs(wl, 0, device="cuda")
    seq = torch.zeros(26, dtype=torch.int32, device="cuda")
    pos = torch.arange(26, dtype=torch.int32, device="cuda")
    ctx.append_latent(cache, c[:25].contiguous(), k[:25].contiguous(), seq[:25], pos[:25])
    ctx.append_latent(cache, c[25:].contiguous(), k[25:].contiguous(), seq[25:], pos[25:])
    out, o_lat, lse = gpu_step(ctx, cache, prob)
    assert ctx.device_status() == 0
    _check_sequences(prob, out, o_lat, lse, [0], naive_heads=range(16))


@pytest.mark.parametrize("idx,scale_down", [(1, 16), (2, 32), (3, 64), (4, 512)])
def test_configs_scaled_down(mla, ctx, idx, scale_down):
    wl = S.make_config(idx, scale_down=scale_down)
    if idx == 1:
        wl.B = 8
        wl.seq_lens = wl.seq_lens[:8]
    _run(mla, ctx, wl, naive_heads=(0, wl.H - 1))


def test_ragged_lengths_small(mla, ctx):
    lens = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 1000]
    tbl, nb, mb = S._paged_tables(3, "ragged", lens)
    wl = S.Workload("ragged_small", len(lens), 128, 1, lens, True, block_table=tbl, num_blocks=nb, max_blocks=mb,
                    seed=3)
    _run(mla, ctx, wl, naive_heads=(5,))


def test_step_then_output_projection(mla, ctx):
    """The decode step followed by the attention block's output projection, against
    the naive oracle's per-head outputs projected by the same W_O (d_model = 2048)."""
    import oracle as O
    wl = S.make_config(1, scale_down=16)
    wl.B = 4
    wl.seq_lens = wl.seq_lens[:4]
    prob, cache, out = _run(mla, ctx, wl, naive_heads=())
    w_o = S.normal_bf16(7, "e2e/w_o", (2048, wl.H * 128), std=0.02, device="cuda")
    y = ctx.out_proj(w_o, out)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    got = f64(y).reshape(wl.B, wl.Hq, 2048)
    for b in range(wl.B):
        o_naive = oracle_naive(prob, b, list(range(wl.H)))
        want = O.output_projection(o_naive, f64(w_o))
        assert_close(got[b], want, what=f"y[b={b}]")


def test_prefill_from_empty_cache_matches_one_shot_causal(mla, ctx):
    """Prefill of a whole prompt as one step: L = Hq = 96 query tokens at positions
    0..95 over a cache that holds exactly those tokens, against the one-shot
    causal forward of the naive path (all heads)."""
    import oracle as O
    L = 96
    wl = S.Workload("prefill_b1_h16_l96", 1, 16, L, [L], False, capacity=L, seed=5)
    prob, cache, out = _run(mla, ctx, wl, naive_heads=(0, 15))
    c, k = prob.token_inputs(0)
    h = prob.host
    want = O.naive_prefill_causal(f64(c), f64(k), h["q_nope"][0], h["q_rope"][0], h["w_uk"], h["w_uv"], SCALE)
    assert_close(f64(out)[0], want, what="prefill vs one-shot causal")


@pytest.mark.parametrize("H,Hq,lens,paged", [(16, 48, [130, 300], False), (128, 8, [40, 700], True),
                                            (16, 256, [300, 521], False),    # 4,096 rows: 64 CTAs a unit, split
                                            (16, 1024, [1024, 1100], True),  # 16,384 rows: one unit, waves
                                            (128, 24, [24, 900], True),      # 3,072 rows: split over 2 units
                                            (128, 160, [200, 460], True)])   # 20,480 rows: one unit, more
                                                                             # row-group pairs than fit
def test_prefill_chunk_after_cached_prefix(mla, ctx, H, Hq, lens, paged):
    """A chunk of Hq new tokens appended after a cached prefix (chunked prefill),
    from a few rows per sequence up to chunks whose CTAs outnumber the SMs (the
    call then runs as one unit, each CTA stopping at its causal limit; on CTA
    pairs, the pairs that fit each walk several row groups)."""
    if paged:
        tbl, nb, mb = S._paged_tables(6, "chunk", lens)
        wl = S.Workload(f"chunk_h{H}", len(lens), H, Hq, lens, True, block_table=tbl, num_blocks=nb, max_blocks=mb,
                        seed=6)
    else:
        wl = S.Workload(f"chunk_h{H}", len(lens), H, Hq, lens, False, capacity=max(lens), seed=6)
    _run(mla, ctx, wl, naive_heads=(1,))


def test_long_prompt_h128_in_one_call(mla, ctx):
    """A 1,024-token prompt at H = 128 prefilled in one decode_attn call (131,072
    query rows: 2,048 CTAs of 64 rows in waves, one unit), from an empty cache,
    against the one-shot causal forward of the naive path on sampled heads."""
    import oracle as O
    L = 1024
    wl = S.Workload("prompt_b1_h128_l1024", 1, 128, L, [L], True, seed=8,
                    **dict(zip(("block_table", "num_blocks", "max_blocks"), S._paged_tables(8, "prompt", [L]))))
    assert ctx.workspace_size(128, 1, L) == 256
    prob = Problem(wl)
    cache = make_cache(mla, wl)
    fill_cache(ctx, cache, prob)
    out, o_lat, lse = gpu_step(ctx, cache, prob)
    assert ctx.device_status() == 0
    heads = [0, 37, 127]
    c, k = prob.token_inputs(0)
    h = prob.host
    want = O.naive_prefill_causal(f64(c), f64(k), h["q_nope"][0][:, heads], h["q_rope"][0][:, heads],
                                  h["w_uk"][heads], h["w_uv"][heads], SCALE)
    assert_close(f64(out)[0][:, heads], want, what="1k-token prompt vs one-shot causal")
    # the rows of the first and the last query token: exact softmax in latent space
    ol = f64(o_lat)[0]
    for j in (0, L - 1):
        o, ol_want, l_want = O.absorbed_decode(f64(c)[:j + 1], f64(k)[:j + 1], h["q_nope"][0][j:j + 1],
                                               h["q_rope"][0][j:j + 1], h["w_uk"], h["w_uv"], SCALE, [j])
        assert_close(ol[j], ol_want[0], what=f"o_lat of query token {j}")


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_configs_full_size_sampled(mla, ctx, idx):
    wl = S.make_config(idx)
    samples = {1: [0, 37, 63], 2: [0, 31], 3: [0, 64, 127], 4: [0, 3]}[idx]
    _run(mla, ctx, wl, seqs=samples, naive_heads=(1,) if idx != 4 else ())


def test_decode_step_graph_replay_matches_direct(mla, ctx):
    """DecodeStep: the captured CUDA graph computes exactly the direct launches."""
    wl = S.make_config(1, scale_down=16)
    wl.B = 8
    wl.seq_lens = wl.seq_lens[:8]
    prob = Problem(wl)
    cache = make_cache(mla, wl)
    fill_cache(ctx, cache, prob)
    st = mla.DecodeStep(ctx, cache, prob.w_uk, prob.w_uv, wl.B, wl.Hq)
    last = torch.tensor([L - 1 for L in wl.seq_lens], dtype=torch.int32)
    c = torch.stack([prob.token_inputs(b, L - 1, L)[0][0] for b, L in enumerate(wl.seq_lens)])
    k = torch.stack([prob.token_inputs(b, L - 1, L)[1][0] for b, L in enumerate(wl.seq_lens)])
    st.c_kv.copy_(c)
    st.k_rope.copy_(k)
    st.seq_idx.copy_(torch.arange(wl.B, dtype=torch.int32))
    st.pos.copy_(last)
    st.q_nope.copy_(prob.q_nope)
    st.q_rope.copy_(prob.q_rope)
    st.q_pos.copy_(prob.q_pos)
    st.seq_lens.copy_(prob.seq_lens)
    st.run()
    torch.cuda.synchronize()
    direct = st.out.clone()
    st.capture(2)
    st.out.zero_()
    st.replay()
    torch.cuda.synchronize()
    assert torch.equal(st.out, direct)
    assert ctx.device_status() == 0
    _check_sequences(prob, st.out, st.o_lat, st.lse, range(wl.B), naive_heads=(0,))

    # host memory to host memory: inputs from the pinned host arena, out back to
    # pinned host memory, all inside one graph replay
    host = st.host_inputs()
    for name, v in host.items():
        v.copy_(getattr(st, name))
    for name in ("q_nope", "q_rope"):
        getattr(st, name).zero_()          # the replay must bring them from the host
    st.capture(1, host_io=True)
    st.out_host.zero_()
    st.replay()
    torch.cuda.current_stream().synchronize()
    assert torch.equal(st.out_host, direct.cpu())
