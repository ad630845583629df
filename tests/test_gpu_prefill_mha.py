"""Prefill in the expanded (MHA) form, mla_prefill_mha, through the C ABI:
against the float64 naive oracle (the definition the form computes), against
the absorbed GPU path on the same inputs, and its device-side checks.

Every cache slot and the whole workspace start as NaN, so rows past a
sequence's end (or workspace bytes the call does not write) that leaked into a
result would show."""
import numpy as np
import pytest
import torch

import mla_synth as S
from mla_testlib import Problem, SCALE, assert_close, f64, fill_cache, gpu_step, make_cache, oracle_naive

pytestmark = pytest.mark.gpu


def _workload(name, H, T, lens, paged, seed):
    if paged:
        tbl, nb, mb = S._paged_tables(seed, name, lens)
        return S.Workload(name, len(lens), H, T, lens, True, block_table=tbl, num_blocks=nb, max_blocks=mb,
                          seed=seed)
    return S.Workload(name, len(lens), H, T, lens, False, capacity=max(lens) + 5, seed=seed)


def _poisoned_cache(mla, ctx, prob):
    cache = make_cache(mla, prob.wl)
    cache.storage.view(torch.int16).fill_(0x7FC0)
    fill_cache(ctx, cache, prob)
    return cache


def _mha(ctx, cache, prob, max_len=None, poison=True):
    wl = prob.wl
    max_len = max(wl.seq_lens) if max_len is None else max_len
    n = ctx.prefill_mha_workspace_size(wl.H, wl.B, wl.Hq, max_len)
    ws = torch.full(((n + 15) // 16, 16), 0xFF if poison else 0, dtype=torch.uint8, device="cuda")
    out = ctx.prefill_mha(cache, prob.w_uk, prob.w_uv, prob.q_nope, prob.q_rope, prob.q_pos, prob.seq_lens,
                          max_len, SCALE, workspace=ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("H,T,lens,paged,heads", [
    (16, 130, [130, 300], False, None),        # two query tiles, the second of 2 rows; a prefix of 170
    (16, 64, [64, 200, 129], True, None),      # one ragged tile per sequence, three sequences
    (32, 257, [300], True, None),              # three query tiles, keys end mid-tile
    (128, 96, [96, 333], True, [0, 77, 127]),  # V3 head count, sampled heads
    (64, 200, [1000], False, [5, 63]),         # a long cached prefix: eight key tiles
])
def test_prefill_mha_vs_naive_oracle(mla, ctx, H, T, lens, paged, heads):
    wl = _workload(f"mha_h{H}_t{T}", H, T, lens, paged, seed=11)
    prob = Problem(wl)
    cache = _poisoned_cache(mla, ctx, prob)
    out = _mha(ctx, cache, prob)
    assert ctx.device_status() == 0
    got = f64(out)
    hs = list(range(H)) if heads is None else heads
    for b in range(wl.B):
        want = oracle_naive(prob, b, hs)
        assert np.all(np.isfinite(got[b]))
        assert_close(got[b][:, hs], want, what=f"mha prefill b={b}")


def test_prefill_mha_matches_absorbed_path(mla, ctx):
    """The two forms of the same chunk (H=16, 300 new tokens after 212 cached
    ones) agree within the bars each meets against the oracle."""
    wl = _workload("mha_vs_abs", 16, 300, [512, 300], True, seed=12)
    prob = Problem(wl)
    cache = _poisoned_cache(mla, ctx, prob)
    out = _mha(ctx, cache, prob)
    ref, _, _ = gpu_step(ctx, cache, prob)   # append of the same rows again, then the absorbed step
    assert ctx.device_status() == 0
    assert_close(f64(out), f64(ref), what="mha vs absorbed")


def test_prefill_mha_long_prompt_h128(mla, ctx):
    """A 1,024-token prompt at H=128 from an empty paged cache in one call,
    against the one-shot causal forward of the naive oracle on every head
    (each head separately: a wrong tile of one head must not hide in the
    others' error)."""
    import oracle as O
    L = 1024
    wl = _workload("mha_prompt", 128, L, [L], True, seed=8)
    prob = Problem(wl)
    cache = _poisoned_cache(mla, ctx, prob)
    out = _mha(ctx, cache, prob)
    assert ctx.device_status() == 0
    c, k = prob.token_inputs(0)
    h = prob.host
    want = O.naive_prefill_causal(f64(c), f64(k), h["q_nope"][0], h["q_rope"][0], h["w_uk"], h["w_uv"], SCALE)
    got = f64(out)[0]
    for hd in range(128):
        assert_close(got[:, hd], want[:, hd], what=f"1k-token prompt, MHA form, head {hd}")


@pytest.mark.parametrize("H,T,lens", [(128, 1024, [1024]), (16, 1024, [4096, 3000])])
def test_prefill_mha_repeats_bit_identical(mla, ctx, H, T, lens):
    """The kernels add nothing with atomics and in no order that depends on
    timing: calls on the same inputs give the same bytes (a race between the
    pipeline's roles would show here first)."""
    wl = _workload(f"mha_det_h{H}", H, T, lens, True, seed=16)
    prob = Problem(wl, keep_host=False)
    cache = make_cache(mla, wl)
    fill_cache(ctx, cache, prob)
    outs = [_mha(ctx, cache, prob, poison=False).view(torch.int16).clone() for _ in range(3)]
    assert ctx.device_status() == 0
    for i in (1, 2):
        assert torch.equal(outs[0], outs[i]), f"call {i} differs from call 0"


def test_prefill_mha_repeat_reuses_workspace(mla, ctx):
    """Two calls back to back on one stream with one workspace (the second
    overwrites what the first's attention reads) give identical bytes."""
    wl = _workload("mha_rep", 16, 192, [192, 400], True, seed=13)
    prob = Problem(wl)
    cache = _poisoned_cache(mla, ctx, prob)
    n = ctx.prefill_mha_workspace_size(16, 2, 192, 400)
    ws = torch.empty(((n + 15) // 16, 16), dtype=torch.uint8, device="cuda")
    a = ctx.prefill_mha(cache, prob.w_uk, prob.w_uv, prob.q_nope, prob.q_rope, prob.q_pos, prob.seq_lens, 400,
                        SCALE, workspace=ws)
    b = ctx.prefill_mha(cache, prob.w_uk, prob.w_uv, prob.q_nope, prob.q_rope, prob.q_pos, prob.seq_lens, 400,
                        SCALE, workspace=ws)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_prefill_mha_length_out_of_range_flagged(mla, ctx):
    """A sequence shorter than the chunk, or longer than max_len, sets
    MLA_DEVICE_LENGTH; the other sequence's rows are still exact."""
    wl = _workload("mha_len", 16, 128, [128, 300], False, seed=14)
    prob = Problem(wl)
    cache = _poisoned_cache(mla, ctx, prob)
    good = _mha(ctx, cache, prob)
    assert ctx.device_status() == 0
    # sequence 1 longer than max_len: flagged and skipped, sequence 0 unchanged
    bad = _mha(ctx, cache, prob, max_len=200)
    assert ctx.device_status() & mla.DEVICE_LENGTH
    assert torch.equal(bad[0].view(torch.int16), good[0].view(torch.int16))
    # sequence 0 shorter than the chunk
    prob.seq_lens[0] = 100
    _mha(ctx, cache, prob)
    assert ctx.device_status() & mla.DEVICE_LENGTH


def test_prefill_mha_rejects_bad_arguments(mla, ctx):
    wl = _workload("mha_args", 16, 64, [64], False, seed=15)
    prob = Problem(wl)
    cache = make_cache(mla, wl)
    n = ctx.prefill_mha_workspace_size(16, 1, 64, 64)
    small = torch.empty(n // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(RuntimeError, match="workspace too small"):
        ctx.prefill_mha(cache, prob.w_uk, prob.w_uv, prob.q_nope, prob.q_rope, prob.q_pos, prob.seq_lens, 64,
                        SCALE, workspace=small)
    with pytest.raises(RuntimeError, match="max_len"):
        ctx.prefill_mha(cache, prob.w_uk, prob.w_uv, prob.q_nope, prob.q_rope, prob.q_pos, prob.seq_lens, 32,
                        SCALE)
    fp8 = make_cache(mla, wl, fp8=True)
    with pytest.raises(ValueError):
        ctx.prefill_mha(fp8, prob.w_uk, prob.w_uv, prob.q_nope, prob.q_rope, prob.q_pos, prob.seq_lens, 64, SCALE)
