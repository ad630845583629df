"""The decode-attention entry point for callers that cannot allocate device
memory (mla_decode_attn_static_scratch), checked against mla_decode_attn with a
caller-provided workspace on the same inputs, twice in a row (the library's
fixed scratch keeps the previous call's contents).

Kept in a file of its own, collected last, so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import mla_synth as S
from mla_testlib import Problem, SCALE, assert_close, f64, fill_cache, make_cache

pytestmark = pytest.mark.gpu


def test_static_scratch_matches_workspace_entry_point(mla, ctx):
    # B=64, H=16, L=512: 256 tiles over the SMs, so sequences are split across
    # units and the partials pass through the scratch.
    wl = S.make_config(1, scale_down=8)
    prob = Problem(wl)
    cache = make_cache(mla, wl)
    fill_cache(ctx, cache, prob)
    q_abs = ctx.absorb_q(prob.w_uk, prob.q_nope, prob.q_rope, prob.q_pos)
    need = ctx.workspace_size(wl.H, wl.B, wl.Hq)
    assert 0 < need <= ctx.static_scratch_bytes()
    want_o, want_l = ctx.decode_attn(cache, q_abs, prob.seq_lens, SCALE)
    torch.cuda.synchronize()
    for _ in range(2):
        o_lat = torch.full_like(want_o, float("nan"))
        lse = torch.full_like(want_l, float("nan"))
        ctx.decode_attn_static_scratch(cache, q_abs, prob.seq_lens, SCALE, o_lat, lse)
        torch.cuda.synchronize()
        assert ctx.device_status() == 0
        assert_close(f64(o_lat), f64(want_o), what="o_lat static scratch vs workspace")
        assert np.max(np.abs(f64(lse) - f64(want_l))) <= 5e-3


def test_static_scratch_rejects_shapes_above_its_size(mla, ctx):
    # B=128, H=128 needs far more than the fixed scratch: refused before any launch
    assert ctx.workspace_size(128, 128, 1) > ctx.static_scratch_bytes()
    cache = mla.Cache.contiguous(128, 8)
    q = torch.zeros(128, 1, 128, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(128, dtype=torch.int32, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        ctx.decode_attn_static_scratch(cache, q, lens, SCALE)
    assert e.value.code == 2 and "static scratch" in str(e.value)
