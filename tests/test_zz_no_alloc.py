"""The decode-attention entry point for callers that cannot allocate device
memory (mla_decode_attn_static_scratch): a serving runtime whose pool owns all
device memory, or a host thread that must not call cudaMalloc/cudaFree. Checked
against mla_decode_attn with a caller-provided workspace on the same inputs,
twice in a row with a call on other inputs in between (the library's fixed
scratch keeps the previous call's contents), and checked to change the
device's free memory by nothing.

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
    # other inputs for the call in between: other lengths (other split points,
    # so other partial slots) and other queries
    other_lens = torch.tensor([1 + (37 * b) % 512 for b in range(wl.B)], dtype=torch.int32, device="cuda")
    other_q = torch.flip(q_abs, dims=[0]).contiguous()
    want_o2, want_l2 = ctx.decode_attn(cache, other_q, other_lens, SCALE)
    o_lat = torch.empty_like(want_o)
    lse = torch.empty_like(want_l)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for it in range(2):
        o_lat.fill_(float("nan"))
        lse.fill_(float("nan"))
        ctx.decode_attn_static_scratch(cache, q_abs, prob.seq_lens, SCALE, o_lat, lse)
        torch.cuda.synchronize()
        assert ctx.device_status() == 0
        assert_close(f64(o_lat), f64(want_o), what=f"o_lat static scratch vs workspace, call {it}")
        assert np.max(np.abs(f64(lse) - f64(want_l))) <= 5e-3
        # a call on other inputs leaves other partials in the scratch
        o_lat.fill_(float("nan"))
        lse.fill_(float("nan"))
        ctx.decode_attn_static_scratch(cache, other_q, other_lens, SCALE, o_lat, lse)
        torch.cuda.synchronize()
        assert ctx.device_status() == 0
        assert_close(f64(o_lat), f64(want_o2), what=f"o_lat static scratch vs workspace, other inputs {it}")
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory changed across static-scratch calls: {free0} -> {free1}"


def test_static_scratch_rejects_shapes_above_its_size(mla, ctx):
    # B=128, H=128 needs far more than the fixed scratch: refused before any launch
    assert ctx.workspace_size(128, 128, 1) > ctx.static_scratch_bytes()
    cache = mla.Cache.contiguous(128, 8)
    q = torch.zeros(128, 1, 128, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(128, dtype=torch.int32, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        ctx.decode_attn_static_scratch(cache, q, lens, SCALE)
    assert e.value.code == 2 and "static scratch" in str(e.value)


@pytest.mark.parametrize("H,B,Hq", [(48, 4, 1), (16, 4, 5), (16, 2000, 1)])
def test_static_scratch_rejects_like_workspace_entry_point(mla, ctx, H, B, Hq):
    # shapes mla_decode_attn refuses get the same code and message here
    cache = mla.Cache.contiguous(B, 8)
    q = torch.zeros(B, Hq, H, 576, dtype=torch.bfloat16, device="cuda")
    lens = torch.full((B,), 8, dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.float32, device="cuda")
    with pytest.raises(mla.MLAError) as want:
        ctx.decode_attn(cache, q, lens, SCALE, workspace=ws)
    with pytest.raises(mla.MLAError) as got:
        ctx.decode_attn_static_scratch(cache, q, lens, SCALE)
    assert got.value.code == want.value.code
    assert str(got.value) == str(want.value)
