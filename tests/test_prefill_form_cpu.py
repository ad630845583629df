"""mla_prefill_choose_form, on CPU (host logic, no GPU): which prefill form a
chunk runs in. Checked here: the decisions the work counts force (decode and
short chunks over long prefixes stay absorbed, long chunks and whole prompts
go to the MHA form), one switch-over as the chunk grows, that a form the
library cannot run for the shape is never chosen, and the argument checks."""
import ctypes

import pytest

import mla_absorbed_latent_02_gb300 as mla


@pytest.fixture(scope="module", autouse=True)
def lib():
    from mla_absorbed_latent_02_gb300 import _build
    return mla.load_library(_build.build())


def choose(H, T, lens, **kw):
    return mla.prefill_choose_form(H, T, lens, **kw)


@pytest.mark.parametrize("H", [16, 32, 64, 128])
def test_decode_and_short_chunks_stay_absorbed(H):
    # one new token per sequence: expanding every cached key for one query never pays
    for lens in ([4096] * 64, [26], [131072] * 4, list(range(1, 200))):
        assert choose(H, 1, lens)[0] == "absorbed"
    # a 64-token chunk over 4,096 cached tokens: each key is seen by 64 queries
    assert choose(H, 64, [4096] * 4)[0] == "absorbed"


@pytest.mark.parametrize("H", [16, 128])
def test_long_chunks_and_prompts_take_the_mha_form(H):
    assert choose(H, 1024, [1024])[0] == "mha"          # a whole 1,024-token prompt
    assert choose(H, 1024, [4096] * 4)[0] == "mha"      # 1,024-token chunks over 3,072 cached
    assert choose(H, 512, [8192, 600, 4000])[0] == "mha"


@pytest.mark.parametrize("H,prefix", [(16, 4032), (128, 4032), (16, 0), (128, 0), (64, 20000)])
def test_one_switch_over_as_the_chunk_grows(H, prefix):
    """For a fixed prefix the choice moves from absorbed to MHA once and stays
    (every step of T the absorbed form can run, T a multiple of 4)."""
    seen_mha = False
    for T in range(4, 2049, 4):
        form, (ta, tm) = choose(H, T, [prefix + T] * 2)
        assert ta > 0 and tm > 0
        if seen_mha:
            assert form == "mha", (H, prefix, T)
        seen_mha = form == "mha"
    assert seen_mha


def test_estimates_follow_the_work_counts():
    # the MHA form expands every cached token: its estimate grows with the prefix at a fixed chunk
    small = choose(128, 64, [1024])[1][1]
    big = choose(128, 64, [16384])[1][1]
    assert big > 4 * small
    # the absorbed form's attention grows with the (query, key) pairs: doubling the prefix of a
    # long-prefix chunk nearly doubles it
    a1 = choose(16, 256, [8192] * 4)[1][0]
    a2 = choose(16, 256, [16384] * 4)[1][0]
    assert 1.7 < a2 / a1 < 2.0
    # eight times the heads: nearly eight times both estimates once the MHA form's items
    # (sequence, head, 128-query tile) outnumber the SMs ...
    e16 = choose(16, 256, [4096] * 8)[1]
    e128 = choose(128, 256, [4096] * 8)[1]
    assert 7 < e128[0] / e16[0] < 8 and 7 < e128[1] / e16[1] < 8
    # ... while with fewer items than SMs the MHA attention's longest item sets its part
    one16 = choose(16, 256, [4096])[1][1]
    one128 = choose(128, 256, [4096])[1][1]
    assert one128 / one16 < 4


def test_split_kv_units_bound_the_absorbed_form():
    """At H=64 over 4,096 cached tokens, 64 new tokens make 64 row CTAs (two
    split-KV units share the keys) and 96 make 96 (one unit walks them all):
    the absorbed estimate nearly doubles for 1.5x the rows and the choice flips."""
    e64 = choose(64, 64, [4096])
    e96 = choose(64, 96, [4096])
    assert e64[0] == "absorbed" and e96[0] == "mha"
    assert e96[1][0] / e64[1][0] > 1.6
    # at H=16 with four sequences the same step keeps several units: linear growth
    f64 = choose(16, 64, [4096] * 4)[1][0]
    f96 = choose(16, 96, [4096] * 4)[1][0]
    assert f96 / f64 < 1.5


def test_a_form_that_cannot_run_is_never_chosen():
    # FP8 cache: the MHA form reads bf16 rows only
    assert choose(16, 1024, [4096] * 4, fp8=True)[0] == "absorbed"
    # the MHA form's workspace (expanded K and V of every cached token) above the caller's limit
    n = mla.load_library().mla_prefill_mha_workspace_size(128, 1, 1024, 1024)
    assert choose(128, 1024, [1024], ws_limit=n)[0] == "mha"
    assert choose(128, 1024, [1024], ws_limit=n - 1)[0] == "absorbed"
    # Hq*H = 96 rows is no shape of the absorbed kernels (16, 32, 64, then multiples of 64)
    assert choose(16, 6, [4096])[0] == "mha"
    # neither form: FP8 and a row count the absorbed kernels do not take
    with pytest.raises(mla.MLAError) as e:
        choose(16, 6, [4096], fp8=True)
    assert e.value.code == 2


def test_argument_checks():
    lib = mla.load_library()
    lens = (ctypes.c_int32 * 2)(100, 50)
    form = ctypes.c_int32(-1)
    assert lib.mla_prefill_choose_form(16, 2, 64, lens, 0, 0, ctypes.byref(form), None) == 1   # 50 < T
    assert lib.mla_prefill_choose_form(16, 2, 32, lens, 0, 0, ctypes.byref(form), None) == 0   # est_us optional
    assert form.value in (0, 1)
    assert lib.mla_prefill_choose_form(48, 2, 32, lens, 0, 0, ctypes.byref(form), None) == 2   # H
    assert lib.mla_prefill_choose_form(16, 0, 32, lens, 0, 0, ctypes.byref(form), None) == 1   # B
    assert lib.mla_prefill_choose_form(16, 2, 0, lens, 0, 0, ctypes.byref(form), None) == 1    # T
    assert lib.mla_prefill_choose_form(16, 2, 32, None, 0, 0, ctypes.byref(form), None) == 1
    assert lib.mla_prefill_choose_form(16, 2, 32, lens, 0, 0, None, None) == 1
