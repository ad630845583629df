"""The seeded input generator (shared by the tests, the benchmark and the oracle
checks) against the definitions it states: splitmix64, Box-Muller in float64,
float32 -> bfloat16 round-to-nearest-even, counter-based slicing, and the
workload recipes' shapes."""
import math

import numpy as np
import torch

import mla_synth as S

M64 = (1 << 64) - 1


def test_splitmix64_reference_sequence():
    # splitmix64 seeded with 0 yields 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
    # 0x06C45D188009454F (Steele, Lea and Flood; the reference generator adds the
    # golden gamma to its state before each finalisation)
    g = 0x9E3779B97F4A7C15
    assert S._splitmix64_int(0) == 0xE220A8397B1DCDAF
    assert S._splitmix64_int(g) == 0x6E789E6AA1B965F4
    assert S._splitmix64_int((2 * g) & M64) == 0x06C45D188009454F


def test_splitmix64_tensor_matches_integer_version():
    rng = np.random.default_rng(1)
    vals = [0, 1, M64, 1 << 63, (1 << 63) - 1] + [int(v) for v in rng.integers(0, 2**63, 200, dtype=np.int64)]
    x = torch.tensor([S._s64(v) for v in vals], dtype=torch.int64)
    got = [int(v) & M64 for v in S.splitmix64(x)]
    assert got == [S._splitmix64_int(v) for v in vals]


def test_bf16_rounding_matches_the_library_cast():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000),
                        [0.0, -0.0, 1.0, 3.0e38, -3.0e38, 1e-40, np.inf, -np.inf]]).astype(np.float32)
    # exact ties: float32 values halfway between two bfloat16 values
    ties = (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties])
    t = torch.from_numpy(x)
    got = S.f32_to_bf16_bits_rne(t)
    want = t.to(torch.bfloat16).view(torch.int16)
    assert torch.equal(got, want)
    nan = S.f32_to_bf16_bits_rne(torch.tensor([float("nan")]))
    assert int(nan[0]) & 0xFFFF == 0x7FC0


def test_normal_draw_is_box_muller_of_the_stream():
    # element i of a stream: two words, top 53 bits each, z = sqrt(-2 ln(1-u1)) cos(2 pi u2)
    key = S.stream_key(3, "probe")
    got = S.normal_bf16(3, "probe", (5,), std=0.5).float()
    for i in range(5):
        w1 = S._splitmix64_int((key + 2 * i) & M64)
        w2 = S._splitmix64_int((key + 2 * i + 1) & M64)
        u1 = (w1 >> 11) / 2.0 ** 53
        u2 = (w2 >> 11) / 2.0 ** 53
        z = math.sqrt(-2.0 * math.log1p(-u1)) * math.cos(2.0 * math.pi * u2) * 0.5
        want = torch.tensor([z], dtype=torch.float32).to(torch.bfloat16).float()
        assert float(got[i]) == float(want[0])


def test_counter_based_slices_and_chunks():
    full = S.normal_bf16(0, "slice", (1000,))
    part = S.normal_bf16(0, "slice", (300,), offset=250)
    assert torch.equal(full[250:550], part)
    chunked = S.normal_bf16_chunked(0, "slice", (1000,), chunk=77)
    assert torch.equal(full, chunked)
    assert not torch.equal(full, S.normal_bf16(0, "slice2", (1000,)))
    assert not torch.equal(full, S.normal_bf16(1, "slice", (1000,)))


def test_normal_moments():
    z = S.normal_bf16(0, "moments", (1 << 20,)).double()
    assert abs(float(z.mean())) < 5e-3
    assert abs(float(z.std()) - 1.0) < 5e-3
    w = S.normal_bf16(0, "moments_w", (1 << 20,), std=0.02).double()
    assert abs(float(w.std()) - 0.02) < 2e-4


def test_integer_draws():
    v = S.uniform_ints(0, "ints", 10000, 1, 32768)
    assert min(v) >= 1 and max(v) <= 32768
    assert abs(np.mean(v) - 16384.5) < 400
    p = S.permutation(0, "perm", 4097)
    assert sorted(p) == list(range(4097)) and p != list(range(4097))


def test_workload_recipes():
    c0 = S.make_config(0)
    assert (c0.B, c0.H, c0.Hq, c0.seq_lens, c0.capacity, c0.paged) == (1, 16, 1, [26], 32, False)
    c1 = S.make_config(1)
    assert (c1.B, c1.H, c1.Hq, c1.paged) == (64, 16, 1, False) and set(c1.seq_lens) == {4096}
    assert c1.total_tokens * 1152 == 301_989_888
    for idx, (B, H, Hq) in {2: (32, 128, 1), 3: (128, 128, 1), 4: (4, 128, 2)}.items():
        wl = S.make_config(idx)
        assert (wl.B, wl.H, wl.Hq, wl.paged) == (B, H, Hq, True)
        blocks = [blk for row in wl.block_table for blk in row]
        assert sorted(blocks) == list(range(wl.num_blocks))      # a permutation of the pool
        for b, L in enumerate(wl.seq_lens):
            assert len(wl.block_table[b]) == (L + 63) // 64
    assert set(S.make_config(2).seq_lens) == {8192} and set(S.make_config(4).seq_lens) == {131072}
    lens3 = S.make_config(3).seq_lens
    assert min(lens3) >= 1 and max(lens3) <= 32768
    assert S.query_positions(S.make_config(4))[0] == [131070, 131071]
