"""The product's choice of CTA tiling (t2s_gemm_f32_plan, a host-only query; no GPU needed).

The plan is pinned to the winners of the measured sweep on a 152-SM GB300 (bit-exact product,
L2 flushed, TFLOP/s of each forced configuration), and the query's argument checks are tested.
"""
from __future__ import annotations

import pytest

from roofline_driven_tiling_gb300 import binding

(BIG, BIG_SHORT_K, TALL88, SMALL48, HUGE, HUGE_TAIL, BIG88, TALL84, PERSISTENT, WIDE74, TINY24,
 PERSISTENT_STORE) = range(12)


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


# (M, N, K) -> the configuration measured fastest (or within 1 % of it) on GB300: each
# configuration forced in turn, L2 flushed, best of the timed calls in TFLOP/s, with the
# current kernels (64-deep K blocks where a launch covers all of K; the 56 x 128 and 64 x 64
# tiles in 2 stages where their CTAs share SMs). 256^3, 384^3, 5120^3 and 8192^3 were measured
# with 32-deep K blocks throughout.
MEASURED = {
    (256, 256, 256): TINY24,          # 3.1; 64 x 64 tiles 2.6
    (384, 384, 384): TINY24,          # 8.8; 64 x 64 tiles 6.7
    (512, 512, 512): TINY24,          # 15.7; 64 x 64 tiles 14.1
    (512, 512, 2048): TINY24,         # 21.6; 64 x 64 tiles 19.2
    (640, 640, 640): SMALL48,         # 22.6; 32 x 32 tiles 19.2
    (768, 768, 768): SMALL48,         # 36.0; 56 x 128 tiles 25.6
    (1024, 1024, 512): WIDE74,        # 42.6; 128 x 64 tiles of 8 warps 39.4
    (1024, 1024, 1024): WIDE74,       # 49.2; 128 x 64 tiles of 8 warps 45.0
    (1024, 1024, 4096): WIDE74,       # 55.0; 128 x 64 tiles of 8 warps 49.8
    (1000, 1003, 997): WIDE74,        # 38.6; 128 x 64 tiles of 8 warps 37.1
    (1152, 1152, 1152): SMALL48,      # 38.0; 56 x 128 tiles 34.5
    (1280, 1280, 1280): SMALL48,      # 47.3; 56 x 128 tiles 43.2
    (1408, 1408, 256): WIDE74,        # 40.4; 128 x 128 tiles of 8 warps 37.4
    (1408, 1408, 512): WIDE74,        # 46.5; 128 x 128 tiles of 8 warps 44.3
    (1408, 1408, 1408): WIDE74,       # 52.2; 128 x 128 tiles of 8 warps 48.4
    (1536, 1536, 1536): BIG88,        # 56.8-57.7; 128 x 64 tiles of 8 warps 55.1
    (1792, 1792, 1792): WIDE74,       # 58.4; 128 x 64 tiles of 8 warps 51.0
    (2048, 1024, 2048): WIDE74,       # 55.7; 128 x 64 tiles of 8 warps 49.8
    (1024, 3584, 1024): TALL88,       # 56.2; 128 x 64 tiles of 8 warps 56.2
    (896, 5760, 256): WIDE74,         # 49.0; 256 x 128 with the tail 42.6
    (2048, 2048, 2048): WIDE74,       # 58.1; 256 x 128 tiles 56.2
    (2048, 4096, 1024): HUGE_TAIL,    # 58.7; 128 x 64 tiles and 56 x 128 tiles 58.1
    (2304, 2304, 2304): HUGE_TAIL,    # 60.4; 56 x 128 tiles 59.3
    (2560, 1920, 512): HUGE,          # 61.0; 56 x 128 tiles 50.9
    (2560, 2560, 2560): HUGE_TAIL,    # 61.1; 128 x 128 tiles 56.6
    (3000, 2000, 1000): HUGE_TAIL,    # 52.9-58.1; 56 x 128 tiles 53.6
    (3072, 3072, 3072): HUGE,         # 64.3; 128 x 128 61.6, with the tail 59.4
    (3584, 3584, 3584): HUGE_TAIL,    # 63.6; 256 x 128 alone 58.7
    (4096, 1024, 4096): WIDE74,       # 59.0; 256 x 128 tiles 56.8
    (4096, 4096, 4096): HUGE_TAIL,    # 66.4; 128 x 128 63.5
    (5120, 5120, 5120): HUGE_TAIL,    # 64.8; 128 x 128 63.6
    (6144, 6144, 6144): HUGE_TAIL,    # 66.5; 128 x 128 63.7
    (8192, 512, 1024): WIDE74,        # 56.5; 256 x 128 tiles 55.0
    (8192, 8192, 8192): HUGE_TAIL,    # 66.3; 128 x 128 66.5
}


@pytest.mark.parametrize("shape", sorted(MEASURED), ids=lambda s: "x".join(map(str, s)))
def test_plan_matches_measured_winner(shape):
    assert binding.t2s_gemm_f32_plan(*shape, 152) == MEASURED[shape]


def test_plan_short_k_and_copies():
    # K < 256 keeps to tiles of at most 128 x 128 with the compact k loop.
    assert binding.t2s_gemm_f32_plan(3072, 3072, 128, 152) == BIG_SHORT_K
    assert binding.t2s_gemm_f32_plan(8192, 8192, 128, 152) == BIG_SHORT_K
    # At most three K blocks and two rounds of 256 x 128 tiles or more: the persistent grid
    # with TMA stores of C (16384^2 x 32: 51.1 against 47.6 TFLOP/s; 8192^2 x 64: 54.2
    # against 53.6).
    assert binding.t2s_gemm_f32_plan(16384, 16384, 32, 152) == PERSISTENT_STORE
    assert binding.t2s_gemm_f32_plan(8192, 8192, 64, 152) == PERSISTENT_STORE
    assert binding.t2s_gemm_f32_plan(6144, 6144, 96, 152) == PERSISTENT_STORE
    assert binding.t2s_gemm_f32_plan(8192, 8192, 97, 152) == BIG_SHORT_K
    # One K block but fewer than two rounds of 256 x 128 tiles: the persistent grid of 128 x 128
    # tiles (400 of them, 200 of 256 x 128).
    assert binding.t2s_gemm_f32_plan(2560, 2560, 32, 152) == PERSISTENT
    assert binding.t2s_gemm_f32_plan(2560, 2560, 33, 152) == BIG_SHORT_K
    # One tile row of 128: the 256-row tile would be half empty.
    assert binding.t2s_gemm_f32_plan(128, 131072, 288, 152) == BIG


def test_plan_tail_only_with_a_whole_round():
    # Fewer 256 x 128 tiles than SMs: no whole round, so no split launch.
    assert binding.t2s_gemm_f32_plan(2560, 1920, 512, 152) == HUGE  # 150 tiles
    # A whole number of rounds: nothing left for a tail.
    assert binding.t2s_gemm_f32_plan(256 * 19, 128 * 16, 1024, 152) != HUGE_TAIL  # 304 tiles
    assert binding.t2s_gemm_f32_plan(2500, 2000, 512, 152) == HUGE_TAIL  # 160 = 152 + 8


def test_plan_eight_warp_tiles():
    # 152 tiles of 56 x 128 on 152 SMs: one each, 8 warps (128 x 64 tiles: 128, less even).
    assert binding.t2s_gemm_f32_plan(1024, 1024, 512, 152) == WIDE74
    # 1152 rows are 21 tiles of 56: 168 > 152; 9 x 16 = 144 tiles of 128 x 64 fit.
    assert binding.t2s_gemm_f32_plan(1152, 1024, 512, 152) == TALL84
    # 162 tiles of 128 x 64 would need a second round on some SMs: not the 8-warp tile.
    assert binding.t2s_gemm_f32_plan(1152, 1152, 1152, 152) != TALL84
    # The 56 x 128 tile (64-deep K blocks over all of K, two CTAs per SM) also at two or more
    # per SM from K = 128 on: 286 tiles at 1408^3, 448 at 1792^3 and 1792^2 x 512, 592 at
    # 2048^2 x 128 (level with 64 x 64 tiles: 39.5 against 39.4); not below K = 128.
    assert binding.t2s_gemm_f32_plan(1408, 1408, 1408, 152) == WIDE74
    assert binding.t2s_gemm_f32_plan(1792, 1792, 512, 152) == WIDE74
    assert binding.t2s_gemm_f32_plan(2048, 2048, 128, 152) == WIDE74
    assert binding.t2s_gemm_f32_plan(1408, 1408, 127, 152) == BIG88
    # 121 tiles of 128 x 128 on a GPU of 128 SMs, where 286 tiles of 56 x 128 take 3 rounds.
    assert binding.t2s_gemm_f32_plan(1408, 1408, 1408, 128) == BIG88


def test_plan_depends_on_sm_count():
    # The same 4096^3 product on a GPU with 128 SMs: 512 tiles are exactly 4 rounds.
    assert binding.t2s_gemm_f32_plan(4096, 4096, 4096, 128) == HUGE


# (M, N, K) -> chunk count of the automatic split-K choice (t2s_gemm_f32_splitk_plan), with
# the measured TFLOP/s of that count and of the best alternative (GB300, L2 flushed, mean of
# 30 calls; 1 is the product alone).
SPLITK_MEASURED = {
    (512, 512, 512): 4,        # 15.2; 5 chunks 15.6, the product 14.1
    (768, 768, 768): 1,        # 32.6; 4 chunks 32.6, 6 chunks 31.4
    (1024, 1024, 1024): 1,     # 44.3; 8 chunks 41.2
    (1000, 1003, 997): 1,      # 26.1; 2 chunks 26.1, 8 chunks 24.6
    (1280, 1280, 1280): 6,     # 48.4; 3 chunks 48.4, the product 44.9
    (1536, 1536, 1536): 1,     # 55.5; 5 chunks 53.1
    (1792, 1792, 1792): 1,     # the product 58.4 (56 x 128 tiles); 3 chunks 56.6, 6 chunks 55.4
    (2048, 2048, 2048): 4,     # 57.9; 2 chunks 56.4, the product 55.4
    (1024, 1024, 4096): 7,     # 55.5; 8 chunks 53.9, the product 50.2
    (512, 512, 4096): 9,       # 43.1; 8 chunks 40.7, the product 18.0 (64 x 64 tiles)
    (256, 256, 8192): 9,       # 28.6; 16 chunks 30.3, the product 4.6 (64 x 64 tiles)
    (4096, 4096, 4096): 1,
}


@pytest.mark.parametrize("shape", sorted(SPLITK_MEASURED), ids=lambda s: "x".join(map(str, s)))
def test_splitk_plan_matches_measured(shape):
    assert binding.t2s_gemm_f32_splitk_plan(*shape, 152) == SPLITK_MEASURED[shape]


def test_splitk_plan_limits():
    # Chunks of at least 128 values: K = 383 allows two chunks, K = 384 three.
    assert binding.t2s_gemm_f32_splitk_plan(64, 64, 383, 152) == 2
    assert binding.t2s_gemm_f32_splitk_plan(64, 64, 384, 152) == 3
    # A split pays for the plane sum's launch: at 256^3 the product alone is faster (3.4
    # TFLOP/s with 32 x 32 tiles against 2.6 in two chunks).
    assert binding.t2s_gemm_f32_splitk_plan(256, 256, 256, 152) == 1
    # At most 16 chunks, however long K is.
    assert binding.t2s_gemm_f32_splitk_plan(64, 64, 1 << 20, 152) == 16
    # Empty problems make no split.
    assert binding.t2s_gemm_f32_splitk_plan(0, 128, 4096, 152) == 1
    assert binding.t2s_gemm_f32_splitk_plan(128, 128, 0, 152) == 1
    for args in [(-1, 4, 4, 152), (4, 4, 4, 0), ((1 << 30) + 1, 4, 4, 152)]:
        assert binding.t2s_gemm_f32_splitk_plan(*args) == -1


@pytest.mark.parametrize("args", [(-1, 4, 4, 152), (4, -1, 4, 152), (4, 4, -1, 152),
                                  ((1 << 30) + 1, 4, 4, 152), (4, 4, 4, 0), (4, 4, 4, -3)])
def test_plan_rejects_bad_arguments(args):
    assert binding.t2s_gemm_f32_plan(*args) == -1


def test_plan_names():
    assert binding.plan(4096, 4096, 4096, 152) == "256x128 tiles in whole rounds, the rest as 64x64 tiles"
    assert binding.plan(1024, 1024, 1024, 152) == "56x128 tiles of 8 warps"
    assert binding.plan(1152, 1024, 512, 152) == "128x64 tiles of 8 warps"
    assert binding.plan(384, 384, 384, 152) == "32x32 tiles"
    assert binding.plan(16384, 16384, 32, 152) == "256x128 tiles on a persistent grid with TMA stores of C"
    assert set(binding.PLAN_NAMES) == set(range(12))
    with pytest.raises(ValueError):
        binding.plan(-1, 4, 4, 152)


def test_plan_properties_on_random_shapes():
    """Invariants of the tiling choice on seeded random shapes: the 128 x 128 and 128 x 64
    tilings of 8 warps only when their tiles fit the SMs once, the tail split only with at least one whole round
    of 256 x 128 tiles and K >= 256, and a split-K count that keeps chunks of 128 values."""
    import numpy as np

    rng = np.random.default_rng(20261202)
    one_round = {BIG88: (128, 128), TALL84: (128, 64)}
    for _ in range(2000):
        M, N = (int(x) for x in rng.integers(1, 9000, size=2))
        K = int(rng.integers(1, 20000))
        sms = int(rng.choice([108, 132, 148, 152]))
        code = binding.t2s_gemm_f32_plan(M, N, K, sms)
        assert code in binding.PLAN_NAMES
        if code in one_round:
            bm, bn = one_round[code]
            assert -(-M // bm) * -(-N // bn) <= sms
        if code == HUGE_TAIL:
            assert K >= 256 and -(-M // 256) * -(-N // 128) > sms
        if code == PERSISTENT:
            assert K <= 32
        s = binding.t2s_gemm_f32_splitk_plan(M, N, K, sms)
        assert 1 <= s <= 16
        assert s == 1 or K // s >= 128
