"""The dispatch plan of sgemm_3xtf32 on the host (no GPU): which kernel form
runs, the k-slice width, the stages and the persistent schedule. The pair
form falls back to single CTAs when the device keeps no CTA pairs resident or
when every tile would be split along K; the two-SM form always takes 32-wide
slices (three stages of half B tiles), single CTAs 16 from K = 1024 up and 32
below; N <= 64 takes 64-wide tiles and N <= 128 (or little 256-wide work)
128-wide tiles, on single CTAs with 32-wide slices. The
GB300 figures (152 SMs, 76 resident pairs) are the ones the GPU runs report in
sgemm_last_config()."""
import numpy as np
import pytest

from dense_fp32_gemm_gb300 import binding

SMS, PAIRS = 152, 76
PAIR, SINGLE = binding.SGEMM_X3_PAIR, binding.SGEMM_X3_SINGLE


def plan(M, N, K, form, pairs=PAIRS, sms=SMS):
    st, p = binding.sgemm_3xtf32_plan(M, N, K, form, pairs, sms)
    assert st == binding.SGEMM_OK
    return p


def test_square4096_in_each_form():
    # 32 x 16 tiles of 128 x 256: 256 tile pairs on 76 clusters, 3.37 waves:
    # three waves whole, the last (a 0.37 wave, at least a quarter) split along K
    p = plan(4096, 4096, 4096, PAIR)
    assert (p["form"], p["bk"], p["stages"], p["ctas"], p["units"], p["bn"]) == (PAIR, 32, 3, 152, 76, 256)
    assert (p["dp_units"], p["split_units"], p["kiters"]) == (228, 28, 128)
    p = plan(4096, 4096, 4096, SINGLE)
    assert (p["form"], p["bk"], p["stages"], p["ctas"], p["units"]) == (SINGLE, 16, 4, 152, 152)
    assert (p["dp_units"], p["split_units"]) == (304, 208)


@pytest.mark.parametrize("form", [PAIR, SINGLE])
def test_pairs_fall_back_when_every_tile_is_split(form):
    # 2048^3: 32 tile pairs on 76 clusters, all split along K
    p = plan(2048, 2048, 2048, form)
    assert (p["form"], p["bk"], p["stages"], p["ctas"]) == (SINGLE, 16, 4, 152)
    assert p["dp_units"] == 0


def test_pairs_fall_back_without_resident_pairs():
    p = plan(4096, 4096, 4096, PAIR, pairs=0)
    assert p["form"] == SINGLE and p["ctas"] == SMS


@pytest.mark.parametrize("K, bk, stages", [(1023, 32, 2), (1024, 16, 4), (777, 32, 2), (16384, 16, 4)])
def test_single_cta_slice_width_follows_k(K, bk, stages):
    p = plan(4200, 2600, K, SINGLE)      # 33 x 11 wide tiles, over 48 slices of 32 per CTA
    assert (p["bn"], p["bk"], p["stages"], p["kiters"]) == (256, bk, stages, (K + bk - 1) // bk)


def test_two_sm_form_keeps_32_wide_slices_at_any_k():
    # 304 wide tiles: two waves of them, so 256-wide tiles at any K
    for K in (64, 1023, 1024, 8192):
        p = plan(128 * 2 * 76 * 2, 256, K, PAIR)
        assert (p["form"], p["bk"], p["stages"]) == (PAIR, 32, 3), K


def test_schedule_covers_every_tile():
    # whole-tile units plus the tiles behind the K-split units cover the grid of tiles
    for (M, N, K, form) in [(4096, 4096, 4096, PAIR), (8192, 8192, 8192, PAIR), (8191, 1000, 777, SINGLE),
                            (16384, 64, 4096, SINGLE), (1000, 1300, 2056, PAIR)]:
        p = plan(M, N, K, form)
        tiles_m, tiles_n = -(-M // 128), -(-N // p["bn"])
        units = tiles_n * (-(-tiles_m // 2) if p["form"] != SINGLE else tiles_m)
        assert p["dp_units"] + p["split_units"] == units, (M, N, K, form)
        assert p["ctas"] == p["units"] * (1 if p["form"] == SINGLE else 2)


def test_argument_errors():
    assert binding.sgemm_3xtf32_plan(0, 4, 4, PAIR, PAIRS, SMS)[0] == binding.SGEMM_ERR_INVALID_DIM
    assert binding.sgemm_3xtf32_plan(4, 4, 0, PAIR, PAIRS, SMS)[0] == binding.SGEMM_ERR_INVALID_DIM
    assert binding.sgemm_3xtf32_plan(4, 4, 4, 0, PAIRS, SMS)[0] == binding.SGEMM_ERR_INVALID_VALUE
    # 3 named a form that shared B tiles between the CTAs of a pair by TMA
    # multicast; it is no longer built and is rejected like any unknown form
    for form in (3, 4):
        assert binding.sgemm_3xtf32_plan(4, 4, 4, form, PAIRS, SMS)[0] == binding.SGEMM_ERR_INVALID_VALUE
    assert binding.sgemm_3xtf32_plan(4, 4, 4, PAIR, -1, SMS)[0] == binding.SGEMM_ERR_INVALID_VALUE
    assert binding.sgemm_3xtf32_plan(4, 4, 4, PAIR, PAIRS, 0)[0] == binding.SGEMM_ERR_INVALID_VALUE


@pytest.mark.parametrize("form", [PAIR, SINGLE])
@pytest.mark.parametrize("N", [1, 33, 64])
def test_narrow_tiles_for_n_up_to_64(N, form):
    # 16384 x N x 4096: 128 tiles of 128 x 64 (not 128 x 256) on single CTAs,
    # 32-wide slices at any K; A's two parts in tensor memory, so a stage
    # holds A's raw tile and B's two parts (32 KB), six of them
    for K in (777, 4096):
        p = plan(16384, N, K, form)
        assert (p["form"], p["bn"], p["bk"], p["stages"]) == (SINGLE, 64, 32, 6), K
        assert p["dp_units"] + p["split_units"] == 128


def test_128_wide_tiles_up_to_n_128():
    # 65 <= N <= 128: 128-wide tiles (a 256-wide tile would compute at least
    # half its columns beyond N); A's parts in tensor memory, four 48 KB stages
    for N in (65, 96, 128):
        p = plan(16384, N, 4096, PAIR)
        assert (p["form"], p["bn"], p["bk"], p["stages"]) == (SINGLE, 128, 32, 4), N


@pytest.mark.parametrize("M, N, K", [(1024, 1024, 1024), (1536, 768, 1024), (6144, 256, 512),
                                     (512, 512, 8192), (1024, 1024, 2048), (1024, 1024, 4096),
                                     (2048, 1024, 1024), (8191, 1000, 777), (6272, 256, 512)])
def test_128_wide_tiles_for_little_wide_work(M, N, K):
    # the 256-wide work is at most 48 slices of 32 per CTA (wide tiles x
    # ceil(K / 32) <= 48 x 152), and the 128-wide tiles are not few
    p = plan(M, N, K, PAIR)
    assert (p["form"], p["bn"], p["bk"], p["stages"]) == (SINGLE, 128, 32, 4)


@pytest.mark.parametrize("M, N, K", [(512, 512, 512), (300, 520, 4096), (256, 256, 256),
                                     (200, 300, 1024), (1024, 1024, 32), (128, 128, 128)])
def test_64_wide_tiles_when_128_wide_tiles_are_few(M, N, K):
    # (sms / tiles)^2 > ceil(K / 32) / 2 with 128-wide tiles: each would be
    # split along K over so many CTAs that adding up their partial tiles
    # outweighs the main loop
    p = plan(M, N, K, PAIR)
    assert (p["form"], p["bn"], p["bk"], p["stages"]) == (SINGLE, 64, 32, 6)
    tiles = -(-M // 128) * -(-N // 128)
    assert 2 * SMS * SMS > -(-K // 32) * tiles * tiles


@pytest.mark.parametrize("M, N, K", [(2048, 2048, 2048), (1024, 1024, 16384), (16384, 129, 4096),
                                     (16384, 4096, 4096), (3072, 2048, 1536)])
def test_256_wide_tiles_past_48_slices_per_cta(M, N, K):
    # more than 48 slices of 32 of 256-wide work per CTA
    assert -(-M // 128) * -(-N // 256) * -(-K // 32) > 48 * SMS
    assert plan(M, N, K, SINGLE)["bn"] == 256


@pytest.mark.parametrize("M, N, K", [(128 * 2 * 76 * 2, 256, 64), (128 * 2 * 76, 512, 32),
                                     (4096, 4096, 32)])
def test_256_wide_tiles_from_two_waves_of_them(M, N, K):
    # at least 2 x 152 wide tiles, however short K
    assert -(-M // 128) * -(-N // 256) >= 2 * SMS
    assert plan(M, N, K, SINGLE)["bn"] == 256


def test_tile_width_rule_has_no_overflow_at_the_largest_sizes():
    big = 2 ** 31 - 1
    for (M, N, K) in [(big, 64, 64), (65536, big // 4, 32), (64, 64, big)]:
        st, p = binding.sgemm_3xtf32_plan(M, N, K, PAIR, PAIRS, SMS)
        assert st == 0 and p["bn"] in (64, 128, 256), (M, N, K)


def test_pair_form_splits_the_last_two_waves_when_the_last_is_thin():
    # 6144 x 4096: 384 tile pairs, 5.05 waves on 76 clusters: the last 0.05 of a
    # wave is too thin to split alone, so the last two waves are split
    p = plan(6144, 4096, 4096, PAIR)
    assert p["form"] == PAIR and p["dp_units"] == 4 * 76 and p["split_units"] == 384 - 4 * 76
    # 8192^3: 1024 pairs, 13.47 waves: only the last wave is split
    p = plan(8192, 8192, 8192, PAIR)
    assert p["dp_units"] == 13 * 76 and p["split_units"] == 1024 - 13 * 76


def test_below_two_waves_of_pairs_single_ctas_run():
    # 3072 x 2048: 96 tile pairs, 1.26 waves on 76 clusters: the two-wave split
    # leaves no whole tiles, so single CTAs run (faster than pairs with a
    # one-wave split)
    p = plan(3072, 2048, 1536, PAIR)
    assert (p["form"], p["dp_units"]) == (SINGLE, 0)


def test_narrow_tiles_fit_tensor_memory_and_shared_memory():
    # narrow tiles: two accumulators of the tile's width plus a 64-column A
    # slot (32 raw + 32 residual TF32 columns) per stage within the 512 TMEM
    # columns; stages of A's raw tile and B's two parts within the 192 KB ring
    rng = np.random.default_rng(5)
    seen = set()
    for _ in range(2000):
        M, N, K = (int(x) for x in rng.integers(1, 20000, 3))
        p = plan(M, N, K, PAIR)
        seen.add(p["bn"])
        if p["bn"] == 256:
            continue
        assert (p["form"], p["bk"]) == (SINGLE, 32), (M, N, K)
        assert 2 * p["bn"] + 64 * p["stages"] <= 512, (M, N, K, p)
        stage_bytes = 128 * 32 * 4 + 2 * p["bn"] * 32 * 4
        assert p["stages"] * stage_bytes <= 192 * 1024 and p["stages"] >= 3, (M, N, K, p)
    assert seen == {64, 128, 256}
