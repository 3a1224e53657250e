"""Host-side choice of the work decomposition (no GPU needed).

fa_fwd runs either row-tile pairs (two 128-row query tiles per CTA item that
share every K/V tile) or key-split items (one query tile whose even and odd
key tiles run side by side). A static cost model of the persistent schedule
picks key-split items when the pairs would leave SMs idle: few row tiles
(the short-sequence case of "NVIDIA闪存注意力实操" section "自动调优") or a
pair whose second row tile is empty.
"""

import pytest

from exact_attention_16_gb300 import api
from exact_attention_16_gb300.workloads import WORKLOADS

SMS = 152


@pytest.fixture(autouse=True)
def _reset_schedule():
    yield
    api.fa_debug_set_schedule(-1)


def choice(w, sms=SMS):
    return api.fa_fwd_schedule(w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.causal, sms)


def test_short_causal_mha_uses_key_split():
    # 1280 x 1536 causal MHA, 16 heads: 80 row-tile pairs for 152 SMs, the
    # longest 12 key tiles; key-split gives 160 items of at most 6 steps
    assert choice(WORKLOADS[1]) == 1


@pytest.mark.parametrize("w", WORKLOADS[2:], ids=lambda w: w.name)
def test_long_causal_gqa_keeps_row_tile_pairs(w):
    # thousands of items: the pairs' shared K/V tiles win
    assert choice(w) == 0


def test_one_row_tile_with_long_keys_uses_key_split():
    # Sq = 128, MHA: each pair's second row tile is empty
    assert api.fa_fwd_schedule(1, 128, 32768, 8, 8, False, SMS) == 1


def test_many_waves_keep_pairs_even_without_causal():
    assert api.fa_fwd_schedule(8, 4096, 4096, 32, 8, False, SMS) == 0


def test_fewer_sms_means_fewer_splits():
    # the same short problem fills a small GPU with pairs already
    w = WORKLOADS[1]
    assert choice(w, sms=8) == 0


def test_override_is_reported():
    assert api.fa_debug_set_schedule(1) == api.FA_OK
    assert choice(WORKLOADS[4]) == 1
    assert api.fa_debug_set_schedule(0) == api.FA_OK
    assert choice(WORKLOADS[1]) == 0
    assert api.fa_debug_set_schedule(-1) == api.FA_OK
    assert choice(WORKLOADS[1]) == 1


@pytest.mark.parametrize("args", [
    (0, 128, 128, 2, 2, 0, SMS), (1, 0, 128, 2, 2, 0, SMS), (1, 128, 0, 2, 2, 0, SMS),
    (1, 128, 128, 3, 2, 0, SMS), (1, 128, 128, 2, 2, 2, SMS), (1, 128, 128, 2, 2, 0, 0),
])
def test_invalid_sizes_rejected(args):
    with pytest.raises(api.FAError):
        api.fa_fwd_schedule(*args)


# (B, Sq, Sk, Hq, Hkv, causal) -> the faster schedule measured on a GB300
# (CUDA-graph timings of both forced schedules, microseconds pairs / split)
MEASURED = [
    ((1, 1280, 1536, 16, 16, 1), 1),   # 22.7 / 14.8
    ((1, 2048, 2048, 8, 8, 1), 1),     # 29.6 / 19.1
    ((1, 4096, 4096, 8, 8, 1), 1),     # 50.5 / 29.6
    ((1, 512, 4096, 32, 8, 1), 1),     # 50.1 / 29.3
    ((1, 128, 32768, 8, 8, 0), 1),     # 367.0 / 199.5
    ((1, 3072, 3072, 16, 16, 1), 1),   # 40.3 / 38.0
    ((1, 16384, 16384, 4, 4, 1), 0),   # 183.4 / 188.7
    ((1, 8192, 8192, 8, 1, 1), 0),     # 94.4 / 96.8
    ((1, 1536, 1536, 16, 16, 0), 0),   # 23.9 / 26.6
    ((4, 512, 512, 32, 32, 0), 0),     # 19.5 / 25.8
    ((1, 4096, 4096, 16, 4, 1), 0),    # 50.7 / 55.7
    ((2, 1024, 1024, 32, 8, 1), 0),    # 20.5 / 27.9
]


@pytest.mark.parametrize("shape,faster", MEASURED, ids=lambda x: str(x))
def test_cost_model_picks_the_measured_faster_schedule(shape, faster):
    assert api.fa_fwd_schedule(*shape, SMS) == faster
