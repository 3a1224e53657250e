"""Host-side choice of the decode split count (no GPU needed). By default
fa_fwd_decode cuts the keys into the most ranges that keep every CTA in one
wave on the GPU's SMs (a CTA fills an SM's shared memory); timed on GB300
decode shapes, one full wave beat the split counts around it by 5 to 30 %."""

import pytest

from exact_attention_16_gb300 import api

# (B, Sq, Sk, Hq, Hkv, D) -> splits on 152 SMs; units = B x Hkv x row tiles
# (a row tile holds floor(128 / G) query positions of a KV group)
CASES = [
    ((16, 1, 16384, 32, 4, 128), 2),    # 64 units: two splits fill 128 of 152 SMs
    ((64, 1, 16384, 32, 4, 128), 1),    # 256 units: already more than one wave
    ((4, 1, 65536, 32, 4, 128), 9),     # 16 units x 9 = 144 CTAs
    ((32, 1, 4096, 32, 4, 128), 1),     # 128 units
    ((1, 1, 300, 8, 1, 64), 3),         # 1 unit: 152 wanted, clamped to 3 key tiles
    ((1, 40, 8192, 8, 8, 128), 19),     # prefill chunk: G = 1, 1 row tile per head: 8 units
]


@pytest.mark.parametrize("shape,splits", CASES, ids=lambda x: str(x))
def test_one_full_wave(shape, splits):
    assert api.fa_decode_splits(*shape, 0, 152) == splits


def test_explicit_count_is_kept_up_to_the_key_tiles():
    assert api.fa_decode_splits(16, 1, 16384, 32, 4, 128, 5, 152) == 5
    assert api.fa_decode_splits(1, 1, 300, 8, 1, 64, 9, 152) == 3


def test_fewer_sms_fewer_splits():
    assert api.fa_decode_splits(16, 1, 16384, 32, 4, 128, 0, 64) == 1
    assert api.fa_decode_splits(16, 1, 16384, 32, 4, 128, 0, 300) == 4


@pytest.mark.parametrize("args", [
    (16, 1, 16384, 32, 4, 128, 0, 0), (0, 1, 16384, 32, 4, 128, 0, 152), (16, 1, 0, 32, 4, 128, 0, 152),
    (16, 1, 16384, 30, 4, 128, 0, 152),
])
def test_invalid(args):
    with pytest.raises(api.FAError):
        api.fa_decode_splits(*args)
