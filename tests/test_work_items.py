"""The persistent kernel's work decomposition, on the CPU: the items fa_fwd
runs (from the same item-numbering and scheduling functions the kernel
executes, through the host-only fa_fwd_work_items query) checked against
the definitions they implement.

* Every (batch, query head, 128-row tile) with a row below Sq is computed
  exactly once, under both decompositions.
* Query head h reads key/value head h // (Hq / Hkv) ("MiniPaged-Qwen: Qwen3
  Prefill FlashAttention" section 6).
* An item visits exactly the key tiles that hold a key visible to its last
  row: key j is visible to query i iff j <= i + Sk - Sq (the bottom-right
  causal limit of section 13 of the same page), counted here by brute force.
* Items are numbered longest first and dealt to CTAs in a serpentine over
  rounds, every item to exactly one CTA ("NVIDIA闪存注意力实操", section
  "ProgramId重映射").
"""

import numpy as np
import pytest

from exact_attention_16_gb300 import api

SHAPES = [
    # B, Sq, Sk, Hq, Hkv, causal
    (1, 300, 400, 8, 2, 1),      # Sk > Sq: offset 100, ragged tails
    (2, 400, 300, 4, 4, 1),      # Sq > Sk: the first 100 rows see nothing
    (1, 1280, 1536, 16, 16, 1),  # the causal MHA workload
    (3, 257, 257, 6, 2, 1),      # odd group size: two row tiles per pair item
    (2, 129, 1000, 32, 4, 0),    # not causal, G = 8
    (1, 1, 77, 2, 1, 1),         # one query row
    (4, 4096, 4096, 32, 8, 1),   # the 4K GQA workload
]


def _tiles_of(items, Sq):
    """(b, hq, r) of every non-empty 128-row tile the items compute."""
    out = []
    for b, hq0, hq1, _, r0, r1, _, _ in items:
        out.append((b, hq0, r0))
        if (hq1, r1) != (hq0, r0) and r1 < Sq:
            out.append((b, hq1, r1))
    return out


def _visible_key_tiles(r, Sq, Sk, causal):
    """Key tiles holding a key visible to some row of the tile starting at r,
    counted key by key."""
    last = min(r + 127, Sq - 1)
    keys = [j for j in range(Sk) if not causal or j <= last + Sk - Sq]
    return 0 if not keys else keys[-1] // 128 + 1


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}_Sq{}_Sk{}_H{}-{}_c{}".format(*s))
@pytest.mark.parametrize("key_split", [0, 1], ids=["pairs", "keysplit"])
def test_every_tile_once_with_its_head_and_key_range(shape, key_split):
    B, Sq, Sk, Hq, Hkv, causal = shape
    items, grid = api.fa_fwd_work_items(B, Sq, Sk, Hq, Hkv, causal, key_split, 152)
    G = Hq // Hkv
    tiles = _tiles_of(items, Sq)
    expected = {(b, h, m * 128) for b in range(B) for h in range(Hq) for m in range((Sq + 127) // 128)}
    assert len(tiles) == len(set(tiles)) and set(tiles) == expected
    for b, hq0, hq1, kvh, r0, r1, n_kv, _ in items:
        assert kvh == hq0 // G == hq1 // G
        want = max(_visible_key_tiles(r0, Sq, Sk, causal),
                   _visible_key_tiles(r1, Sq, Sk, causal) if r1 < Sq else 0)
        assert n_kv == want
        if key_split:
            assert (hq1, r1) == (hq0, r0)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}_Sq{}_Sk{}_H{}-{}_c{}".format(*s))
@pytest.mark.parametrize("key_split", [0, 1], ids=["pairs", "keysplit"])
def test_longest_first_serpentine_schedule(shape, key_split):
    B, Sq, Sk, Hq, Hkv, causal = shape
    for sms in (152, 7):
        items, grid = api.fa_fwd_work_items(B, Sq, Sk, Hq, Hkv, causal, key_split, sms)
        n = len(items)
        assert grid == min(n, sms)
        assert np.all(np.diff(items[:, 6]) <= 0)            # no item longer than one numbered before it
        cta = items[:, 7]
        assert cta.min() >= 0 and cta.max() < grid          # every item has one CTA
        for idx in range(n):
            rnd, pos = divmod(idx, grid)
            assert cta[idx] == (pos if rnd % 2 == 0 else grid - 1 - pos)


def test_pairs_share_key_value_heads_when_the_group_is_even():
    items, _ = api.fa_fwd_work_items(1, 512, 512, 8, 2, 1, 0, 152)
    assert np.all(items[:, 2] == items[:, 1] + 1) and np.all(items[:, 4] == items[:, 5])
    items, _ = api.fa_fwd_work_items(1, 512, 512, 6, 2, 1, 0, 152)    # G = 3: two row tiles of one head
    assert np.all(items[:, 2] == items[:, 1]) and np.all(items[:, 5] == items[:, 4] + 128)


@pytest.mark.parametrize("args", [
    (0, 128, 128, 2, 2, 1, 0, 152), (1, 128, 128, 3, 2, 1, 0, 152), (1, 128, 128, 2, 2, 2, 0, 152),
    (1, 128, 128, 2, 2, 1, 2, 152), (1, 128, 128, 2, 2, 1, 0, 0)])
def test_invalid_sizes_rejected(args):
    with pytest.raises(api.FAError):
        api.fa_fwd_work_items(*args)
