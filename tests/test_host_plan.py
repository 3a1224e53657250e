"""fa_fwd_host's chunk plan, on the CPU (host-only fa_fwd_host_plan query):
the chunks partition the work, every key a chunk's kernel reads has been
copied in by then, and the bottom-right mask each chunk's kernel applies to
its own rows and keys equals the mask of the whole problem (key j visible to
query i iff j <= i + Sk - Sq, "MiniPaged-Qwen: Qwen3 Prefill FlashAttention"
section 13), checked key by key."""

import numpy as np
import pytest

from exact_attention_16_gb300 import api

SHAPES = [
    # B, Sq, Sk, Hq, Hkv, D, causal
    (1, 16384, 16384, 32, 4, 128, 1),   # the bench workload: 4 KV-head ranges x 2 row halves
    (4, 4096, 4096, 32, 8, 128, 1),     # batches x KV-head ranges
    (2, 8192, 8192, 16, 8, 128, 1),
    (1, 1280, 1536, 16, 16, 128, 1),    # small: one chunk
    (1, 8192, 6000, 16, 2, 128, 1),     # Sq > Sk: the first rows see nothing
    (1, 6000, 9000, 8, 8, 128, 1),      # Sk > Sq
    (1, 9000, 9000, 8, 2, 64, 0),       # not causal: the second row range copies no keys
    (3, 333, 700, 6, 3, 96, 1),
    (1, 100, 0, 4, 2, 128, 1),          # no keys
]


def _visible(i, Sq, Sk, causal):
    return Sk if not causal else max(0, min(Sk, i + Sk - Sq + 1))


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}_Sq{}_Sk{}_H{}-{}_D{}_c{}".format(*s))
def test_chunks_partition_the_work_and_keep_the_mask(shape):
    B, Sq, Sk, Hq, Hkv, D, causal = shape
    plan = api.fa_fwd_host_plan(B, Sq, Sk, Hq, Hkv, D, causal)
    assert 1 <= len(plan) <= 8
    cover = np.zeros((B, Hkv, Sq), dtype=np.int32)
    copied = {}                                       # (b, h) -> keys copied so far, in chunk order
    for b0, b1, h0, h1, r0, r1, k0, k1, lim in plan:
        assert 0 <= b0 < b1 <= B and 0 <= h0 < h1 <= Hkv and 0 <= r0 < r1 <= Sq
        cover[b0:b1, h0:h1, r0:r1] += 1
        for b in range(b0, b1):
            for h in range(h0, h1):
                done = copied.get((b, h), 0)
                assert k0 == done and k1 >= k0      # copies continue where the last chunk stopped
                copied[(b, h)] = k1
                assert lim <= k1                      # every key the kernel reads is on the device
        # the chunk's kernel: rows [r0, r1) as its own Sq' = r1 - r0 queries
        # against keys [0, lim) with the bottom-right mask of those sizes
        rows = np.arange(r0, r1)
        chunk_vis = np.array([_visible(i - r0, r1 - r0, lim, causal) for i in rows])
        whole_vis = np.array([_visible(i, Sq, Sk, causal) for i in rows])
        assert np.array_equal(chunk_vis, whole_vis)
    assert np.all(cover == 1)                         # every (batch, KV head, row) exactly once
    for (b, h), k in copied.items():
        assert k == max(_visible(Sq - 1, Sq, Sk, causal), 0)   # and no key beyond what the last row sees


def test_plan_follows_the_size_rule():
    # about one chunk per 24 MiB of copies, at most eight
    assert len(api.fa_fwd_host_plan(1, 1280, 1536, 16, 16, 128, 1)) == 1
    assert len(api.fa_fwd_host_plan(1, 16384, 16384, 32, 4, 128, 1)) == 8
    assert len(api.fa_fwd_host_plan(4, 4096, 4096, 32, 8, 128, 1)) == 8


@pytest.mark.parametrize("args", [
    (0, 128, 128, 2, 2, 128, 1), (1, 128, 128, 3, 2, 128, 1), (1, 128, -1, 2, 2, 128, 1),
    (1, 128, 128, 2, 2, 0, 1), (1, 128, 128, 2, 2, 128, 2)])
def test_invalid_sizes_rejected(args):
    with pytest.raises(api.FAError):
        api.fa_fwd_host_plan(*args)
