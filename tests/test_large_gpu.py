"""Tensors past 2^31 elements: the CUDA path against the fp64 oracle on
sampled rows at the far end of each buffer, where a 32-bit element or byte
offset would wrap.

Inputs are several GB, so they are drawn on the device (seeded Philox) and
the oracle reads back only the (batch, head) slices it checks. Each case
holds 10-27 GB of device memory and frees it before the next.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_attention_16_gb300 import api  # noqa: E402
from exact_attention_16_gb300.workloads import draw_device  # noqa: E402

from parity import compare  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _rows(S, rng, n_random=24):
    rows = set(range(S - 130, S)) | {0, 1, 127, 128} | set(int(x) for x in rng.integers(0, S, size=n_random))
    return np.array(sorted(r for r in rows if 0 <= r < S), dtype=np.int64)


def _check_heads(q, k, v, o, lse, scale, causal, heads, rng):
    """Oracle rows of each (b, hq) from that head's slices of q, k and v."""
    B, Sq, Hq, D = q.shape
    Hkv = k.shape[2]
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for b, hq in heads:
        kvh = hq // (Hq // Hkv)
        rows = _rows(Sq, rng)
        idx = torch.from_numpy(rows).to(q.device)
        q1 = q[b:b + 1, :, hq:hq + 1, :].float().cpu().numpy()
        k1 = k[b:b + 1, :, kvh:kvh + 1, :].float().cpu().numpy()
        v1 = v[b:b + 1, :, kvh:kvh + 1, :].float().cpu().numpy()
        ro, rl = oracle.attention_rows(q1, k1, v1, scale, causal, 0, 0, rows)
        got_o.append(o[b, :, hq, :].index_select(0, idx).float().cpu().numpy())
        got_l.append(lse[b, hq].index_select(0, idx).cpu().numpy())
        ref_o.append(ro)
        ref_l.append(rl)
    return compare(np.concatenate(got_o), np.concatenate(got_l), np.concatenate(ref_o), np.concatenate(ref_l))


def test_prefill_pairs_output_past_2_pow_31_elements():
    """Row-tile-pair kernel, D = 128: q and O hold 2.4e9 elements (4.8 GB)."""
    B, S, Hq, Hkv, D = 2, 73728, 128, 8, 128
    assert B * S * Hq * D > 2 ** 31
    q = draw_device((B, S, Hq, D), "bf16", 1.0, 501)
    k = draw_device((B, S, Hkv, D), "bf16", 1.0, 502)
    v = draw_device((B, S, Hkv, D), "bf16", 1.0, 503)
    scale = D ** -0.5
    o, lse = api.fa_fwd(q, k, v, scale=scale, causal=True)
    assert api.fa_status() == 0
    _check_heads(q, k, v, o, lse, scale, True, [(B - 1, Hq - 1), (B - 1, Hq // 2), (0, 3)],
                 np.random.default_rng(1))


def test_prefill_one_tile_output_past_2_pow_31_elements():
    """One-tile kernel (D = 256, direct O stores): 2.7e9 elements (5.4 GB)."""
    B, S, Hq, Hkv, D = 2, 40960, 128, 8, 256
    assert B * S * Hq * D > 2 ** 31
    q = draw_device((B, S, Hq, D), "bf16", 1.0, 511)
    k = draw_device((B, S, Hkv, D), "bf16", 1.0, 512)
    v = draw_device((B, S, Hkv, D), "bf16", 1.0, 513)
    scale = D ** -0.5
    o, lse = api.fa_fwd(q, k, v, scale=scale, causal=True)
    assert api.fa_status() == 0
    _check_heads(q, k, v, o, lse, scale, True, [(B - 1, Hq - 1), (0, 17)], np.random.default_rng(2))


def test_decode_keys_past_2_pow_31_elements():
    """Split-KV decode over 1.1 M keys: k and v hold 2.25e9 elements each."""
    B, Sq, Sk, Hq, Hkv, D = 1, 1, 1_100_000, 64, 16, 128
    assert B * Sk * Hkv * D > 2 ** 31
    q = draw_device((B, Sq, Hq, D), "fp16", 1.0, 521)
    k = draw_device((B, Sk, Hkv, D), "fp16", 1.0, 522)
    v = draw_device((B, Sk, Hkv, D), "fp16", 1.0, 523)
    scale = D ** -0.5
    o, lse = api.fa_fwd_decode(q, k, v, scale=scale, causal=True)
    assert api.fa_status() == 0
    _check_heads(q, k, v, o, lse, scale, True, [(0, Hq - 1), (0, 0)], np.random.default_rng(3))


@pytest.mark.parametrize("Sq", [300_000, 540_000], ids=["rows_x_D_above_2_pow_31", "rows_x_D_above_2_pow_32"])
def test_merge_past_32_bit_indices(Sq):
    """fa_merge of two bf16 parts of B * Sq * Hq * D elements each: above
    2^31 (unsigned 32-bit indexing) and above 2^32 (64-bit indexing)."""
    n, B, Hq, D = 2, 1, 64, 128
    o_parts = draw_device((n, B, Sq, Hq, D), "bf16", 1.0, 530 + Sq % 7)
    lse_parts = draw_device((n, B, Hq, Sq), "fp32", 3.0, 540 + Sq % 7)
    lse_parts[0, 0, Hq - 1, Sq - 2] = float("-inf")             # a part with no key
    lse_parts[:, 0, Hq - 1, Sq - 1] = float("-inf")             # a row with none at all
    o, lse = api.fa_merge(o_parts, lse_parts)
    assert api.fa_status() == 0
    rng = np.random.default_rng(4)
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for h in (Hq - 1, 5):
        rows = _rows(Sq, rng)
        idx = torch.from_numpy(rows).cuda()
        op = o_parts[:, :, :, h, :].index_select(2, idx)[:, :, :, None, :].float().cpu().numpy()
        lp = lse_parts[:, :, h, :].index_select(2, idx)[:, :, None, :].cpu().numpy()
        ro, rl = oracle.merge_partials(op, lp)                  # (1, k, 1, D), (1, 1, k)
        got_o.append(o[0, :, h, :].index_select(0, idx).float().cpu().numpy())
        got_l.append(lse[0, h].index_select(0, idx).cpu().numpy())
        ref_o.append(ro[0, :, 0, :])
        ref_l.append(rl[0, 0])
    compare(np.concatenate(got_o), np.concatenate(got_l), np.concatenate(ref_o), np.concatenate(ref_l))
