"""CUDA path (through the C ABI) against the fp64 oracle, element by element.

Small and ragged shapes are compared on every element; so are the five
workloads at full size, in the exact launch configuration the bench times.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from exact_attention_16_gb300 import api  # noqa: E402
from exact_attention_16_gb300.workloads import WORKLOADS, Workload  # noqa: E402

from parity import check_every_element_pooled, check_full, run_gpu  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def W(B, Sq, Sk, Hq, Hkv, D, dtype="bf16", causal=False, sigma=1.0, seed=7):
    return Workload("case", B, Sq, Sk, Hq, Hkv, D, dtype, causal, sigma, 1.0, seed)


# ---- one tile, then several tiles and ragged tails, both head pairings
SMALL = [
    W(1, 128, 128, 2, 2, 128),                       # one tile pair, MHA (row-tile pairs)
    W(1, 128, 128, 2, 1, 128),                       # GQA 2:1 (head pairs)
    W(1, 128, 128, 2, 2, 64),
    W(1, 256, 256, 4, 2, 128, causal=True),
    W(1, 300, 257, 4, 4, 128, causal=False),         # ragged query and key tails
    W(1, 300, 257, 4, 4, 128, causal=True),          # Sq > Sk: first rows see nothing
    W(2, 257, 300, 8, 2, 128, "fp16", causal=True),  # Sk > Sq: offset 43
    W(1, 1, 1, 2, 1, 128),
    W(1, 1, 77, 2, 2, 64, causal=True),              # one query sees every key
    W(1, 77, 1, 2, 2, 64, causal=True),              # only the last row sees the key
    W(1, 520, 520, 6, 2, 64, "fp16", causal=True),   # G = 3 (odd): row-tile pairs
    W(2, 384, 640, 8, 8, 128, causal=True, sigma=2.0),   # sharp softmax: |O| up to ~4.5
    W(1, 2048, 2048, 4, 2, 128, causal=True, sigma=2.0),
    W(1, 1000, 1000, 4, 1, 128, "fp16", causal=True, sigma=2.0),
    W(1, 640, 384, 4, 1, 128, causal=True),          # G = 4
    W(1, 129, 1000, 32, 4, 128, causal=False),       # G = 8
    W(1, 384, 384, 4, 2, 256, causal=True),          # D = 256 (one-tile kernel, one key range)
    W(2, 200, 333, 4, 4, 256, "fp16", causal=False),
    W(1, 300, 257, 8, 1, 256, causal=True),          # D = 256, G = 8, Sq > Sk
    W(1, 300, 400, 32, 1, 128, causal=True),         # MQA, G = 32 (head pairs of one KV head)
    W(1, 200, 200, 64, 1, 64, "fp16", causal=False),  # MQA, G = 64
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: f"B{w.B}_Sq{w.Sq}_Sk{w.Sk}_H{w.Hq}-{w.Hkv}_D{w.D}_{w.dtype}_{'c' if w.causal else 'n'}")
def test_small_shapes_every_element(w):
    check_full(w)


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_full_size_workloads_every_element(w):
    """The five workloads at full size, launched as the bench launches them
    (preallocated O and LSE, the current stream), compared with the oracle on
    every element of every (batch, head): the oracle runs head by head in a
    pool of spawned processes. The error figures are printed and, when
    FA_PARITY_REPORT names a file, appended to it as one JSON line."""
    from exact_attention_16_gb300.workloads import draw_inputs
    q, k, v = draw_inputs(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.full_like(qd, float("nan"))
    lse = torch.full((w.B, w.Hq, w.Sq), float("nan"), dtype=torch.float32, device="cuda")
    api.fa_fwd(qd, kd, vd, scale=w.scale, causal=w.causal, out=out, lse=lse)
    assert api.fa_status() == 0
    check_every_element_pooled(w, out, lse, q, k, v)


# More row-tile-pair items than a 152-SM grid has CTAs, so CTAs run items back
# to back (each item's first Q K^T issued from the previous item's last K/V
# slot). At D = 64 P has tensor-memory columns of its own and the next Q K^T
# runs beside the softmax; at D = 128 P overwrites S.
SEVERAL_ITEMS = [
    W(1, 1280, 1280, 32, 16, 64, causal=True, seed=71),            # 160 items, causal lengths 1..10
    W(2, 1000, 1100, 24, 6, 64, "fp16", causal=False, seed=72),    # 192 items, ragged row and key tails
    W(1, 2560, 2800, 16, 16, 64, causal=True, sigma=2.0, seed=73),  # MHA: pairs of row tiles, offset mask
    W(1, 1280, 1280, 32, 16, 128, causal=True, seed=74),
]


@pytest.mark.parametrize("w", SEVERAL_ITEMS, ids=["d64_causal_160", "d64_ragged_192", "d64_mha_offset",
                                                  "d128_causal_160"])
def test_row_tile_pairs_several_items_per_cta_every_element(w):
    assert api.fa_debug_set_schedule(0) == api.FA_OK
    try:
        check_full(w)
    finally:
        api.fa_debug_set_schedule(-1)


def test_sk_zero_gives_zero_output_and_neg_inf_lse():
    q = torch.randn(1, 5, 2, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(1, 0, 2, 128, dtype=torch.bfloat16, device="cuda")
    o, lse = api.fa_fwd(q, k, k.clone(), causal=True)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(lse == float("-inf"))


def test_lse_optional_and_output_overwritten():
    w = W(1, 200, 200, 2, 2, 128, causal=True)
    from exact_attention_16_gb300.workloads import draw_inputs
    q, k, v = (t.cuda() for t in draw_inputs(w))
    o_ref, _ = api.fa_fwd(q, k, v, causal=True)
    out = torch.full_like(q, float("nan"))
    o2, l2 = api.fa_fwd(q, k, v, causal=True, out=out, return_lse=False)
    torch.cuda.synchronize()
    assert l2 is None and torch.equal(o2, o_ref)


def test_repeatable_and_stream_ordered():
    w = W(1, 512, 512, 4, 2, 128, causal=True)
    from exact_attention_16_gb300.workloads import draw_inputs
    q, k, v = (t.cuda() for t in draw_inputs(w))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1 = api.fa_fwd(q, k, v, causal=True)
        o2, l2 = api.fa_fwd(q, k, v, causal=True)
    s.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def _oracle_compare(q, k, v, o, lse, scale, causal):
    import oracle
    from parity import compare
    o_ref, l_ref = oracle.attention(q.float().cpu().numpy(), k.float().cpu().numpy(), v.float().cpu().numpy(),
                                    scale, causal)
    return compare(o.float().cpu().numpy().transpose(0, 2, 1, 3), lse.cpu().numpy(),
                   o_ref.transpose(0, 2, 1, 3), l_ref)


def test_bhsd_layout_with_strided_output():
    """(B, H, S, D) storage passed as transposed views, O written into a
    (B, H, S, D) buffer through its transposed view."""
    from exact_attention_16_gb300.workloads import draw_inputs
    w = W(2, 300, 333, 8, 2, 128, causal=True, seed=11)
    q, k, v = draw_inputs(w)
    qb, kb, vb = (t.transpose(1, 2).contiguous().cuda() for t in (q, k, v))   # (B, H, S, D)
    o_store = torch.full((w.B, w.Hq, w.Sq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    o, lse = api.fa_fwd(qb.transpose(1, 2), kb.transpose(1, 2), vb.transpose(1, 2), scale=w.scale, causal=True,
                        out=o_store.transpose(1, 2))
    assert api.fa_status() == 0
    assert o.data_ptr() == o_store.data_ptr()
    _oracle_compare(q, k, v, o, lse, w.scale, True)


def test_packed_qkv_views():
    """Q, K, V as views into one (B, S, 3, H, D) buffer (MHA), D = 64."""
    g = torch.Generator().manual_seed(12)
    B, S, H, D = 2, 257, 4, 64
    qkv = (torch.randn(B, S, 3, H, D, generator=g)).to(torch.float16)
    qkv_d = qkv.cuda()
    q, k, v = qkv_d[:, :, 0], qkv_d[:, :, 1], qkv_d[:, :, 2]
    assert not q.is_contiguous()
    o, lse = api.fa_fwd(q, k, v, causal=False)
    assert api.fa_status() == 0
    _oracle_compare(qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2], o, lse, D ** -0.5, False)


def test_d256_strided_bhsd():
    from exact_attention_16_gb300.workloads import draw_inputs
    w = W(1, 250, 260, 4, 2, 256, causal=True, seed=13)
    q, k, v = draw_inputs(w)
    qb, kb, vb = (t.transpose(1, 2).contiguous().cuda() for t in (q, k, v))
    o_store = torch.full((w.B, w.Hq, w.Sq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    o, lse = api.fa_fwd(qb.transpose(1, 2), kb.transpose(1, 2), vb.transpose(1, 2), scale=w.scale, causal=True,
                        out=o_store.transpose(1, 2))
    assert api.fa_status() == 0
    _oracle_compare(q, k, v, o, lse, w.scale, True)


PADDED_D = [
    W(1, 300, 257, 4, 2, 32, causal=True),           # kernel D 64, zero padded
    W(1, 200, 200, 2, 2, 16, "fp16", causal=False),
    W(2, 130, 190, 4, 4, 48, causal=True),
    W(1, 257, 300, 8, 2, 96, causal=True),           # kernel D 128
    W(1, 256, 256, 4, 1, 80, "fp16", causal=False),
    W(1, 129, 129, 2, 2, 112, causal=True),
    W(1, 200, 211, 4, 2, 160, causal=True),          # kernel D 256 (one-tile path)
    W(1, 150, 150, 2, 2, 192, "fp16", causal=False),
]


@pytest.mark.parametrize("w", PADDED_D, ids=lambda w: f"D{w.D}_{w.dtype}_{'c' if w.causal else 'n'}_Sq{w.Sq}_Sk{w.Sk}")
def test_head_dims_padded_to_the_kernel_tile(w):
    check_full(w)


def test_padded_head_dim_strided_bhsd():
    from exact_attention_16_gb300.workloads import draw_inputs
    w = W(1, 220, 230, 4, 2, 96, causal=True, seed=14)
    q, k, v = draw_inputs(w)
    qb, kb, vb = (t.transpose(1, 2).contiguous().cuda() for t in (q, k, v))
    o, lse = api.fa_fwd(qb.transpose(1, 2), kb.transpose(1, 2), vb.transpose(1, 2), scale=w.scale, causal=True)
    assert api.fa_status() == 0
    _oracle_compare(q, k, v, o, lse, w.scale, True)


def _far_below_zero(B, Sq, Sk, Hq, Hkv, D, seed=5):
    """Inputs whose scores all sit near -181 (about -261 in log2 units): every
    weight 2^(s - m) underflows fp32 unless m comes from the row's own scores,
    yet the softmax is an ordinary one over score differences of a few units."""
    g = torch.Generator().manual_seed(seed)
    q = (4.0 + 0.05 * torch.randn(B, Sq, Hq, D, generator=g)).to(torch.bfloat16)
    k = (-4.0 + 0.05 * torch.randn(B, Sk, Hkv, D, generator=g)).to(torch.bfloat16)
    v = torch.randn(B, Sk, Hkv, D, generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("mode", [0, 1], ids=["pairs", "keysplit"])
@pytest.mark.parametrize("D", [64, 128])
def test_scores_far_below_zero(mode, D):
    q, k, v = _far_below_zero(1, 300, 300, 4, 2, D)
    assert api.fa_debug_set_schedule(mode) == api.FA_OK
    try:
        o, lse = api.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
        torch.cuda.synchronize()
    finally:
        api.fa_debug_set_schedule(-1)
    assert api.fa_status() == 0
    _oracle_compare(q, k, v, o, lse, D ** -0.5, True)


def test_scores_far_below_zero_one_tile_kernel():
    # D = 256 runs the one-tile split-KV kernel; the decode entry splits the keys
    q, k, v = _far_below_zero(1, 200, 333, 4, 1, 256)
    o, lse = api.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    _oracle_compare(q, k, v, o, lse, 256 ** -0.5, True)
    q1, k1, v1 = _far_below_zero(4, 1, 2000, 8, 2, 128, seed=6)
    o1, l1 = api.fa_fwd_decode(q1.cuda(), k1.cuda(), v1.cuda(), causal=True, num_splits=3)
    torch.cuda.synchronize()
    assert api.fa_status() == 0
    _oracle_compare(q1, k1, v1, o1, l1, 128 ** -0.5, True)


def test_scores_far_above_zero():
    """Every score near +181 (about +261 in log2 units): 2^s overflows fp32, so
    the result is finite only if each weight is taken relative to the row's
    running max. Both decompositions, the one-tile kernel and decode splits."""
    q, k, v = _far_below_zero(1, 300, 300, 4, 2, 128, seed=8)
    k = -k.float()
    k = k.to(torch.bfloat16)
    for mode in (0, 1):
        assert api.fa_debug_set_schedule(mode) == api.FA_OK
        try:
            o, lse = api.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
            torch.cuda.synchronize()
        finally:
            api.fa_debug_set_schedule(-1)
        assert api.fa_status() == 0
        _oracle_compare(q, k, v, o, lse, 128 ** -0.5, True)
    q2, k2, v2 = _far_below_zero(2, 100, 700, 8, 2, 256, seed=9)
    k2 = (-k2.float()).to(torch.bfloat16)
    o2, l2 = api.fa_fwd(q2.cuda(), k2.cuda(), v2.cuda(), causal=False)
    torch.cuda.synchronize()
    _oracle_compare(q2, k2, v2, o2, l2, 256 ** -0.5, False)
    q3, k3, v3 = _far_below_zero(3, 1, 2000, 8, 2, 128, seed=10)
    k3 = (-k3.float()).to(torch.bfloat16)
    o3, l3 = api.fa_fwd_decode(q3.cuda(), k3.cuda(), v3.cuda(), causal=True, num_splits=4)
    torch.cuda.synchronize()
    assert api.fa_status() == 0
    _oracle_compare(q3, k3, v3, o3, l3, 128 ** -0.5, True)


@pytest.mark.parametrize("scale", [1e-3, 0.05, 0.5, 3.0], ids=["s1e-3", "s0.05", "s0.5", "s3"])
def test_explicit_scales(scale):
    """The scale is an argument, not 1/sqrt(D): near-uniform weights (1e-3)
    up to near one-hot rows (3.0, scores with a spread of about 34), through
    each kernel: row-tile pairs (D = 128), key-split items (D = 64), the
    one-tile kernel (D = 256) and decode splits."""
    from exact_attention_16_gb300.workloads import draw_inputs
    cases = [(W(2, 333, 517, 8, 2, 128, causal=True, seed=21), 0, "fwd"),
             (W(1, 300, 300, 4, 4, 64, "fp16", causal=False, seed=22), 1, "fwd"),
             (W(1, 200, 333, 4, 1, 256, causal=True, seed=23), -1, "fwd"),
             (W(4, 1, 3000, 16, 4, 128, causal=True, seed=24), -1, "decode")]
    for w, mode, entry in cases:
        q, k, v = draw_inputs(w)
        assert api.fa_debug_set_schedule(mode) == api.FA_OK
        try:
            if entry == "fwd":
                o, lse = api.fa_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=w.causal)
            else:
                o, lse = api.fa_fwd_decode(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=w.causal,
                                           num_splits=5)
            torch.cuda.synchronize()
        finally:
            api.fa_debug_set_schedule(-1)
        assert api.fa_status() == 0
        _oracle_compare(q, k, v, o, lse, scale, w.causal)


# LSE bound for integer-valued inputs. With q, k integers in [-2, 2) every
# product q_d k_d is an integer and the fp32 accumulation of D <= 256 of them
# is exact, so the scores carry no error and the LSE error comes from the
# softmax arithmetic alone: the fp32 rounding of scale * log2(e) (relative
# 6e-8 on scaled scores of a few tens), the fp32 sums of at most a few thousand
# weights per row (a few 1e-6 relative), the approximate exp2 and log2
# (about 2^-22 relative) and the final (m + log2 l) * ln 2 in fp32 (two
# roundings of a value below 70). Together these stay below 1.5e-5; the bound
# keeps a margin of three on top, twenty times tighter than the general 1e-3.
INT_LSE_MAX_ABS = 5e-5


def _rising_scores(B, Sq, Sk, Hq, Hkv, D, seed=41):
    """Scores that rise by about 10 (in log2 units) every 128 keys: q is all
    ones and every component of key j is 0.054 j / sqrt(D), so with the
    default scale s_ij = 0.054 j. Each key tile raises the row max past the
    lazy-rescale threshold, so O~ is rescaled on every tile, and a rescale
    that landed after P V had started, or was skipped, would leave earlier
    tiles weighted 2^10 too high."""
    g = torch.Generator().manual_seed(seed)
    q = torch.ones(B, Sq, Hq, D).to(torch.bfloat16)
    c = (0.054 * torch.arange(Sk, dtype=torch.float64) / D ** 0.5).to(torch.float32)
    k = c.view(1, Sk, 1, 1).expand(B, Sk, Hkv, D).contiguous().to(torch.bfloat16)
    v = torch.randn(B, Sk, Hkv, D, generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mode", [0, 1], ids=["pairs", "keysplit"])
def test_rescale_on_every_key_tile(mode, D, causal):
    q, k, v = _rising_scores(2, 300, 700, 4, 2, D)
    assert api.fa_debug_set_schedule(mode) == api.FA_OK
    try:
        o, lse = api.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
        torch.cuda.synchronize()
    finally:
        api.fa_debug_set_schedule(-1)
    assert api.fa_status() == 0
    _oracle_compare(q, k, v, o, lse, D ** -0.5, causal)


def _integer_inputs(B, Sq, Sk, Hq, Hkv, D, dtype, seed):
    """Integer-valued q, k, v in [-2, 2) (the integer test inputs of the
    CuTe-DSL example "ampere/flash_attention_v2.py", whose Q K^T is exact in
    every precision)."""
    g = torch.Generator().manual_seed(seed)
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    return tuple(torch.randint(-2, 2, shape, generator=g).to(dt)
                 for shape in ((B, Sq, Hq, D), (B, Sk, Hkv, D), (B, Sk, Hkv, D)))


def _int_lse_check(q, k, v, o, lse, scale, causal):
    import oracle
    from parity import compare
    o_ref, l_ref = oracle.attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), scale, causal)
    got = lse.cpu().numpy().astype(np.float64)
    compare(o.float().cpu().numpy().transpose(0, 2, 1, 3), got, o_ref.transpose(0, 2, 1, 3), l_ref)
    live = np.isfinite(l_ref)
    assert np.array_equal(live, np.isfinite(got))
    err = float(np.abs(got[live] - l_ref[live]).max()) if live.any() else 0.0
    assert err <= INT_LSE_MAX_ABS, err


@pytest.mark.parametrize("mode,D,dtype,causal", [
    (0, 128, "bf16", True), (1, 128, "bf16", True), (0, 64, "fp16", False), (1, 64, "fp16", False),
    (-1, 256, "bf16", True)], ids=["d128_bf16_causal_pairs", "d128_bf16_causal_keysplit", "d64_fp16_pairs",
                                   "d64_fp16_keysplit", "d256_bf16_causal"])
def test_integer_inputs_exact_scores(mode, D, dtype, causal):
    """Exact scores isolate the softmax: O within the general tolerance and
    LSE within the tighter bound above, for both work decompositions at
    D = 64 / 128 and for the one-tile kernel that D = 256 runs."""
    q, k, v = _integer_inputs(2, 300, 421, 8, 2, D, dtype, seed=31 + D)
    assert api.fa_debug_set_schedule(mode) == api.FA_OK
    try:
        o, lse = api.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
        torch.cuda.synchronize()
    finally:
        api.fa_debug_set_schedule(-1)
    assert api.fa_status() == 0
    _int_lse_check(q, k, v, o, lse, D ** -0.5, causal)


def test_integer_inputs_exact_scores_decode_splits():
    """The split-KV decode path and its merge of partial states on exact
    scores: the merged LSE obeys the same bound."""
    q, k, v = _integer_inputs(3, 2, 3000, 16, 4, 128, "bf16", seed=77)
    o, lse = api.fa_fwd_decode(q.cuda(), k.cuda(), v.cuda(), causal=True, num_splits=5)
    torch.cuda.synchronize()
    assert api.fa_status() == 0
    _int_lse_check(q, k, v, o, lse, 128 ** -0.5, True)


def _random_shapes(n=24, seed=2024):
    """Seeded random shapes across every argument the path takes: batch,
    ragged lengths (Sq > Sk and Sq < Sk), GQA groups 1-8, head dims 32-256
    (padded ones included), both dtypes, causal or not, sharp or flat
    softmax."""
    import numpy as np
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        hkv = int(rng.choice([1, 2, 4]))
        g = int(rng.choice([1, 2, 3, 4, 8]))
        d = int(rng.choice([32, 64, 96, 128, 128, 192, 256]))
        sq = int(rng.integers(1, 700))
        sk = int(rng.integers(1, 700))
        out.append(Workload(f"r{i}", int(rng.integers(1, 4)), sq, sk, g * hkv, hkv, d,
                            str(rng.choice(["bf16", "fp16"])), bool(rng.integers(0, 2)),
                            float(rng.choice([0.5, 1.0, 2.0])), 1.0, int(rng.integers(1, 1 << 30))))
    return out


@pytest.mark.parametrize("i", range(24))
def test_random_shapes_every_element(i):
    w = _random_shapes()[i]
    mode = i % 2 if w.D <= 128 else -1   # alternate the forced schedule
    assert api.fa_debug_set_schedule(mode) == api.FA_OK
    try:
        check_full(w)
    finally:
        api.fa_debug_set_schedule(-1)
