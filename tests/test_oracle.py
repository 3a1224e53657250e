"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these tests re-types the oracle's formula: each compares it with a
closed form, an invariant, a library routine it does not use (SciPy), a
brute-force loop, the online recurrence, or a table printed on the pages.
A final group plants plausible mistakes in the oracle and checks that some
pin catches each one.
"""

import math
import os

import numpy as np
import pytest
import scipy.special as sps

import oracle
from oracle import exact as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_qkv(seed, B, Sq, Sk, Hq, Hkv, D, sigma=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Sq, Hq, D)) * sigma
    k = rng.standard_normal((B, Sk, Hkv, D)) * sigma
    v = rng.standard_normal((B, Sk, Hkv, D))
    return q, k, v


def n_visible(i, Sq, Sk, causal):
    """Closed-form count of keys row i sees (bottom-right causal)."""
    if not causal:
        return Sk
    return min(Sk, max(0, i + Sk - Sq + 1))


# --------------------------------------------------------------------------
# Tables printed on the pages
# --------------------------------------------------------------------------

def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


def test_gqa_head_map_matches_printed_tables():
    rows = _read_table("gqa_head_map.txt")
    assert len(rows) >= 10
    for Hq, Hkv, qh, kvh in rows:
        assert oracle.kv_head_of(qh, Hq, Hkv) == kvh


def test_causal_limit_matches_printed_example():
    rows = _read_table("causal_limit.txt")
    assert rows
    for q_len, kv_len, qi, first_invisible in rows:
        vis = oracle.visibility([qi], q_len, kv_len, causal=True)[0]
        assert vis[:first_invisible].all()
        assert not vis[first_invisible:].any()


# --------------------------------------------------------------------------
# Invariants and closed forms
# --------------------------------------------------------------------------

SHAPES = [
    # (Sq, Sk, causal)
    (7, 7, False),
    (7, 7, True),
    (5, 11, True),     # more keys than queries: offset +6
    (11, 5, True),     # more queries than keys: rows 0..5 see nothing
    (9, 13, False),
]


@pytest.mark.parametrize("Sq,Sk,causal", SHAPES)
def test_probability_rows_sum_to_one(Sq, Sk, causal):
    q, k, _ = rand_qkv(1, 1, Sq, Sk, 2, 1, 8, sigma=2.0)
    for hq in range(2):
        P = oracle.probabilities(q, k, 0.37, causal, 0, hq)
        for i in range(Sq):
            cnt = n_visible(i, Sq, Sk, causal)
            if cnt == 0:
                assert np.all(P[i] == 0.0)
            else:
                assert abs(P[i].sum() - 1.0) < 1e-12
                assert np.all(P[i, cnt:] == 0.0)      # masked keys carry no weight
                assert np.all(P[i, :cnt] > 0.0)


@pytest.mark.parametrize("Sq,Sk,causal", SHAPES)
def test_constant_v_returns_the_constant(Sq, Sk, causal):
    B, Hq, Hkv, D = 2, 4, 2, 6
    q, k, _ = rand_qkv(2, B, Sq, Sk, Hq, Hkv, D, sigma=3.0)
    c = np.arange(B * Hkv * D, dtype=np.float64).reshape(B, 1, Hkv, D) * 0.25 - 1.0
    v = np.broadcast_to(c, (B, Sk, Hkv, D)).copy()
    o, lse = oracle.attention(q, k, v, 0.5, causal)
    for b in range(B):
        for hq in range(Hq):
            g = hq // (Hq // Hkv)
            for i in range(Sq):
                if n_visible(i, Sq, Sk, causal) == 0:
                    assert np.all(o[b, i, hq] == 0.0)
                    assert lse[b, hq, i] == -np.inf
                else:
                    np.testing.assert_allclose(o[b, i, hq], c[b, 0, g], rtol=0, atol=1e-12)


@pytest.mark.parametrize("Sq,Sk,causal", SHAPES)
def test_zero_scores_give_prefix_means(Sq, Sk, causal):
    """q = 0: P is uniform on the visible keys, so O_i is the mean of the
    visible v rows and LSE_i = ln(#visible). The means come from cumulative
    sums, which pins the bottom-right mask offset exactly."""
    B, Hq, Hkv, D = 1, 2, 2, 5
    _, k, v = rand_qkv(3, B, Sq, Sk, Hq, Hkv, D)
    q = np.zeros((B, Sq, Hq, D))
    o, lse = oracle.attention(q, k, v, 1.0, causal)
    csum = np.cumsum(v, axis=1)
    for hq in range(Hq):
        for i in range(Sq):
            cnt = n_visible(i, Sq, Sk, causal)
            if cnt == 0:
                assert lse[0, hq, i] == -np.inf
                continue
            np.testing.assert_allclose(o[0, i, hq], csum[0, cnt - 1, hq] / cnt, atol=1e-12)
            assert abs(lse[0, hq, i] - math.log(cnt)) < 1e-12


@pytest.mark.parametrize("Sq,Sk,causal", SHAPES)
def test_zero_scale_gives_prefix_means(Sq, Sk, causal):
    """scale = 0 with random q: every visible score is 0 whatever q and k
    are, so the rows are the same prefix means as for q = 0 and LSE_i =
    ln(#visible) (the scale is a free argument of softmax(scale Q K^T + M))."""
    B, Hq, Hkv, D = 1, 2, 1, 5
    q, k, v = rand_qkv(13, B, Sq, Sk, Hq, Hkv, D, sigma=3.0)
    o, lse = oracle.attention(q, k, v, 0.0, causal)
    csum = np.cumsum(v, axis=1)
    for hq in range(Hq):
        for i in range(Sq):
            cnt = n_visible(i, Sq, Sk, causal)
            if cnt == 0:
                assert lse[0, hq, i] == -np.inf and np.all(o[0, i, hq] == 0.0)
                continue
            np.testing.assert_allclose(o[0, i, hq], csum[0, cnt - 1, 0] / cnt, atol=1e-12)
            assert abs(lse[0, hq, i] - math.log(cnt)) < 1e-12


@pytest.mark.parametrize("Sq,Sk,causal", SHAPES)
def test_negative_scale_equals_negated_queries(Sq, Sk, causal):
    """scale * (q . k) = (-scale) * ((-q) . k): a negative scale gives the
    result of its magnitude on negated queries (negation is exact in fp64)."""
    q, k, v = rand_qkv(14, 2, Sq, Sk, 4, 2, 6)
    o1, l1 = oracle.attention(q, k, v, -0.7, causal)
    o2, l2 = oracle.attention(-q, k, v, 0.7, causal)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    live = np.isfinite(l2)
    assert np.array_equal(live, np.isfinite(l1))
    np.testing.assert_allclose(l1[live], l2[live], rtol=0, atol=1e-12)


def test_negative_scale_two_keys_favour_the_lower_score():
    """With a negative scale the key with the LOWER dot product gets the
    larger weight: two keys give sigmoid weights of scale * (a - b)."""
    rng = np.random.default_rng(15)
    q = rng.standard_normal((1, 5, 1, 4))
    k = rng.standard_normal((1, 2, 1, 4))
    v = rng.standard_normal((1, 2, 1, 4))
    scale = -1.3
    o, lse = oracle.attention(q, k, v, scale, causal=False)
    for i in range(5):
        a = float(np.dot(q[0, i, 0], k[0, 0, 0]))
        b = float(np.dot(q[0, i, 0], k[0, 1, 0]))
        w0 = sps.expit(scale * (a - b))
        np.testing.assert_allclose(o[0, i, 0], w0 * v[0, 0, 0] + (1 - w0) * v[0, 1, 0], atol=1e-13)
        assert abs(lse[0, 0, i] - np.logaddexp(scale * a, scale * b)) < 1e-12


def test_two_keys_weights_are_sigmoids():
    rng = np.random.default_rng(4)
    Sq, Sk, D = 6, 2, 3
    q = rng.standard_normal((1, Sq, 1, D)) * 2
    k = rng.standard_normal((1, Sk, 1, D)) * 2
    v = rng.standard_normal((1, Sk, 1, D))
    scale = 0.8
    o, lse = oracle.attention(q, k, v, scale, causal=False)
    for i in range(Sq):
        a = scale * float(np.dot(q[0, i, 0], k[0, 0, 0]))
        b = scale * float(np.dot(q[0, i, 0], k[0, 1, 0]))
        w0, w1 = sps.expit(a - b), sps.expit(b - a)
        np.testing.assert_allclose(o[0, i, 0], w0 * v[0, 0, 0] + w1 * v[0, 1, 0], atol=1e-13)
        assert abs(lse[0, 0, i] - np.logaddexp(a, b)) < 1e-12


def test_dominant_key_without_overflow():
    """One key scores >= 60 above the others at |s| ~ 1000: exp(s) alone
    would overflow, so this also pins the max subtraction."""
    Sq, Sk, D = 4, 9, 3
    q = np.zeros((1, Sq, 1, D))
    q[..., 0] = 1.0
    k = np.zeros((1, Sk, 1, D))
    k[0, :, 0, 0] = 900.0 + np.arange(Sk)       # scores 900..908
    k[0, 5, 0, 0] = 1000.0                      # dominant, margin 92
    v = np.random.default_rng(5).standard_normal((1, Sk, 1, D))
    o, lse = oracle.attention(q, k, v, 1.0, causal=False)
    assert np.all(np.isfinite(o))
    for i in range(Sq):
        np.testing.assert_allclose(o[0, i, 0], v[0, 5, 0], rtol=0, atol=1e-30)
        assert abs(lse[0, 0, i] - 1000.0) < 1e-12


def test_single_key():
    q, k, v = rand_qkv(6, 2, 5, 1, 4, 2, 7)
    scale = 0.3
    o, lse = oracle.attention(q, k, v, scale, causal=False)
    for b in range(2):
        for hq in range(4):
            g = hq // 2
            np.testing.assert_allclose(o[b, :, hq], np.broadcast_to(v[b, 0, g], (5, 7)), atol=1e-14)
            s = scale * np.einsum("id,d->i", q[b, :, hq], k[b, 0, g])
            np.testing.assert_allclose(lse[b, hq], s, atol=1e-13)


@pytest.mark.parametrize("Sq,Sk,causal", SHAPES)
def test_matches_scipy_softmax_and_logsumexp(Sq, Sk, causal):
    q, k, v = rand_qkv(7, 1, Sq, Sk, 1, 1, 4, sigma=1.5)
    scale = 0.6
    o, lse = oracle.attention(q, k, v, scale, causal)
    P = oracle.probabilities(q, k, scale, causal, 0, 0)
    s = scale * np.einsum("id,jd->ij", q[0, :, 0], k[0, :, 0])
    for i in range(Sq):
        cnt = n_visible(i, Sq, Sk, causal)
        if cnt == 0:
            continue
        ref_p = sps.softmax(s[i, :cnt])
        np.testing.assert_allclose(P[i, :cnt], ref_p, atol=1e-14)
        np.testing.assert_allclose(o[0, i, 0], ref_p @ v[0, :cnt, 0], atol=1e-13)
        assert abs(lse[0, 0, i] - sps.logsumexp(s[i, :cnt])) < 1e-12


# --------------------------------------------------------------------------
# Brute force, online recurrence, GQA, mask forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("Sq,Sk,causal", SHAPES)
def test_brute_force_equals_two_pass(Sq, Sk, causal):
    q, k, v = rand_qkv(8, 2, Sq, Sk, 4, 2, 3, sigma=1.3)
    o1, l1 = oracle.attention(q, k, v, 0.45, causal)
    o2, l2 = oracle.attention_brute(q, k, v, 0.45, causal)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(l1), np.isinf(l2))
    fin = np.isfinite(l2)
    np.testing.assert_allclose(l1[fin], l2[fin], atol=1e-12)


@pytest.mark.parametrize("Sq,Sk,causal", SHAPES)
def test_online_recurrence_equals_two_pass_for_every_tile_size(Sq, Sk, causal):
    q, k, v = rand_qkv(9, 1, Sq, Sk, 2, 1, 4, sigma=2.0)
    o_ref, l_ref = oracle.attention(q, k, v, 0.7, causal)
    fin = np.isfinite(l_ref)
    for bn in range(1, Sk + 1):
        o, l = oracle.attention_online(q, k, v, 0.7, causal, bn)
        np.testing.assert_allclose(o, o_ref, atol=1e-12)
        np.testing.assert_array_equal(np.isfinite(l), fin)
        np.testing.assert_allclose(l[fin], l_ref[fin], atol=1e-12)


def test_gqa_equals_mha_with_repeated_heads():
    B, Sq, Sk, Hq, Hkv, D = 2, 6, 9, 8, 2, 4
    q, k, v = rand_qkv(10, B, Sq, Sk, Hq, Hkv, D)
    G = Hq // Hkv
    k_rep = np.repeat(k, G, axis=2)      # head h of k_rep is kv head h // G
    v_rep = np.repeat(v, G, axis=2)
    for causal in (False, True):
        o1, l1 = oracle.attention(q, k, v, 0.5, causal)
        o2, l2 = oracle.attention(q, k_rep, v_rep, 0.5, causal)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


def test_bottom_right_equals_top_left_when_square():
    """With Sq == Sk the causal set is the lower triangle (i >= j) of
    "NVIDIA闪存注意力实操" section "因果注意力"; compare with an explicit
    np.tril mask applied through SciPy's softmax."""
    S, D = 10, 3
    q, k, v = rand_qkv(11, 1, S, S, 1, 1, D, sigma=1.7)
    o, _ = oracle.attention(q, k, v, 1.1, causal=True)
    s = 1.1 * q[0, :, 0] @ k[0, :, 0].T
    tri = np.tril(np.ones((S, S), dtype=bool))
    p = sps.softmax(np.where(tri, s, -np.inf), axis=1)
    np.testing.assert_allclose(o[0, :, 0], p @ v[0, :, 0], atol=1e-13)


def test_attention_rows_matches_full():
    q, k, v = rand_qkv(12, 2, 40, 33, 4, 2, 8)
    o, l = oracle.attention(q, k, v, 0.35, True, row_chunk=16)
    rows = [0, 3, 7, 20, 39]
    o_r, l_r = oracle.attention_rows(q, k, v, 0.35, True, 1, 3, rows)
    np.testing.assert_array_equal(np.isinf(l_r), np.isinf(l[1, 3, rows]))
    np.testing.assert_allclose(o_r, o[1, rows, 3], atol=1e-14)


def test_empty_inputs():
    q = np.zeros((1, 0, 2, 4))
    k = np.zeros((1, 5, 2, 4))
    o, l = oracle.attention(q, k, k, 1.0, True)
    assert o.shape == (1, 0, 2, 4) and l.shape == (1, 2, 0)
    q = np.ones((1, 3, 2, 4))
    k = np.zeros((1, 0, 2, 4))
    o, l = oracle.attention(q, k, k, 1.0, False)
    assert np.all(o == 0) and np.all(l == -np.inf)


def test_rejects_bad_gqa():
    with pytest.raises(ValueError):
        oracle.kv_head_of(0, 6, 4)


# --------------------------------------------------------------------------
# Planted mistakes: each must be caught by at least one pin above
# --------------------------------------------------------------------------

def _pins_fail(monkeypatch_fn):
    """Run a representative subset of the pins; True if any fails."""
    checks = [
        test_gqa_head_map_matches_printed_tables,
        lambda: test_zero_scores_give_prefix_means(5, 11, True),
        lambda: test_zero_scores_give_prefix_means(11, 5, True),
        lambda: test_single_key(),
        lambda: test_dominant_key_without_overflow(),
        lambda: test_two_keys_weights_are_sigmoids(),
        lambda: test_constant_v_returns_the_constant(5, 11, True),
        lambda: test_gqa_equals_mha_with_repeated_heads(),
        lambda: test_matches_scipy_softmax_and_logsumexp(7, 7, True),
    ]
    failed = False
    for c in checks:
        try:
            with np.errstate(all="ignore"):
                c()
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            failed = True
    return failed


def _mutant_rows(kind):
    def rows(q_rows, k_h, v_h, scale, vis):
        s = scale * (q_rows @ k_h.T)
        if kind == "no_scale":
            s = q_rows @ k_h.T
        s_masked = np.where(vis, s, -np.inf)
        any_vis = vis.any(axis=1)
        m = np.where(any_vis, s_masked.max(axis=1, initial=-np.inf), 0.0)
        if kind == "no_max":
            m = np.zeros_like(m)
        e = np.where(vis, np.exp(s_masked - m[:, None]), 0.0)
        l = e.sum(axis=1)
        safe_l = np.where(any_vis, l, 1.0)
        if kind == "v_transposed":
            o = (e @ v_h[::-1]) / safe_l[:, None]
        else:
            o = (e @ v_h) / safe_l[:, None]
        o[~any_vis] = 0.0
        lse = np.where(any_vis, (0.0 if kind == "lse_no_max" else m) + np.log(safe_l), -np.inf)
        return o, lse
    return rows


@pytest.mark.parametrize("kind", ["no_scale", "no_max", "v_transposed", "lse_no_max"])
def test_planted_arithmetic_mistakes_are_caught(monkeypatch, kind):
    monkeypatch.setattr(oa, "_rows_two_pass", _mutant_rows(kind))
    assert _pins_fail(None), kind


def test_planted_head_map_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(oa, "kv_head_of", lambda hq, Hq, Hkv: hq % Hkv)
    monkeypatch.setattr(oracle, "kv_head_of", lambda hq, Hq, Hkv: hq % Hkv)
    assert _pins_fail(None)


@pytest.mark.parametrize("kind", ["top_left", "off_by_one"])
def test_planted_mask_mistakes_are_caught(monkeypatch, kind):
    def vis(rows, Sq, Sk, causal):
        rows = np.asarray(rows, dtype=np.int64).reshape(-1)
        j = np.arange(Sk)[None, :]
        if not causal:
            return np.ones((rows.size, Sk), dtype=bool)
        if kind == "top_left":
            return j <= rows[:, None]
        return j < rows[:, None] + (Sk - Sq)
    monkeypatch.setattr(oa, "visibility", vis)
    assert _pins_fail(None)


# --------------------------------------------------------------------------
# Merging partial (O, LSE) over key shards
# --------------------------------------------------------------------------

@pytest.mark.parametrize("cuts", [(4,), (1, 6), (3, 5, 9)])
def test_merge_of_key_shards_equals_attention_over_all_keys(cuts):
    """Non-causal: attention over key shards [c_r, c_{r+1}) merged by LSE
    equals attention over every key."""
    B, Sq, Sk, Hq, Hkv, D = 2, 5, 11, 4, 2, 3
    q, k, v = rand_qkv(13, B, Sq, Sk, Hq, Hkv, D, sigma=1.5)
    o_full, l_full = oracle.attention(q, k, v, 0.6, causal=False)
    edges = [0, *cuts, Sk]
    parts = [oracle.attention(q, k[:, a:b], v[:, a:b], 0.6, causal=False) for a, b in zip(edges[:-1], edges[1:])]
    o, l = oracle.merge_partials(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(o, o_full, atol=1e-12)
    np.testing.assert_allclose(l, l_full, atol=1e-12)


def test_merge_with_causal_suffix_shard():
    """Causal, Sk >= Sq: keys [0, a) with a <= Sk - Sq + 1 are visible to every
    query (non-causal shard); keys [a, Sk) keep the bottom-right mask of their
    own lengths. Merging the two equals causal attention over all keys,
    including rows that see nothing in the second shard."""
    B, Sq, Sk, Hq, D = 1, 4, 9, 2, 3
    q, k, v = rand_qkv(14, B, Sq, Sk, Hq, Hq, D)
    o_full, l_full = oracle.attention(q, k, v, 0.9, causal=True)
    a = Sk - Sq + 1
    p0 = oracle.attention(q, k[:, :a], v[:, :a], 0.9, causal=False)
    p1 = oracle.attention(q, k[:, a:], v[:, a:], 0.9, causal=True)
    assert np.isinf(p1[1]).any()                     # row 0 sees no key of the suffix
    o, l = oracle.merge_partials(np.stack([p0[0], p1[0]]), np.stack([p0[1], p1[1]]))
    np.testing.assert_allclose(o, o_full, atol=1e-12)
    np.testing.assert_allclose(l, l_full, atol=1e-12)


def test_merge_all_empty_parts_and_single_part():
    o_parts = np.random.default_rng(15).standard_normal((3, 1, 2, 2, 4))
    lse = np.full((3, 1, 2, 2), -np.inf)
    o, l = oracle.merge_partials(o_parts, lse)
    assert np.all(o == 0) and np.all(l == -np.inf)
    lse1 = np.random.default_rng(16).standard_normal((1, 1, 2, 2))
    o1, l1 = oracle.merge_partials(o_parts[:1], lse1)
    np.testing.assert_allclose(o1, o_parts[0], atol=1e-15)
    np.testing.assert_allclose(l1, lse1[0], atol=1e-15)


def test_planted_merge_mistake_is_caught(monkeypatch):
    real = oa.merge_partials

    def no_rescale(o_parts, lse_parts):        # plain average of the parts
        o, l = real(o_parts, lse_parts)
        return np.asarray(o_parts).mean(axis=0), l
    monkeypatch.setattr(oracle, "merge_partials", no_rescale)
    with pytest.raises(AssertionError):
        test_merge_of_key_shards_equals_attention_over_all_keys((4,))
