"""Both work decompositions of fa_fwd, each forced through the test hook,
against the fp64 oracle on every element (and on sampled rows at full size).

Row-tile pairs: a CTA item is two 128-row query tiles sharing every K/V tile.
Key-split: an item is one query tile whose even and odd key tiles run in the
CTA's two slots, combined before the store. The cases cover one key tile
(slot 1 idle), odd and even tile counts, row tiles that see no key, ragged
tails, GQA group sizes 1/2/3/4/8, fp16 and bf16, padded head dimensions,
strided views, several persistent rounds per CTA and sharp softmax rows.
"""

import pytest

torch = pytest.importorskip("torch")

from exact_attention_16_gb300 import api  # noqa: E402
from exact_attention_16_gb300.workloads import WORKLOADS, Workload, draw_inputs  # noqa: E402

from parity import check_full, check_sampled  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.fixture(params=[0, 1], ids=["pairs", "keysplit"])
def mode(request):
    assert api.fa_debug_set_schedule(request.param) == api.FA_OK
    yield request.param
    api.fa_debug_set_schedule(-1)


def W(B, Sq, Sk, Hq, Hkv, D, dtype="bf16", causal=False, sigma=1.0, seed=21):
    return Workload("case", B, Sq, Sk, Hq, Hkv, D, dtype, causal, sigma, 1.0, seed)


CASES = [
    W(1, 128, 128, 2, 2, 128),                          # one key tile: slot 1 idle
    W(1, 128, 256, 2, 2, 128),                          # two key tiles: one per slot
    W(1, 128, 384, 2, 1, 64),                           # three: slot 0 runs two
    W(1, 400, 100, 2, 2, 128, causal=True),             # two row tiles see no key at all
    W(1, 300, 257, 4, 4, 128, causal=True),             # Sq > Sk: first rows see nothing
    W(2, 257, 300, 8, 2, 128, "fp16", causal=True),     # Sk > Sq: offset 43
    W(1, 520, 520, 6, 2, 64, "fp16", causal=True),      # G = 3
    W(1, 640, 384, 4, 1, 128, causal=True),             # G = 4
    W(1, 129, 1000, 32, 4, 128),                        # G = 8
    W(1, 2048, 2048, 4, 2, 128, causal=True, sigma=2.0),
    W(1, 1000, 1000, 4, 1, 128, "fp16", causal=True, sigma=2.0),
    W(3, 700, 1300, 16, 4, 96, causal=True),            # D 96 on the 128 tile
    W(1, 333, 555, 4, 2, 32, "fp16", causal=True),      # D 32 on the 64 tile
    W(2, 1024, 1024, 48, 8, 128, causal=True),          # several items per CTA
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: f"B{w.B}_Sq{w.Sq}_Sk{w.Sk}_H{w.Hq}-{w.Hkv}_D{w.D}_{w.dtype}_{'c' if w.causal else 'n'}")
def test_every_element(w, mode):
    check_full(w)


def test_short_causal_mha_workload_every_element(mode):
    check_full(WORKLOADS[1])


@pytest.mark.parametrize("w", [WORKLOADS[2], WORKLOADS[4]], ids=lambda w: w.name)
def test_key_split_at_full_size_sampled_rows(w):
    assert api.fa_debug_set_schedule(1) == api.FA_OK
    try:
        check_sampled(w, heads={(0, 0), (w.B - 1, w.Hq - 1), (0, w.Hq // 2 + 1)})
    finally:
        api.fa_debug_set_schedule(-1)


def test_strided_bhsd_views(mode):
    w = W(2, 300, 333, 8, 2, 128, causal=True, seed=22)
    q, k, v = draw_inputs(w)
    qb, kb, vb = (t.transpose(1, 2).contiguous().cuda() for t in (q, k, v))
    o_store = torch.full((w.B, w.Hq, w.Sq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    o, lse = api.fa_fwd(qb.transpose(1, 2), kb.transpose(1, 2), vb.transpose(1, 2), scale=w.scale, causal=True,
                        out=o_store.transpose(1, 2))
    assert api.fa_status() == 0
    import oracle
    from parity import compare
    o_ref, l_ref = oracle.attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), w.scale, True)
    compare(o.float().cpu().numpy().transpose(0, 2, 1, 3), lse.cpu().numpy(), o_ref.transpose(0, 2, 1, 3), l_ref)


def test_both_schedules_agree_closely():
    """Same inputs through both decompositions: they differ only in the order
    of fp32 sums and in where P is rounded against which maximum."""
    w = W(1, 1280, 1536, 16, 16, 128, "fp16", causal=True, seed=23)
    q, k, v = (t.cuda() for t in draw_inputs(w))
    out = {}
    try:
        for m in (0, 1):
            api.fa_debug_set_schedule(m)
            out[m] = api.fa_fwd(q, k, v, causal=True)
            assert api.fa_status() == 0
    finally:
        api.fa_debug_set_schedule(-1)
    (o0, l0), (o1, l1) = out[0], out[1]
    assert (o0.float() - o1.float()).abs().max().item() <= 1e-2
    assert (l0 - l1).abs().max().item() <= 1e-4
