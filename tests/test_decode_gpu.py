"""fa_fwd_decode (split-KV over the keys, per-split partials merged) against
the fp64 oracle, every element, over decode-like shapes (one or a few query
positions, GQA groups packed into one tile) and small prefill shapes (several
row tiles of floor(128 / G) positions), causal and not, ragged key counts,
one split, automatic splits and explicit split counts."""

import pytest

torch = pytest.importorskip("torch")

from exact_attention_16_gb300 import api  # noqa: E402
from exact_attention_16_gb300.workloads import Workload, draw_inputs  # noqa: E402

from parity import compare  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def W(B, Sq, Sk, Hq, Hkv, D, dtype="bf16", causal=True, sigma=1.0, seed=31):
    return Workload("dec", B, Sq, Sk, Hq, Hkv, D, dtype, causal, sigma, 1.0, seed)


CASES = [
    (W(2, 1, 3000, 32, 4, 128), 0),              # GQA 8, one query, automatic splits
    (W(2, 1, 3000, 32, 4, 128, causal=False), 5),
    (W(1, 4, 1037, 16, 2, 128), 0),              # 8 heads x 4 positions = 32 rows
    (W(1, 16, 700, 64, 8, 128), 3),              # 8 x 16 = 128 rows (a full tile)
    (W(3, 1, 513, 8, 8, 64, "fp16"), 0),         # MHA decode, D = 64
    (W(1, 2, 100, 4, 1, 128), 0),                # fewer keys than one tile
    (W(1, 8, 5, 4, 2, 128), 1),                  # Sq > Sk, causal: first rows see nothing
    (W(2, 1, 4096, 16, 8, 128, sigma=2.0), 1),   # one split writes O directly
    (W(1, 1, 2048, 32, 4, 128), 16),             # as many splits as key tiles
    # prefill-sized query counts: several row tiles of floor(128 / G) positions
    (W(1, 1280, 1536, 16, 16, 128, "fp16"), 0),  # MHA, 128 positions per tile, offset 256
    (W(2, 300, 333, 8, 2, 128), 3),              # G = 4: 32 positions per tile, ragged
    (W(1, 257, 129, 6, 2, 64, "fp16"), 0),       # G = 3: 42 positions per tile, Sq > Sk
    (W(1, 640, 640, 4, 4, 128, causal=False), 2),
    (W(2, 1, 2000, 16, 2, 256), 0),              # D = 256 decode, splits merged
    (W(1, 70, 900, 8, 4, 256, "fp16"), 4),
    (W(2, 1, 1500, 16, 2, 96), 0),               # padded head dims through the split path
    (W(1, 3, 700, 8, 8, 32, "fp16"), 3),
    (W(1, 1, 600, 4, 4, 160), 2),
    (W(2, 3, 1000, 64, 1, 128), 0),              # MQA, G = 64: 2 positions per tile
    (W(1, 1, 3000, 128, 1, 128), 3),             # G = 128: one position fills a tile
]


@pytest.mark.parametrize("w,splits", CASES, ids=lambda x: str(x) if isinstance(x, int) else
                         f"B{x.B}_Sq{x.Sq}_Sk{x.Sk}_H{x.Hq}-{x.Hkv}_D{x.D}_{x.dtype}_{'c' if x.causal else 'n'}")
def test_decode_every_element(w, splits):
    import oracle
    q, k, v = draw_inputs(w)
    o, lse = api.fa_fwd_decode(q.cuda(), k.cuda(), v.cuda(), scale=w.scale, causal=w.causal, num_splits=splits)
    assert api.fa_status() == 0
    o_ref, l_ref = oracle.attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), w.scale, w.causal)
    compare(o.float().cpu().numpy().transpose(0, 2, 1, 3), lse.cpu().numpy(), o_ref.transpose(0, 2, 1, 3), l_ref)


def test_decode_matches_prefill_kernel():
    """Same inputs through fa_fwd and fa_fwd_decode: both within tolerance of
    each other (different key grouping, same arithmetic)."""
    w = W(2, 2, 2500, 32, 4, 128)
    q, k, v = (t.cuda() for t in draw_inputs(w))
    o1, l1 = api.fa_fwd(q, k, v, causal=True)
    o2, l2 = api.fa_fwd_decode(q, k, v, causal=True)
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_decode_rejects_small_workspace():
    w = W(1, 1, 2048, 32, 4, 128)
    q, k, v = (t.cuda() for t in draw_inputs(w))
    need = api.fa_decode_workspace_size(1, 1, 2048, 32, 4, 128, 4)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.FAError):
        api.fa_fwd_decode(q, k, v, causal=True, num_splits=4, workspace=small)


def test_binding_rejects_result_buffers_that_do_not_fit():
    """The kernels write every element of O and LSE, so the binding refuses a
    caller buffer of another shape, dtype or device (and a workspace in host
    memory) before anything is launched; buffers that fit are used as given."""
    w = W(2, 1, 1000, 16, 4, 128)
    q, k, v = (t.cuda() for t in draw_inputs(w))
    few_heads = torch.empty(2, 1, 8, 128, dtype=q.dtype, device="cuda")
    with pytest.raises(ValueError):
        api.fa_fwd_decode(q, k, v, out=few_heads)
    with pytest.raises(ValueError):
        api.fa_fwd_decode(q, k, v, lse=torch.empty(2, 16, 2, device="cuda"))
    with pytest.raises(ValueError):
        api.fa_fwd_decode(q, k, v, num_splits=4, workspace=torch.empty(1 << 20, dtype=torch.uint8))
    with pytest.raises(ValueError):
        api.fa_fwd_decode_noalloc(q, k, v, out=few_heads)
    with pytest.raises(ValueError):
        api.fa_fwd_decode_noalloc(q, k, v, lse=torch.empty(2, 16, 1, dtype=torch.float16, device="cuda"))
    with pytest.raises(ValueError):
        api.fa_fwd_decode_noalloc(q, k[:, :, :2].contiguous(), v)
    parts_o = torch.zeros(3, 2, 1, 16, 128, dtype=q.dtype, device="cuda")
    parts_l = torch.zeros(3, 2, 16, 1, device="cuda")
    with pytest.raises(ValueError):
        api.fa_merge(parts_o, parts_l, out=few_heads)
    with pytest.raises(ValueError):
        api.fa_merge(parts_o, parts_l, lse=torch.empty(2, 16, 1, dtype=torch.float64, device="cuda"))
    out = torch.empty_like(q)
    lse = torch.empty(2, 16, 1, device="cuda")
    o, l = api.fa_merge(parts_o, parts_l, out=out, lse=lse)
    torch.cuda.synchronize()
    assert o is out and l is lse
    assert torch.all(out == 0) and torch.allclose(lse, torch.full_like(lse, float(torch.log(torch.tensor(3.0)))))
