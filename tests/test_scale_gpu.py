"""Any finite softmax scale, and the plain contiguous entry point.

The scale is a free argument of softmax(scale * Q K^T + M) ("MiniPaged-Qwen:
Qwen3 Prefill FlashAttention" section 1; the CuTe-DSL example
"ampere/flash_attention_v2.py" passes ``softmax_scale`` explicitly), so zero
and negative scales are valid. Each case runs through every kernel: row-tile
pairs, key-split items, the one-tile kernel (D = 256) and decode splits with
their merge, against the fp64 oracle. Scale 0 is also checked against its
closed form (prefix means, LSE = ln #visible), and a negative scale against
the kernel's own result on negated queries, which must be identical bit for
bit (scale * (q . k) = (-scale) * ((-q) . k), and both sides round the same
fp32 values).

``fa_fwd`` (contiguous tensors) is called here through ctypes directly; the
Python binding routes every call through ``fa_fwd_strided``.
"""

import ctypes
import math

import numpy as np
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


def W(B, Sq, Sk, Hq, Hkv, D, dtype="bf16", causal=False, sigma=1.0, seed=7):
    return Workload("case", B, Sq, Sk, Hq, Hkv, D, dtype, causal, sigma, 1.0, seed)


# (workload, forced schedule of fa_fwd or -1, entry point)
CASES = [
    (W(2, 333, 517, 8, 2, 128, causal=True, seed=51), 0, "fwd"),             # row-tile pairs, head pairs
    (W(1, 300, 257, 6, 2, 128, "fp16", causal=True, seed=52), 0, "fwd"),     # pairs of row tiles, Sq > Sk
    (W(1, 300, 300, 4, 4, 64, "fp16", causal=False, seed=53), 1, "fwd"),     # key-split items
    (W(1, 257, 700, 4, 2, 128, causal=True, seed=54), 1, "fwd"),             # key-split, offset mask
    (W(1, 200, 333, 4, 1, 256, causal=True, seed=55), -1, "fwd"),            # one-tile kernel
    (W(4, 1, 3000, 16, 4, 128, causal=True, seed=56), -1, "decode"),         # decode splits + merge
    (W(2, 3, 1500, 8, 8, 64, causal=False, seed=57), -1, "decode"),
]
CASE_IDS = ["pairs_heads", "pairs_rows_sq_gt_sk", "keysplit_d64", "keysplit_offset", "d256", "decode_d128",
            "decode_d64"]


def _run(w, mode, entry, q, k, v, scale):
    assert api.fa_debug_set_schedule(mode) == api.FA_OK
    try:
        if entry == "fwd":
            o, lse = api.fa_fwd(q, k, v, scale=scale, causal=w.causal)
        else:
            o, lse = api.fa_fwd_decode(q, k, v, scale=scale, causal=w.causal, num_splits=5)
        torch.cuda.synchronize()
    finally:
        api.fa_debug_set_schedule(-1)
    assert api.fa_status() == 0
    return o, lse


def _oracle_compare(q, k, v, o, lse, scale, causal):
    import oracle
    o_ref, l_ref = oracle.attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), scale, causal)
    return compare(o.float().cpu().numpy().transpose(0, 2, 1, 3), lse.cpu().numpy(), o_ref.transpose(0, 2, 1, 3),
                   l_ref)


@pytest.mark.parametrize("scale_kind", ["zero", "minus_inv_sqrt_d", "minus3"])
@pytest.mark.parametrize("case", range(len(CASES)), ids=CASE_IDS)
def test_zero_and_negative_scales_match_the_oracle(case, scale_kind):
    w, mode, entry = CASES[case]
    scale = {"zero": 0.0, "minus_inv_sqrt_d": -1.0 / math.sqrt(w.D), "minus3": -3.0}[scale_kind]
    q, k, v = draw_inputs(w)
    o, lse = _run(w, mode, entry, q.cuda(), k.cuda(), v.cuda(), scale)
    _oracle_compare(q, k, v, o, lse, scale, w.causal)


@pytest.mark.parametrize("case", range(len(CASES)), ids=CASE_IDS)
def test_zero_scale_gives_prefix_means(case):
    """Closed form, independent of the oracle: with scale 0 every visible key
    has weight 1, so O_i is the mean of the v rows row i sees and LSE_i is
    ln of their number; a row that sees none gets O = 0, LSE = -inf."""
    w, mode, entry = CASES[case]
    q, k, v = draw_inputs(w)
    o, lse = _run(w, mode, entry, q.cuda(), k.cuda(), v.cuda(), 0.0)
    G = w.Hq // w.Hkv
    vf = v.double().numpy()
    csum = np.concatenate([np.zeros((w.B, 1, w.Hkv, w.D)), np.cumsum(vf, axis=1)], axis=1)
    i = np.arange(w.Sq)
    cnt = np.clip(i + w.Sk - w.Sq + 1, 0, w.Sk) if w.causal else np.full(w.Sq, w.Sk)
    og = o.double().cpu().numpy()
    lg = lse.double().cpu().numpy()
    for b in range(w.B):
        for hq in range(w.Hq):
            means = csum[b, cnt, hq // G] / np.maximum(cnt, 1)[:, None]
            means[cnt == 0] = 0.0
            err = np.abs(og[b, :, hq] - means)
            assert err.max() <= 2e-2 and err.mean() <= 2e-3, (b, hq, err.max(), err.mean())
            with np.errstate(divide="ignore"):
                want = np.where(cnt > 0, np.log(np.maximum(cnt, 1)), -np.inf)
            assert np.array_equal(np.isfinite(lg[b, hq]), cnt > 0)
            live = cnt > 0
            assert np.abs(lg[b, hq][live] - want[live]).max() <= 1e-5


@pytest.mark.parametrize("case", range(len(CASES)), ids=CASE_IDS)
def test_negative_scale_equals_negated_queries_bitwise(case):
    w, mode, entry = CASES[case]
    q, k, v = (t.cuda() for t in draw_inputs(w))
    c = 1.0 / math.sqrt(w.D)
    o1, l1 = _run(w, mode, entry, q, k, v, -c)
    o2, l2 = _run(w, mode, entry, -q, k, v, c)
    assert torch.equal(o1, o2)
    assert torch.equal(l1, l2)


@pytest.mark.parametrize("wl", [W(2, 300, 257, 8, 2, 128, causal=True, seed=61),
                                W(1, 200, 200, 4, 4, 64, "fp16", causal=False, seed=62),
                                W(1, 150, 260, 4, 2, 256, causal=True, seed=63),
                                W(1, 129, 129, 4, 2, 96, causal=True, seed=64)],
                         ids=["d128_causal", "d64_fp16", "d256", "d96_padded"])
def test_plain_fa_fwd_entry_point(wl):
    """The contiguous entry point itself, through ctypes with device tensors."""
    q, k, v = draw_inputs(wl)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((wl.B, wl.Hq, wl.Sq), float("nan"), dtype=torch.float32, device="cuda")
    code = api.FA_DTYPE_BF16 if wl.dtype == "bf16" else api.FA_DTYPE_FP16
    rc = api.lib().fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(), wl.B, wl.Sq,
                          wl.Sk, wl.Hq, wl.Hkv, wl.D, ctypes.c_float(wl.scale), int(wl.causal), code,
                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == api.FA_OK
    torch.cuda.synchronize()
    assert api.fa_status() == 0
    _oracle_compare(q, k, v, o, lse, wl.scale, wl.causal)
