"""fa_fwd_host: host tensors in, host tensors out, with the copies and the
kernels pipelined per chunk of batches or KV heads. Checked against the fp64
oracle, and bit for bit against fa_fwd on the same inputs under each forced
work decomposition (a chunk is a strided view of the same computation, so
every row gets the same arithmetic)."""

import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_attention_16_gb300 import api  # noqa: E402
from exact_attention_16_gb300.workloads import Workload, draw_inputs  # noqa: E402

from parity import compare  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def W(B, Sq, Sk, Hq, Hkv, D, dtype="bf16", causal=True, seed=31):
    return Workload("case", B, Sq, Sk, Hq, Hkv, D, dtype, causal, 1.0, 1.0, seed)


# Small problems (under 48 MiB of copies) run as one chunk.
CASES = [
    W(1, 300, 257, 8, 4, 128),
    W(1, 520, 600, 6, 3, 64, "fp16"),           # G = 2
    W(3, 257, 300, 8, 2, 128),
    W(5, 128, 384, 4, 4, 128, causal=False),
    W(2, 200, 211, 4, 2, 256),                  # D = 256 (one-tile kernel)
    W(1, 129, 1000, 32, 4, 96, causal=False),   # padded head dimension
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: f"B{w.B}_Sq{w.Sq}_Sk{w.Sk}_H{w.Hq}-{w.Hkv}_D{w.D}")
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_entry_matches_oracle(w, pinned):
    q, k, v = draw_inputs(w)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o, lse = api.fa_fwd_host(q, k, v, scale=w.scale, causal=w.causal)
    assert api.fa_status() == 0
    assert not o.is_cuda and not lse.is_cuda
    o_ref, l_ref = oracle.attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), w.scale, w.causal)
    compare(o.float().numpy().transpose(0, 2, 1, 3), lse.numpy(), o_ref.transpose(0, 2, 1, 3), l_ref)


@pytest.mark.parametrize("mode", [0, 1], ids=["pairs", "keysplit"])
def test_host_entry_equals_device_entry(mode):
    w = W(2, 700, 700, 8, 2, 128, seed=32)
    q, k, v = (t.pin_memory() for t in draw_inputs(w))
    assert api.fa_debug_set_schedule(mode) == api.FA_OK
    try:
        o_h, l_h = api.fa_fwd_host(q, k, v, causal=True)
        o_d, l_d = api.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
        torch.cuda.synchronize()
    finally:
        api.fa_debug_set_schedule(-1)
    assert api.fa_status() == 0
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


def test_host_entry_without_lse_and_into_given_buffers():
    w = W(1, 256, 256, 4, 2, 128, seed=33)
    q, k, v = (t.pin_memory() for t in draw_inputs(w))
    out = torch.full(q.shape, float("nan"), dtype=q.dtype).pin_memory()
    need = api.fa_fwd_host_workspace_size(w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o, lse = api.fa_fwd_host(q, k, v, causal=True, out=out, return_lse=False, workspace=ws)
    assert lse is None and o.data_ptr() == out.data_ptr()
    o_d, _ = api.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert not torch.isnan(o.float()).any()
    o_ref, l_ref = oracle.attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), w.scale, True)
    compare(o.float().numpy().transpose(0, 2, 1, 3), l_ref, o_ref.transpose(0, 2, 1, 3), l_ref)


def test_host_entry_async_on_a_side_stream():
    w = W(2, 384, 384, 8, 8, 64, seed=34)
    q, k, v = (t.pin_memory() for t in draw_inputs(w))
    s = torch.cuda.Stream()
    o, lse = api.fa_fwd_host(q, k, v, causal=True, stream=s, synchronize=False)
    s.synchronize()
    o_ref, l_ref = oracle.attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), w.scale, True)
    compare(o.float().numpy().transpose(0, 2, 1, 3), lse.numpy(), o_ref.transpose(0, 2, 1, 3), l_ref)


def test_host_entry_no_keys():
    q = torch.randn(1, 5, 2, 128).to(torch.bfloat16).pin_memory()
    k = torch.empty(1, 0, 2, 128, dtype=torch.bfloat16).pin_memory()
    o, lse = api.fa_fwd_host(q, k, k.clone(), causal=True)
    assert torch.all(o == 0) and torch.all(lse == float("-inf"))


# Problems of 48 MiB of copies or more run as several chunks: (B = 1) ranges
# of KV heads (four, and three uneven ones), two row halves of one KV head
# with the keys each newly needs, a first row half that sees no key at all
# (Sq > Sk, causal); (B >= 2) ranges of batches alone and times two or four
# ranges of KV heads; and a mask-free problem.
LARGE = [
    W(1, 8192, 8192, 32, 4, 128, seed=35),
    W(1, 5000, 2000, 32, 8, 128, seed=37),
    W(1, 16384, 16384, 8, 1, 128, seed=39),
    W(1, 12000, 4000, 16, 1, 128, seed=40),
    W(4, 2048, 2048, 16, 8, 128, seed=36),
    W(4, 4096, 4096, 32, 8, 128, seed=42),              # batches x two KV-head halves
    W(2, 4096, 4096, 16, 8, 128, seed=43),              # 2 batches x 2 KV-head ranges
    W(3, 4096, 4096, 16, 8, 128, seed=44),              # 3 batches x 2 KV-head ranges
    W(2, 4096, 1024, 16, 4, 128, causal=False, seed=38),
]


@pytest.mark.parametrize("w", LARGE, ids=lambda w: f"B{w.B}_S{w.Sq}_H{w.Hq}-{w.Hkv}")
def test_host_entry_in_several_chunks(w):
    import numpy as np
    q, k, v = (t.pin_memory() for t in draw_inputs(w))
    assert api.fa_debug_set_schedule(0) == api.FA_OK
    try:
        o_h, l_h = api.fa_fwd_host(q, k, v, causal=w.causal)
        o_d, l_d = api.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=w.causal)
        torch.cuda.synchronize()
    finally:
        api.fa_debug_set_schedule(-1)
    assert api.fa_status() == 0
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())
    # sampled rows of the first and last head of every batch against the oracle
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(0, 130), np.arange(w.Sq - 130, w.Sq), rng.integers(0, w.Sq, 64)]))
    qf, kf, vf = q.float().numpy(), k.float().numpy(), v.float().numpy()
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for b in range(w.B):
        for hq in (0, w.Hq - 1):
            ro, rl = oracle.attention_rows(qf, kf, vf, w.scale, w.causal, b, hq, rows)
            got_o.append(o_h[b, rows, hq].float().numpy())
            got_l.append(l_h[b, hq, rows].numpy())
            ref_o.append(ro)
            ref_l.append(rl)
    compare(np.concatenate(got_o), np.concatenate(got_l), np.concatenate(ref_o), np.concatenate(ref_l))
