"""fa_merge (partial (O, LSE) over disjoint key sets) against the oracle:
element parity on random partial states, and context-parallel attention
(fa_fwd on key shards, then fa_merge) against attention over all keys."""

import numpy as np
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


def _bshd_to_bhsd(x):
    return x.transpose(0, 2, 1, 3)


@pytest.mark.parametrize("dt,n,D", [(torch.bfloat16, 3, 128), (torch.float16, 5, 64), (torch.bfloat16, 1, 256)])
def test_merge_random_partials(dt, n, D):
    g = torch.Generator().manual_seed(20 + n)
    B, Sq, Hq = 2, 77, 6
    o_parts = (torch.randn(n, B, Sq, Hq, D, generator=g) * 2).to(dt)
    lse_parts = torch.randn(n, B, Hq, Sq, generator=g) * 3
    lse_parts[0, 0, 0, :5] = float("-inf")                 # some parts hold no key
    lse_parts[:, 1, 2, 3] = float("-inf")                  # a row where no part does
    o, lse = api.fa_merge(o_parts.cuda(), lse_parts.cuda())
    assert api.fa_status() == 0
    o_ref, l_ref = oracle.merge_partials(o_parts.float().numpy(), lse_parts.numpy())
    compare(_bshd_to_bhsd(o.float().cpu().numpy()), lse.cpu().numpy(), _bshd_to_bhsd(o_ref), l_ref)


def test_context_parallel_noncausal_three_shards():
    w = Workload("cp", 1, 640, 1000, 8, 2, 128, "bf16", False, 1.0, 1.0, 21)
    q, k, v = draw_inputs(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    edges = [0, 300, 301, 1000]                              # includes a one-key shard
    parts = [api.fa_fwd(qd, kd[:, a:b].contiguous(), vd[:, a:b].contiguous(), scale=w.scale)
             for a, b in zip(edges[:-1], edges[1:])]
    o, lse = api.fa_merge(torch.stack([p[0] for p in parts]).contiguous(),
                          torch.stack([p[1] for p in parts]).contiguous())
    assert api.fa_status() == 0
    o_ref, l_ref = oracle.attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), w.scale, False)
    compare(_bshd_to_bhsd(o.float().cpu().numpy()), lse.cpu().numpy(), _bshd_to_bhsd(o_ref), l_ref)


def test_context_parallel_causal_prefix_and_suffix():
    """Keys [0, a) with a = Sk - Sq + 1 are visible to every query; keys
    [a, Sk) keep the bottom-right causal mask of their own length."""
    w = Workload("cp", 2, 384, 1024, 4, 4, 128, "fp16", True, 1.0, 1.0, 22)
    q, k, v = draw_inputs(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    a = w.Sk - w.Sq + 1
    p0 = api.fa_fwd(qd, kd[:, :a].contiguous(), vd[:, :a].contiguous(), scale=w.scale, causal=False)
    p1 = api.fa_fwd(qd, kd[:, a:].contiguous(), vd[:, a:].contiguous(), scale=w.scale, causal=True)
    o, lse = api.fa_merge(torch.stack([p0[0], p1[0]]).contiguous(), torch.stack([p0[1], p1[1]]).contiguous())
    assert api.fa_status() == 0
    o_ref, l_ref = oracle.attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), w.scale, True)
    compare(_bshd_to_bhsd(o.float().cpu().numpy()), lse.cpu().numpy(), _bshd_to_bhsd(o_ref), l_ref)
