"""The seeded workload generator: determinism, shapes, dtype rounding."""

import numpy as np
import torch

from exact_attention_16_gb300 import workloads as wl


def test_five_workloads_match_their_descriptions():
    names = [w.name for w in wl.WORKLOADS]
    assert len(names) == 5 and len(set(names)) == 5
    c2 = wl.WORKLOADS[1]
    assert (c2.Sq, c2.Sk, c2.Hq, c2.Hkv, c2.D, c2.dtype, c2.causal) == (1280, 1536, 16, 16, 128, "fp16", True)
    c4 = wl.WORKLOADS[3]
    assert c4.sigma_qk == 2.0 and c4.sigma_v == 1.0
    for w in wl.WORKLOADS:
        assert w.Hq % w.Hkv == 0
        assert abs(w.scale - w.D ** -0.5) < 1e-15


def test_generator_is_deterministic_and_seed_dependent():
    w = wl.WORKLOADS[0]
    a = wl.draw_numpy(w)
    b = wl.draw_numpy(w)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    c = wl.draw_numpy(w.with_sizes(seed=w.seed + 1))
    assert not np.array_equal(a[0], c[0])


def test_generator_stream_is_pinned():
    # PCG64 streams are stable across platforms; pin the first draws.
    q, k, v = wl.draw_numpy(wl.WORKLOADS[0].with_sizes(Sq=1, Sk=1, Hq=1, Hkv=1, D=2))
    ref = np.random.Generator(np.random.PCG64(1000)).standard_normal(6, dtype=np.float32)
    np.testing.assert_array_equal(np.concatenate([q.ravel(), k.ravel(), v.ravel()]), ref)


def test_inputs_are_rounded_to_dtype():
    w = wl.WORKLOADS[0].with_sizes(Sq=8, Sk=8)
    q, k, v = wl.draw_inputs(w)
    assert q.dtype == torch.bfloat16 and q.shape == (1, 8, 2, 64)
    qf, _, _ = wl.draw_numpy(w)
    assert torch.equal(q, torch.from_numpy(qf).to(torch.bfloat16))
    w2 = wl.WORKLOADS[1].with_sizes(Sq=4, Sk=4, Hq=2, Hkv=2)
    q2, _, _ = wl.draw_inputs(w2)
    assert q2.dtype == torch.float16
