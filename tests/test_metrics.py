"""FLOP accounting against a direct count of the oracle's visibility matrix."""

import numpy as np
import pytest

import oracle
from exact_attention_16_gb300 import metrics
from exact_attention_16_gb300.workloads import WORKLOADS


@pytest.mark.parametrize("Sq,Sk", [(1, 1), (7, 7), (5, 11), (11, 5), (128, 300), (300, 128), (1, 77), (77, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_unmasked_pairs_matches_visibility_count(Sq, Sk, causal):
    vis = oracle.visibility(np.arange(Sq), Sq, Sk, causal)
    assert metrics.unmasked_pairs(Sq, Sk, causal) == int(vis.sum())
    assert sum(metrics.visible_keys(i, Sq, Sk, causal) for i in range(Sq)) == int(vis.sum())


def test_workload_flops_match_the_documented_values():
    got = [metrics.flops(w.B, w.Sq, w.Sk, w.Hq, w.D, w.causal) for w in WORKLOADS]
    ref = [8.389e6, 9.400e9, 5.499e11, 5.498e11, 2.199e12]
    for g, r in zip(got, ref):
        assert abs(g - r) / r < 1e-3
