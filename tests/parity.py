"""Shared parity harness: run the CUDA path through the C ABI binding and the
fp64 oracle on the same seeded inputs, and compare.

Tolerances (fixed for this operation): O max-abs <= 2e-2 and mean-abs <= 2e-3
for bf16/fp16 outputs; LSE max-abs <= 1e-3; rows that see no key must give
O == 0 and LSE == -inf on both sides.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from exact_attention_16_gb300 import api
from exact_attention_16_gb300.workloads import Workload, draw_inputs

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3


def run_gpu(q, k, v, scale, causal):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = api.fa_fwd(qd, kd, vd, scale=scale, causal=causal)
    status = api.fa_status()
    assert status == 0, api.fa_status_string(status)
    return o, lse


def compare(o_gpu, lse_gpu, o_ref, lse_ref):
    """o_gpu/o_ref: (..., D) arrays; lse_*: matching row arrays."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    assert np.all(np.isfinite(o_gpu)), "non-finite O"
    err = np.abs(o_gpu - o_ref)
    stats = {"o_max_abs": float(err.max()) if err.size else 0.0,
             "o_mean_abs": float(err.mean()) if err.size else 0.0}
    dead = ~np.isfinite(lse_ref)
    assert np.array_equal(dead, ~np.isfinite(lse_gpu)), "rows with no visible key differ"
    assert np.all(lse_gpu[dead] == -np.inf)
    if dead.any():
        assert np.all(o_gpu[dead] == 0.0)
    live = ~dead
    stats["lse_max_abs"] = float(np.abs(lse_gpu[live] - lse_ref[live]).max()) if live.any() else 0.0
    assert stats["o_max_abs"] <= O_MAX_ABS, stats
    assert stats["o_mean_abs"] <= O_MEAN_ABS, stats
    assert stats["lse_max_abs"] <= LSE_MAX_ABS, stats
    return stats


def check_full(w: Workload):
    """Every element against the oracle (sizes the oracle finishes quickly)."""
    q, k, v = draw_inputs(w)
    o, lse = run_gpu(q, k, v, w.scale, w.causal)
    o_ref, lse_ref = oracle.attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), w.scale, w.causal)
    # compare in (B, Hq, Sq, D) order so O rows line up with LSE entries
    o_gpu = o.float().cpu().numpy().transpose(0, 2, 1, 3)
    return compare(o_gpu, lse.cpu().numpy(), o_ref.transpose(0, 2, 1, 3), lse_ref)


def sample_rows(Sq, rng, n_random=64):
    rows = set(range(min(Sq, 130)))
    rows |= set(range(max(0, Sq - 130), Sq))
    mid = (Sq // 2) // 128 * 128
    rows |= set(range(max(0, mid - 2), min(Sq, mid + 130)))
    rows |= set(int(x) for x in rng.integers(0, Sq, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)


def check_sampled(w: Workload, heads=None, seed=0, all_rows=False):
    """Full-size launch; rows of a few (batch, head) pairs against the oracle
    (sampled rows, or every row of those heads with ``all_rows``)."""
    q, k, v = draw_inputs(w)
    o, lse = run_gpu(q, k, v, w.scale, w.causal)
    rng = np.random.default_rng(seed)
    if heads is None:
        heads = {(0, 0), (w.B - 1, w.Hq - 1), (int(rng.integers(w.B)), int(rng.integers(w.Hq))),
                 (int(rng.integers(w.B)), int(rng.integers(w.Hq)))}
    qf = q.float().numpy()
    kf = k.float().numpy()
    vf = v.float().numpy()
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for (b, hq) in sorted(heads):
        rows = np.arange(w.Sq) if all_rows else sample_rows(w.Sq, rng)
        ro, rl = oracle.attention_rows(qf, kf, vf, w.scale, w.causal, b, hq, rows)
        idx = torch.from_numpy(rows).cuda()
        got_o.append(o[b, :, hq, :].index_select(0, idx).float().cpu().numpy())
        got_l.append(lse[b, hq].index_select(0, idx).cpu().numpy())
        ref_o.append(ro)
        ref_l.append(rl)
    return compare(np.concatenate(got_o), np.concatenate(got_l), np.concatenate(ref_o), np.concatenate(ref_l))
