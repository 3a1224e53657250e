"""Shared parity harness: run the CUDA path through the C ABI binding and the
fp64 oracle on the same seeded inputs, and compare.

Tolerances (fixed for this operation): O max-abs <= 2e-2 and mean-abs <= 2e-3
for bf16/fp16 outputs; LSE max-abs <= 1e-3; rows that see no key must give
O == 0 and LSE == -inf on both sides.
"""

from __future__ import annotations

import json
import multiprocessing as mp
import os

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


# ---------------------------------------------------------------- every element at full size
def _head_stats(task):
    """One (batch, query head) of a full-size launch against the oracle, in a
    worker process: returns (max |dO|, sum |dO|, #O elements, max |dLSE| on
    live rows, #dead rows). The dead-row rules of :func:`compare` are checked
    here too (rows that see no key: O == 0 and LSE == -inf on both sides)."""
    q_h, k_h, v_h, o_gpu, lse_gpu, scale, causal = task
    import oracle as _oracle

    # (1, S, 1, D) views: one head against its KV head, the oracle's own definition
    o_ref, lse_ref = _oracle.attention(q_h[None, :, None, :], k_h[None, :, None, :], v_h[None, :, None, :],
                                       scale, causal)
    o_ref = o_ref[0, :, 0, :]
    lse_ref = lse_ref[0, 0]
    o_gpu = o_gpu.astype(np.float64)
    lse_gpu = lse_gpu.astype(np.float64)
    if not np.all(np.isfinite(o_gpu)):
        raise AssertionError("non-finite O")
    dead = ~np.isfinite(lse_ref)
    if not np.array_equal(dead, ~np.isfinite(lse_gpu)):
        raise AssertionError("rows with no visible key differ")
    if dead.any() and not (np.all(lse_gpu[dead] == -np.inf) and np.all(o_gpu[dead] == 0.0)):
        raise AssertionError("a row with no visible key is not O = 0, LSE = -inf")
    err = np.abs(o_gpu - o_ref)
    live = ~dead
    lse_err = float(np.abs(lse_gpu[live] - lse_ref[live]).max()) if live.any() else 0.0
    return float(err.max()), float(err.sum()), int(err.size), lse_err, int(dead.sum())


def check_every_element_pooled(w: Workload, o, lse, q, k, v, workers=None):
    """Every element of a (possibly full-size) launch against the oracle: the
    oracle runs head by head in a pool of spawned processes (one BLAS thread
    each), and the statistics over all heads are checked against the
    tolerances. Returns the statistics (max-abs and mean-abs O error, LSE
    max-abs, dead rows)."""
    import oracle as _oracle

    qf = q.float().numpy()
    kf = k.float().numpy()
    vf = v.float().numpy()
    og = o.float().cpu().numpy()
    lg = lse.cpu().numpy()
    tasks = []
    for b in range(w.B):
        for hq in range(w.Hq):
            kvh = _oracle.kv_head_of(hq, w.Hq, w.Hkv)
            tasks.append((np.ascontiguousarray(qf[b, :, hq, :]), np.ascontiguousarray(kf[b, :, kvh, :]),
                          np.ascontiguousarray(vf[b, :, kvh, :]), np.ascontiguousarray(og[b, :, hq, :]),
                          np.ascontiguousarray(lg[b, hq]), w.scale, w.causal))
    workers = workers or max(1, min(len(tasks), os.cpu_count() or 1))
    saved = {v_: os.environ.get(v_) for v_ in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for v_ in saved:
        os.environ[v_] = "1"
    try:
        with mp.get_context("spawn").Pool(workers) as pool:
            res = pool.map(_head_stats, tasks, chunksize=1)
    finally:
        for v_, val in saved.items():
            if val is None:
                os.environ.pop(v_, None)
            else:
                os.environ[v_] = val
    n = sum(r[2] for r in res)
    stats = {"workload": w.name, "o_max_abs": max(r[0] for r in res), "o_mean_abs": sum(r[1] for r in res) / n,
             "lse_max_abs": max(r[3] for r in res), "elements": n, "rows": w.B * w.Hq * w.Sq,
             "dead_rows": sum(r[4] for r in res)}
    report = os.environ.get("FA_PARITY_REPORT")
    if report:
        with open(report, "a") as f:
            f.write(json.dumps(stats) + "\n")
    print(json.dumps(stats))
    assert stats["o_max_abs"] <= O_MAX_ABS, stats
    assert stats["o_mean_abs"] <= O_MEAN_ABS, stats
    assert stats["lse_max_abs"] <= LSE_MAX_ABS, stats
    return stats
