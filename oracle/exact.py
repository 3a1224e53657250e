"""Plain fp64 restatement of exact (softmax) attention.

TEST INFRASTRUCTURE ONLY (see the package docstring). Sources, cited by page
title and section:

* [MiniPaged-Qwen] "MiniPaged-Qwen: Qwen3 Prefill FlashAttention"
  (blog.zsmgc.love), sections 1, 4, 4.1, 6 and 13.
* [cuTile-FMHA] "NVIDIA闪存注意力实操：极速提升4倍性能" (nmedialink.com),
  sections "在线Softmax算法" and "因果注意力与分组查询注意力".
* [FA-demo] "FlashAttention 个人实现思路" (blueriverlhr.github.io), the
  ``torch_attn`` listing of the introduction and section "Online Softmax".
* [CuTeDSL-FA2] CUTLASS CuTe-DSL example ``ampere/flash_attention_v2.py``,
  functions ``softmax_rescale_O`` and ``normalize_softmax``.

Tensors use the (batch, seq, heads, head_dim) layout of [FA-demo]'s
introduction: q is (B, Sq, Hq, D); k and v are (B, Sk, Hkv, D). Any real
dtype is accepted and upcast to float64 before any arithmetic, so a bf16/fp16
input given as the float32 array of its exact values is used exactly.

Readings taken where the pages are silent or disagree:

* causal masking is bottom-right aligned: query i sees key j iff
  ``j <= i + Sk - Sq`` ([MiniPaged-Qwen] section 13, ``causal_limit``); it is
  the top-left form of [cuTile-FMHA] when Sq == Sk;
* a query row that sees no key gets O = 0 and LSE = -inf ([CuTeDSL-FA2]
  ``normalize_softmax`` turns a zero row sum into an all-zero output);
* LSE is the natural-log log-sum-exp of the scaled, masked scores of a row.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "kv_head_of",
    "visibility",
    "attention",
    "attention_rows",
    "probabilities",
    "attention_brute",
    "attention_online",
    "merge_partials",
]


def kv_head_of(hq: int, Hq: int, Hkv: int) -> int:
    """GQA head map: query head ``hq`` reads key/value head ``hq // (Hq/Hkv)``.

    [MiniPaged-Qwen] section 6 (group_size = Hq/Hkv, kvh = floor(qh/group_size));
    [cuTile-FMHA] "分组查询注意力" (kv_head_idx = head_idx // query_group_size).
    """
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError("Hq must be a positive multiple of Hkv")
    return hq // (Hq // Hkv)


def visibility(rows, Sq: int, Sk: int, causal: bool) -> np.ndarray:
    """Boolean matrix ``vis[r, j]``: may query ``rows[r]`` attend to key j?

    Non-causal: every key j < Sk. Causal: bottom-right alignment, key j is
    visible to query i iff ``j <= i + Sk - Sq`` ([MiniPaged-Qwen] section 13,
    ``causal_limit = kv_len - q_len + qi + 1`` is the exclusive bound).
    """
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    j = np.arange(Sk, dtype=np.int64)[None, :]
    if not causal:
        return np.ones((rows.size, Sk), dtype=bool)
    return j <= rows[:, None] + (Sk - Sq)


def _check_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be 4-D (batch, seq, heads, head_dim)")
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if k.shape != v.shape or Bk != B or Dk != D:
        raise ValueError("k and v must be (B, Sk, Hkv, D) matching q")
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError("Hq must be a positive multiple of Hkv")
    return B, Sq, Sk, Hq, Hkv, D


def _rows_two_pass(q_rows, k_h, v_h, scale, vis):
    """Two-pass softmax attention for a block of query rows of one head.

    Step 1 ([MiniPaged-Qwen] section 1): s = scale * q k^T, then the mask
    M = -inf on invisible keys. Step 2, pass 1: m = row max over visible
    keys. Pass 2: l = sum exp(s - m) ([MiniPaged-Qwen] section 4, the
    max-subtracted softmax). Step 3: O = (exp(s - m) v) / l and
    LSE = m + ln l. Rows with no visible key return O = 0, LSE = -inf.
    """
    s = scale * (q_rows @ k_h.T)                       # (n, Sk), fp64
    s_masked = np.where(vis, s, -np.inf)
    any_vis = vis.any(axis=1)
    m = np.where(any_vis, s_masked.max(axis=1, initial=-np.inf), 0.0)
    e = np.where(vis, np.exp(s_masked - m[:, None]), 0.0)
    l = e.sum(axis=1)
    safe_l = np.where(any_vis, l, 1.0)
    o = (e @ v_h) / safe_l[:, None]
    o[~any_vis] = 0.0
    with np.errstate(divide="ignore"):
        lse = np.where(any_vis, m + np.log(safe_l), -np.inf)
    return o, lse


def attention(q, k, v, scale: float, causal: bool, row_chunk: int = 512):
    """Exact attention of every query row: returns (O, LSE) in float64.

    O has q's shape (B, Sq, Hq, D); LSE is (B, Hq, Sq), natural log.
    Memory is bounded by computing ``row_chunk`` query rows at a time; this is
    only a loop split of the same two-pass definition (no online softmax).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, Sk, Hq, Hkv, D = _check_shapes(q, k, v)
    o = np.zeros((B, Sq, Hq, D), dtype=np.float64)
    lse = np.full((B, Hq, Sq), -np.inf, dtype=np.float64)
    if Sq == 0 or Sk == 0:
        return o, lse
    for b in range(B):
        for hq in range(Hq):
            kvh = kv_head_of(hq, Hq, Hkv)
            k_h = k[b, :, kvh, :]
            v_h = v[b, :, kvh, :]
            for r0 in range(0, Sq, row_chunk):
                rows = np.arange(r0, min(Sq, r0 + row_chunk))
                vis = visibility(rows, Sq, Sk, causal)
                o_r, lse_r = _rows_two_pass(q[b, rows, hq, :], k_h, v_h, scale, vis)
                o[b, rows, hq, :] = o_r
                lse[b, hq, rows] = lse_r
    return o, lse


def attention_rows(q, k, v, scale: float, causal: bool, b: int, hq: int, rows):
    """Exact attention of selected query rows of one (batch, head).

    Same definition as :func:`attention`; used to check full-size outputs on
    sampled rows. Returns (O rows (n, D), LSE (n,)) in float64.
    """
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    kvh = kv_head_of(hq, Hq, Hkv)
    q_rows = np.asarray(q[b, rows, hq, :], dtype=np.float64)
    k_h = np.asarray(k[b, :, kvh, :], dtype=np.float64)
    v_h = np.asarray(v[b, :, kvh, :], dtype=np.float64)
    if Sk == 0:
        return np.zeros((rows.size, D)), np.full(rows.size, -np.inf)
    vis = visibility(rows, Sq, Sk, causal)
    return _rows_two_pass(q_rows, k_h, v_h, scale, vis)


def probabilities(q, k, scale: float, causal: bool, b: int, hq: int):
    """The softmax matrix P (Sq, Sk) of one (batch, head), float64.

    P = softmax(scale * q k^T + M) row by row ([MiniPaged-Qwen] section 1);
    a row with no visible key is all zero.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    Sq, Hq = q.shape[1], q.shape[2]
    Sk, Hkv = k.shape[1], k.shape[2]
    kvh = kv_head_of(hq, Hq, Hkv)
    s = scale * (q[b, :, hq, :] @ k[b, :, kvh, :].T)
    vis = visibility(np.arange(Sq), Sq, Sk, causal)
    s = np.where(vis, s, -np.inf)
    any_vis = vis.any(axis=1)
    m = np.where(any_vis, s.max(axis=1, initial=-np.inf), 0.0)
    e = np.where(vis, np.exp(s - m[:, None]), 0.0)
    l = e.sum(axis=1)
    return e / np.where(any_vis, l, 1.0)[:, None]


def attention_brute(q, k, v, scale: float, causal: bool):
    """Pure-Python triple loop over (row, key, d); for tiny inputs only.

    Written independently of the vectorised path: scores by explicit sums,
    the mask by the causal_limit bound of [MiniPaged-Qwen] section 13, the
    softmax by the max-subtracted ratio of [FA-demo] "Online Softmax" (first
    formula) and O as the probability-weighted sum of v rows.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, Sk, Hq, Hkv, D = _check_shapes(q, k, v)
    group = Hq // Hkv
    o = np.zeros((B, Sq, Hq, D))
    lse = np.full((B, Hq, Sq), -math.inf)
    for b in range(B):
        for h in range(Hq):
            g = h // group
            for i in range(Sq):
                limit = Sk - Sq + i + 1 if causal else Sk
                keys = [j for j in range(min(Sk, max(limit, 0)))]
                if not keys:
                    continue
                s = []
                for j in keys:
                    acc = 0.0
                    for d in range(D):
                        acc += float(q[b, i, h, d]) * float(k[b, j, g, d])
                    s.append(scale * acc)
                mx = max(s)
                w = [math.exp(x - mx) for x in s]
                tot = sum(w)
                for d in range(D):
                    acc = 0.0
                    for wj, j in zip(w, keys):
                        acc += wj * float(v[b, j, g, d])
                    o[b, i, h, d] = acc / tot
                lse[b, h, i] = mx + math.log(tot)
    return o, lse


def attention_online(q, k, v, scale: float, causal: bool, block_n: int):
    """The tile recurrence of online softmax, in the pages' order.

    For each (b, head) and key tile t of ``block_n`` keys ([MiniPaged-Qwen]
    section 4; [cuTile-FMHA] "在线Softmax算法"):

        m_t      = rowmax(S_t)            (masked keys are -inf)
        m_new    = max(m_old, m_t)
        alpha    = exp(m_old - m_new)     (0 when m_old = -inf,
                                           [MiniPaged-Qwen] section 13)
        P_t      = exp(S_t - m_new)
        l_new    = alpha * l_old + rowsum(P_t)
        O~_new   = alpha * O~_old + P_t V_t

    and O = O~ / l after the last tile. Used to pin the claim that the
    recurrence is exact ([MiniPaged-Qwen] section 4.1). Returns (O, LSE).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, Sk, Hq, Hkv, D = _check_shapes(q, k, v)
    if block_n <= 0:
        raise ValueError("block_n must be positive")
    o = np.zeros((B, Sq, Hq, D))
    lse = np.full((B, Hq, Sq), -np.inf)
    rows = np.arange(Sq)
    for b in range(B):
        for hq in range(Hq):
            kvh = kv_head_of(hq, Hq, Hkv)
            m_old = np.full(Sq, -np.inf)
            l_old = np.zeros(Sq)
            acc = np.zeros((Sq, D))
            for c0 in range(0, Sk, block_n):
                cols = np.arange(c0, min(Sk, c0 + block_n))
                s_t = scale * (q[b, :, hq, :] @ k[b, cols, kvh, :].T)
                vis = visibility(rows, Sq, Sk, causal)[:, cols]
                s_t = np.where(vis, s_t, -np.inf)
                m_t = s_t.max(axis=1)
                m_new = np.maximum(m_old, m_t)
                live = np.isfinite(m_new)
                ref = np.where(live, m_new, 0.0)
                alpha = np.where(np.isfinite(m_old), np.exp(m_old - ref), 0.0)
                p_t = np.exp(s_t - ref[:, None])
                l_old = alpha * l_old + p_t.sum(axis=1)
                acc = alpha[:, None] * acc + p_t @ v[b, cols, kvh, :]
                m_old = m_new
            live = l_old > 0
            o[b, :, hq, :] = np.where(live[:, None], acc / np.where(live, l_old, 1.0)[:, None], 0.0)
            with np.errstate(divide="ignore"):
                lse[b, hq, :] = np.where(live, m_old + np.log(np.where(live, l_old, 1.0)), -np.inf)
    return o, lse


def merge_partials(o_parts, lse_parts):
    """Combine attention outputs computed over disjoint key sets.

    o_parts: (n, B, Sq, Hq, D); lse_parts: (n, B, Hq, Sq) natural-log LSE of
    each part. With m the running maximum and alpha the rescale factor of the
    online-softmax recurrence ([MiniPaged-Qwen] section 4; [cuTile-FMHA]
    "在线Softmax算法"), part r holds O_r = sum_j e^{s_j - LSE_r} v_j over its
    keys, so the whole is

        LSE = ln sum_r e^{LSE_r},    O = sum_r e^{LSE_r - LSE} O_r.

    Parts with LSE_r = -inf (no visible key) contribute nothing; a row with
    no part holding a key gets O = 0 and LSE = -inf. Returns float64 arrays.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    if o_parts.ndim != 5 or lse_parts.ndim != 4 or o_parts.shape[0] != lse_parts.shape[0]:
        raise ValueError("o_parts must be (n, B, Sq, Hq, D) and lse_parts (n, B, Hq, Sq)")
    n, B, Sq, Hq, D = o_parts.shape
    lse_bshq = lse_parts.transpose(0, 1, 3, 2)                 # (n, B, Sq, Hq)
    m = lse_bshq.max(axis=0)                                    # (B, Sq, Hq)
    live = np.isfinite(m)
    ref = np.where(live, m, 0.0)
    w = np.exp(lse_bshq - ref[None])                            # 0 for -inf parts
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(live, ref + np.log(np.where(live, tot, 1.0)), -np.inf)
    o = (w[..., None] * o_parts).sum(axis=0) / np.where(live, tot, 1.0)[..., None]
    o[~live] = 0.0
    return o, lse.transpose(0, 2, 1)
