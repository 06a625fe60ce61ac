"""Float64 CPU oracle for exact softmax attention.

TEST INFRASTRUCTURE ONLY.  This module is the checker the CUDA library is
compared against; it is not part of the product.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  It shares no code with the CUDA path and
imports nothing from the ``io_aware_exact_11_gb300`` package: callers hand it
plain NumPy arrays.

Sources, cited by page and section:

* [Lesson]  "FlashAttention：IO-aware 的注意力 kernel"
  (inference-learning-path.pages.dev, part 2): §2 mental model, §3.1 the
  S×S intermediate, §3.2 online softmax equations, §4 the runnable proof.
* [Notes]   FlashAttention interview notes (omica.com.cn news 1422242):
  §二.3 block-merge rule for (m, ℓ, o), §二.5 recomputation.
* [Walk]    FlashAttention walkthrough (kyonqi.github.io, nano-vllm series):
  "Safe Softmax", "online softmax" proof, "Flash Attention Forward",
  "Flash Attention Backward".

Every function computes in float64.  What each one follows:

* ``attention_forward`` / ``attention_rows`` / ``attention_probs``: the
  materialised definition S = σ·QKᵀ, P = softmax(S) (max-subtracted, as in
  [Walk] "Safe Softmax"), O = P·V, LSE = m + ln ℓ.  This is the plain
  definition the tiled method reproduces exactly ([Lesson] §1, §3.1, §6).
* ``online_attention``: the streaming recurrence of [Lesson] §3.2 in the
  pages' order (running max m, normaliser ℓ, accumulator O, rescale by
  e^(m − m_new), divide by ℓ once at the end).  It exists so the tests can
  check that the recurrence and the definition agree; it is not used as the
  oracle for the kernels.
* ``split_partials`` / ``merge_partials``: unnormalised per-chunk triples
  (m_c, ℓ_c, o_c) and the block-merge rule of [Notes] §二.3.
* ``causal=True`` (forward, rows, backward): the causal mask of the lesson's
  memory lab (§5, ``is_causal=True``), bottom-right aligned: query i of Nq
  sees keys j <= i + (Nk − Nq).  Masked scores are −∞ before the softmax,
  the plain definition with those entries removed.
* ``attention_forward_gqa``: grouped-query attention as used by the model the
  lesson's lab takes its shapes from (Qwen2.5-7B, [Lesson] §5): query head h
  reads key/value head h // G, G = H_q / H_kv.  Written as that index map over
  the plain definition.
* ``gather_pages`` / ``attention_decode_paged``: decode over a paged key/value
  cache, the block-table addressing the lesson's vLLM read-along (§4) says the
  fused kernel receives.  Logical key t of sequence b lives in page
  block_table[b, t // bs] at slot t % bs; the oracle gathers the sequence's
  keys in logical order and applies the plain definition.
* ``attention_backward``: the pages give no gradient formulas, only that the
  backward recomputes S and P from Q, K, V and the saved statistics
  ([Walk] "Flash Attention Backward", [Notes] §二.5).  The oracle uses the
  textbook gradient of O = softmax(σQKᵀ)V, written out in full.

Parity pins: every function above is pinned in ``tests/test_oracle.py``
against values the pages print, closed forms, library routines
(scipy.special), brute force on tiny inputs and finite differences.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "scores",
    "causal_visible",
    "attention_probs",
    "attention_forward",
    "attention_rows",
    "attention_forward_gqa",
    "gather_pages",
    "attention_decode_paged",
    "online_attention",
    "split_partials",
    "merge_partials",
    "attention_backward",
    "backward_delta",
]


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def scores(q, k, scale: float) -> np.ndarray:
    """S = σ·Q Kᵀ for 2-D Q [Nq, d] and K [Nk, d] ([Lesson] §3.1)."""
    q = _f64(q)
    k = _f64(k)
    return float(scale) * (q @ k.T)


def causal_visible(rows, nq: int, nk: int) -> np.ndarray:
    """Boolean [len(rows), nk]: key j is visible to query row i when j <= i + nk − nq."""
    rows = np.asarray(rows, dtype=np.int64)
    return np.arange(nk)[None, :] <= (rows[:, None] + (nk - nq))


def _mask(s, rows, nq, nk, causal):
    if not causal:
        return s
    return np.where(causal_visible(rows, nq, nk), s, -np.inf)


def _softmax_rows(s: np.ndarray):
    """Row softmax with the row max subtracted ([Walk] "Safe Softmax").

    Returns (P, m, ℓ) where m is the row max and ℓ = Σ e^(s − m).
    """
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    l = e.sum(axis=1)
    return e / l[:, None], m, l


def attention_probs(q, k, scale: float, causal: bool = False) -> np.ndarray:
    """P = softmax(σ·QKᵀ) for 2-D inputs, fully materialised."""
    nq, nk = q.shape[0], k.shape[0]
    p, _, _ = _softmax_rows(_mask(scores(q, k, scale), np.arange(nq), nq, nk, causal))
    return p


def _head_forward(q, k, v, scale, row_block, causal=False, rows=None, nq_total=None):
    nq = q.shape[0]
    rows = np.arange(nq) if rows is None else np.asarray(rows, dtype=np.int64)
    nq_total = nq if nq_total is None else nq_total
    o = np.empty((nq, v.shape[1]), dtype=np.float64)
    lse = np.empty((nq,), dtype=np.float64)
    step = nq if row_block is None else int(row_block)
    for r0 in range(0, nq, step):
        r1 = min(nq, r0 + step)
        s = _mask(scores(q[r0:r1], k, scale), rows[r0:r1], nq_total, k.shape[0], causal)
        p, m, l = _softmax_rows(s)
        o[r0:r1] = p @ v
        lse[r0:r1] = m + np.log(l)
    return o, lse


def attention_forward(q, k, v, scale: float, row_block: int | None = 256, causal: bool = False):
    """Exact attention, materialised one block of query rows at a time.

    q: [..., Nq, d], k and v: [..., Nk, d] (any leading batch dims, e.g. B, H).
    Returns (O [..., Nq, d], LSE [..., Nq]) in float64, LSE = m + ln ℓ over the
    scaled scores (natural log).  Each query row's softmax is complete over all
    Nk keys; ``row_block`` only bounds how many rows are held at once, and rows
    are independent, so it does not change any value.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    lead = q.shape[:-2]
    assert k.shape[:-2] == lead and v.shape[:-2] == lead
    assert k.shape[-2] == v.shape[-2] and q.shape[-1] == k.shape[-1]
    qf = q.reshape((-1,) + q.shape[-2:])
    kf = k.reshape((-1,) + k.shape[-2:])
    vf = v.reshape((-1,) + v.shape[-2:])
    o = np.empty(qf.shape[:-1] + (vf.shape[-1],), dtype=np.float64)
    lse = np.empty(qf.shape[:-1], dtype=np.float64)
    if causal:
        assert q.shape[-2] <= k.shape[-2], "causal attention needs Nq <= Nk"
    for g in range(qf.shape[0]):
        o[g], lse[g] = _head_forward(qf[g], kf[g], vf[g], scale, row_block, causal)
    return o.reshape(lead + o.shape[-2:]), lse.reshape(lead + lse.shape[-1:])


def attention_rows(q_head, k_head, v_head, scale: float, rows, causal: bool = False):
    """Exact attention for selected query rows of one head.

    q_head [Nq, d], k_head/v_head [Nk, d]; ``rows`` indexes q_head.  Rows are
    independent ([Lesson] §3.3: the outer loop is over query rows), so this is
    the same function as ``attention_forward`` restricted to those rows.
    """
    rows = np.asarray(rows, dtype=np.int64)
    q = _f64(q_head)[rows]
    return _head_forward(q, _f64(k_head), _f64(v_head), scale, None, causal, rows, q_head.shape[0])


def online_attention(q, k, v, scale: float, block: int):
    """Streaming (online-softmax) attention for 2-D inputs, [Lesson] §3.2.

    Keys and values are consumed ``block`` at a time.  Per query row the state
    is the running max m (starting at −∞), the running normaliser ℓ (0) and the
    unnormalised accumulator O (0).  For each block with scores s_j:
        m_new = max(m, max_j s_j)
        ℓ     = e^(m − m_new)·ℓ + Σ_j e^(s_j − m_new)
        O     = e^(m − m_new)·O + Σ_j e^(s_j − m_new)·v_j
    with the rescale factor taken as 0 while m is still −∞ ([Lesson] §4).
    After the last block O/ℓ is the output; LSE = m + ln ℓ.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    nq, nk = q.shape[0], k.shape[0]
    m = np.full((nq,), -np.inf)
    l = np.zeros((nq,))
    acc = np.zeros((nq, v.shape[1]))
    for j0 in range(0, nk, int(block)):
        s = scores(q, k[j0:j0 + block], scale)
        m_new = np.maximum(m, s.max(axis=1))
        corr = np.where(np.isneginf(m), 0.0, np.exp(m - m_new))
        p = np.exp(s - m_new[:, None])
        l = corr * l + p.sum(axis=1)
        acc = corr[:, None] * acc + p @ v[j0:j0 + block]
        m = m_new
    return acc / l[:, None], m + np.log(l)


def attention_forward_gqa(q, k, v, scale: float, causal: bool = False):
    """Grouped-query attention: q [B, Hq, Nq, d], k/v [B, Hkv, Nk, d], Hq % Hkv == 0.

    Query head h attends with key/value head h // (Hq / Hkv); everything else
    is ``attention_forward``.  Returns (O [B, Hq, Nq, d], LSE [B, Hq, Nq]).
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    B, Hq = q.shape[:2]
    Hkv = k.shape[1]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    o = np.empty(q.shape[:3] + (v.shape[-1],))
    lse = np.empty(q.shape[:3])
    for b in range(B):
        for h in range(Hq):
            o[b, h], lse[b, h] = attention_forward(q[b, h], k[b, h // G], v[b, h // G], scale, causal=causal)
    return o, lse


def gather_pages(cache, block_table, seq_len: int, head: int):
    """Logical rows [0, seq_len) of one key/value head from a paged cache.

    cache [num_blocks, H_kv, bs, d]; block_table: the sequence's page ids.
    """
    cache = np.asarray(cache)
    bs = cache.shape[2]
    rows = [cache[int(block_table[t // bs]), head, t % bs] for t in range(int(seq_len))]
    return _f64(np.stack(rows)) if rows else np.zeros((0, cache.shape[3]))


def attention_decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale: float):
    """One query row per head against a paged cache; q [B, Hq, d].

    Query head h of sequence b reads key/value head h // (Hq / H_kv) over the
    sequence's seq_lens[b] logical keys.  Returns (O [B, Hq, d], LSE [B, Hq]).
    """
    q = _f64(q)
    B, Hq, d = q.shape
    Hkv = np.asarray(k_cache).shape[1]
    G = Hq // Hkv
    o = np.empty((B, Hq, d))
    lse = np.empty((B, Hq))
    for b in range(B):
        for h in range(Hq):
            k = gather_pages(k_cache, block_table[b], seq_lens[b], h // G)
            v = gather_pages(v_cache, block_table[b], seq_lens[b], h // G)
            ob, lb = attention_forward(q[b, h][None, :], k, v, scale)
            o[b, h], lse[b, h] = ob[0], lb[0]
    return o, lse


def split_partials(q, k, v, scale: float, n_splits: int):
    """Per-chunk unnormalised triples for split-KV decode.

    q [Nq, d]; the keys are cut into ``n_splits`` contiguous chunks of
    ceil(Nk / n_splits) keys (the last may be shorter or empty).  For chunk c,
    over its own keys only: m_c = max s, ℓ_c = Σ e^(s − m_c),
    o_c = Σ e^(s − m_c)·v (not divided by ℓ_c).  An empty chunk gives
    (−∞, 0, 0).  Returns arrays m [n_splits, Nq], ℓ [n_splits, Nq],
    o [n_splits, Nq, d].
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    nk = k.shape[0]
    chunk = -(-nk // int(n_splits))
    ms = np.full((n_splits, q.shape[0]), -np.inf)
    ls = np.zeros((n_splits, q.shape[0]))
    os_ = np.zeros((n_splits, q.shape[0], v.shape[1]))
    for c in range(n_splits):
        j0, j1 = c * chunk, min(nk, (c + 1) * chunk)
        if j1 <= j0:
            continue
        s = scores(q, k[j0:j1], scale)
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        ms[c], ls[c], os_[c] = m, e.sum(axis=1), e @ v[j0:j1]
    return ms, ls, os_


def merge_partials(ms, ls, os_):
    """Block-merge rule of [Notes] §二.3, folded over the chunks in order.

    Two triples (m_a, ℓ_a, o_a), (m_b, ℓ_b, o_b) combine as
        m = max(m_a, m_b),  ℓ = ℓ_a e^(m_a − m) + ℓ_b e^(m_b − m),
        o = o_a e^(m_a − m) + o_b e^(m_b − m).
    A chunk with m = −∞ (no keys) contributes nothing.  Returns the final
    (O = o/ℓ, LSE = m + ln ℓ).
    """
    ms = _f64(ms)
    ls = _f64(ls)
    os_ = _f64(os_)
    m = ms[0].copy()
    l = ls[0].copy()
    o = os_[0].copy()
    for c in range(1, ms.shape[0]):
        m_new = np.maximum(m, ms[c])
        wa = np.where(np.isneginf(m), 0.0, np.exp(m - m_new))
        wb = np.where(np.isneginf(ms[c]), 0.0, np.exp(ms[c] - m_new))
        l = l * wa + ls[c] * wb
        o = o * wa[..., None] + os_[c] * wb[..., None]
        m = m_new
    return o / l[..., None], m + np.log(l)


def backward_delta(do, o) -> np.ndarray:
    """D_i = Σ_t dO_it·O_it, the row term of the softmax gradient."""
    return np.sum(_f64(do) * _f64(o), axis=-1)


def _head_backward(q, k, v, do, scale, causal=False):
    p = attention_probs(q, k, scale, causal)  # recomputed, never stored by the kernels
    o = p @ v
    dv = p.T @ do                             # O = P V  ⇒  dV = Pᵀ dO
    dp = do @ v.T                             #            dP = dO Vᵀ
    dsum = np.sum(p * dp, axis=1)             # Σ_j P_ij dP_ij  (= Σ_t dO_it O_it)
    ds = p * (dp - dsum[:, None])             # softmax Jacobian applied row-wise
    dq = scale * (ds @ k)                     # S = σ Q Kᵀ
    dk = scale * (ds.T @ q)
    return dq, dk, dv, o


def attention_backward(q, k, v, do, scale: float, causal: bool = False):
    """Gradients of O = softmax(σ·QKᵀ)·V with respect to Q, K, V.

    q/k/v/do: [..., N, d].  The textbook derivation: dV = Pᵀ·dO,
    dP = dO·Vᵀ, dS = P ∘ (dP − rowsum(P ∘ dP)), dQ = σ·dS·K, dK = σ·dSᵀ·Q.
    P is recomputed here from Q and K (with the causal mask when ``causal``:
    masked entries of P are 0, so they drop out of every product).  Returns
    (dQ, dK, dV) in float64.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    do = _f64(do)
    lead = q.shape[:-2]
    qf = q.reshape((-1,) + q.shape[-2:])
    kf = k.reshape((-1,) + k.shape[-2:])
    vf = v.reshape((-1,) + v.shape[-2:])
    dof = do.reshape((-1,) + do.shape[-2:])
    dq = np.empty_like(qf)
    dk = np.empty_like(kf)
    dv = np.empty_like(vf)
    for g in range(qf.shape[0]):
        dq[g], dk[g], dv[g], _ = _head_backward(qf[g], kf[g], vf[g], dof[g], scale, causal)
    return dq.reshape(q.shape), dk.reshape(k.shape), dv.reshape(v.shape)
