"""Pins for the float64 oracle (CPU only).

Each test ties the oracle to something outside itself: the worked example the
lesson prints ("FlashAttention：IO-aware 的注意力 kernel", §4), closed forms,
invariants of softmax attention, scipy's softmax / logsumexp, brute force on
tiny inputs and central finite differences for the backward.
"""

import json
import math
import os

import numpy as np
import pytest
from scipy import special

import oracle

RNG = np.random.default_rng(1234)


def _worked(golden_dir):
    with open(os.path.join(golden_dir, "worked_example.json")) as f:
        g = json.load(f)
    q = np.array(g["q"])[None, :]
    K = np.array(g["K"])
    V = np.array(g["V"])
    return g, q, K, V, 1.0 / math.sqrt(q.shape[1])


def test_worked_example_matches_printed_output(golden_dir):
    g, q, K, V, scale = _worked(golden_dir)
    o, lse = oracle.attention_forward(q, K, V, scale)
    assert np.all(np.round(o[0], g["O_decimals"]) == np.array(g["O_printed"]))
    # The printed values are rounded to 6 decimals.
    assert np.max(np.abs(o[0] - np.array(g["O_printed"]))) <= 5e-7
    assert np.isfinite(lse).all()


@pytest.mark.parametrize("block", [1, 2, 3, 6])
def test_worked_example_online_equals_full(golden_dir, block):
    g, q, K, V, scale = _worked(golden_dir)
    o_full, lse_full = oracle.attention_forward(q, K, V, scale)
    o_on, lse_on = oracle.online_attention(q, K, V, scale, block)
    # The lesson prints 1.11e-16 for block=2: floating point noise, not error.
    assert np.max(np.abs(o_full - o_on)) <= 4 * np.finfo(np.float64).eps
    assert np.max(np.abs(lse_full - lse_on)) <= 8 * np.finfo(np.float64).eps
    assert np.all(np.round(o_on[0], 6) == np.array(g["O_printed"]))


def test_worked_example_by_brute_force(golden_dir):
    """Independent scalar evaluation with math.fsum on the printed example."""
    g, q, K, V, scale = _worked(golden_dir)
    s = [math.fsum(a * b for a, b in zip(q[0], k)) / 2.0 for k in K]   # sqrt(4) = 2
    z = math.fsum(math.exp(x) for x in s)
    o = [math.fsum(math.exp(s[i]) / z * V[i][t] for i in range(len(K))) for t in range(4)]
    lse = math.log(z)
    o_ref, lse_ref = oracle.attention_forward(q, K, V, scale)
    assert np.max(np.abs(np.array(o) - o_ref[0])) < 1e-15
    assert abs(lse - lse_ref[0]) < 1e-15


@pytest.mark.parametrize("nq,nk,d", [(5, 7, 3), (16, 33, 8), (1, 1, 4)])
def test_matches_scipy_softmax_and_logsumexp(nq, nk, d):
    q = RNG.standard_normal((nq, d))
    k = RNG.standard_normal((nk, d))
    v = RNG.standard_normal((nk, d))
    scale = 1.0 / math.sqrt(d)
    s = np.einsum("it,jt->ij", q, k) * scale
    o, lse = oracle.attention_forward(q, k, v, scale)
    assert np.allclose(o, special.softmax(s, axis=1) @ v, rtol=0, atol=1e-13)
    assert np.allclose(lse, special.logsumexp(s, axis=1), rtol=0, atol=1e-13)


def test_values_all_ones_give_all_ones():
    q = RNG.standard_normal((9, 6))
    k = RNG.standard_normal((13, 6))
    o, _ = oracle.attention_forward(q, k, np.ones((13, 6)), 0.4)
    assert np.allclose(o, 1.0, atol=1e-14)


def test_identity_values_give_probabilities_with_unit_row_sums():
    n = 11
    q = RNG.standard_normal((7, n))
    k = RNG.standard_normal((n, n))
    o, _ = oracle.attention_forward(q, k, np.eye(n), 0.3)
    p = oracle.attention_probs(q, k, 0.3)
    assert np.allclose(o, p, atol=1e-15)
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-12)
    assert (p > 0).all()


def test_shift_of_all_keys_shifts_lse_not_output():
    q = RNG.standard_normal((8, 5))
    k = RNG.standard_normal((10, 5))
    v = RNG.standard_normal((10, 5))
    w = RNG.standard_normal(5) * 3
    scale = 0.7
    o0, l0 = oracle.attention_forward(q, k, v, scale)
    o1, l1 = oracle.attention_forward(q, k + w, v, scale)
    assert np.allclose(o0, o1, atol=1e-12)
    assert np.allclose(l1 - l0, scale * (q @ w), atol=1e-12)


def test_equal_keys_give_uniform_weights():
    n, d = 12, 4
    q = RNG.standard_normal((3, d))
    k = np.tile(RNG.standard_normal((1, d)), (n, 1))
    v = RNG.standard_normal((n, d))
    o, lse = oracle.attention_forward(q, k, v, 0.5)
    assert np.allclose(o, v.mean(axis=0)[None, :], atol=1e-14)
    assert np.allclose(lse, 0.5 * (q @ k[0]) + math.log(n), atol=1e-13)


def test_single_key_returns_its_value_and_score():
    q = RNG.standard_normal((4, 3))
    k = RNG.standard_normal((1, 3))
    v = RNG.standard_normal((1, 3))
    o, lse = oracle.attention_forward(q, k, v, 1.3)
    assert np.allclose(o, np.tile(v, (4, 1)), atol=1e-15)
    assert np.allclose(lse, 1.3 * (q @ k[0]), atol=1e-15)


def test_head_dim_one_by_hand():
    """d = 1, σ = 1: q = ln 2, keys (1, 0) give scores (ln 2, 0), softmax weights (2/3, 1/3); with values
    (3, 6) the output is 2/3·3 + 1/3·6 = 4 and LSE = ln(2 + 1) = ln 3."""
    q = np.array([[math.log(2.0)]])
    k = np.array([[1.0], [0.0]])
    v = np.array([[3.0], [6.0]])
    o, lse = oracle.attention_forward(q, k, v, 1.0)
    assert abs(o[0, 0] - 4.0) <= 1e-14
    assert abs(lse[0] - math.log(3.0)) <= 1e-14


def test_large_scores_are_stable():
    q = RNG.standard_normal((4, 8)) * 40
    k = RNG.standard_normal((20, 8)) * 40
    v = RNG.standard_normal((20, 8))
    o, lse = oracle.attention_forward(q, k, v, 1.0)
    s = q @ k.T
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert np.allclose(lse, special.logsumexp(s, axis=1), rtol=1e-15, atol=1e-12)


def test_permutation_equivariance():
    q = RNG.standard_normal((6, 4))
    k = RNG.standard_normal((9, 4))
    v = RNG.standard_normal((9, 4))
    pk = RNG.permutation(9)
    pq = RNG.permutation(6)
    o, lse = oracle.attention_forward(q, k, v, 0.5)
    o2, lse2 = oracle.attention_forward(q[pq], k[pk], v[pk], 0.5)
    assert np.allclose(o[pq], o2, atol=1e-14)
    assert np.allclose(lse[pq], lse2, atol=1e-14)


def test_row_block_does_not_change_result():
    q = RNG.standard_normal((2, 3, 37, 8))
    k = RNG.standard_normal((2, 3, 29, 8))
    v = RNG.standard_normal((2, 3, 29, 8))
    ref = oracle.attention_forward(q, k, v, 0.35, row_block=None)
    for rb in (1, 7, 16, 256):
        o, lse = oracle.attention_forward(q, k, v, 0.35, row_block=rb)
        assert np.max(np.abs(o - ref[0])) <= 1e-12
        assert np.max(np.abs(lse - ref[1])) <= 1e-12


def test_rows_helper_matches_full():
    q = RNG.standard_normal((40, 8))
    k = RNG.standard_normal((50, 8))
    v = RNG.standard_normal((50, 8))
    o, lse = oracle.attention_forward(q, k, v, 0.3)
    rows = [0, 5, 39, 17]
    o2, lse2 = oracle.attention_rows(q, k, v, 0.3, rows)
    assert np.max(np.abs(o2 - o[rows])) <= 1e-14
    assert np.max(np.abs(lse2 - lse[rows])) <= 1e-14


@pytest.mark.parametrize("block", [1, 5, 16, 64])
def test_online_matches_definition_random(block):
    q = RNG.standard_normal((12, 16))
    k = RNG.standard_normal((61, 16)) * 2
    v = RNG.standard_normal((61, 16))
    o, lse = oracle.attention_forward(q, k, v, 0.25)
    o2, lse2 = oracle.online_attention(q, k, v, 0.25, block)
    assert np.max(np.abs(o - o2)) <= 1e-13
    assert np.max(np.abs(lse - lse2)) <= 1e-13


@pytest.mark.parametrize("nk,n_splits", [(256, 32), (100, 32), (8, 32), (1000, 7), (5, 1)])
def test_split_merge_equals_full_row(nk, n_splits):
    q = RNG.standard_normal((1, 16))
    k = RNG.standard_normal((nk, 16))
    v = RNG.standard_normal((nk, 16))
    o, lse = oracle.attention_forward(q, k, v, 0.25)
    ms, ls, os_ = oracle.split_partials(q, k, v, 0.25, n_splits)
    o2, lse2 = oracle.merge_partials(ms, ls, os_)
    assert np.max(np.abs(o - o2)) <= 1e-13
    assert np.max(np.abs(lse - lse2)) <= 1e-13


def test_merge_of_two_single_key_chunks_closed_form():
    # Chunk a holds one key with score sa, chunk b one key with score sb:
    # the merged result is the two-key softmax, worked out by hand.
    sa, sb = 0.3, -1.1
    va, vb = np.array([[1.0, 2.0]]), np.array([[-3.0, 0.5]])
    ms = np.array([[sa], [sb]])
    ls = np.array([[1.0], [1.0]])
    os_ = np.stack([va, vb])
    o, lse = oracle.merge_partials(ms, ls, os_)
    wa = 1.0 / (1.0 + math.exp(sb - sa))
    assert np.allclose(o[0], wa * va[0] + (1 - wa) * vb[0], atol=1e-15)
    assert abs(lse[0] - (sa + math.log1p(math.exp(sb - sa)))) < 1e-15


# ---------------------------------------------------------------- backward


def _loss(q, k, v, do, scale):
    o, _ = oracle.attention_forward(q, k, v, scale)
    return float(np.sum(o * do))


@pytest.mark.parametrize("n,nk,d", [(4, 4, 3), (6, 8, 4), (1, 5, 2)])
def test_backward_matches_finite_differences(n, nk, d):
    rng = np.random.default_rng(n * 100 + nk * 10 + d)
    q = rng.standard_normal((n, d))
    k = rng.standard_normal((nk, d))
    v = rng.standard_normal((nk, d))
    do = rng.standard_normal((n, d))
    scale = 1.0 / math.sqrt(d)
    if n == nk:
        dq, dk, dv = oracle.attention_backward(q, k, v, do, scale)
    else:
        # The library's backward is square (self-attention); the oracle's
        # per-head gradient is general, exercise it directly.
        from oracle.attention import _head_backward
        dq, dk, dv, _ = _head_backward(q, k, v, do, scale)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp = x.copy()
            xm = x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name] = xp
            args_m[name] = xm
            num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], do, scale)
                        - _loss(args_m["q"], args_m["k"], args_m["v"], do, scale)) / (2 * h)
        err = np.linalg.norm(num - g) / max(np.linalg.norm(num), 1e-30)
        assert err <= 1e-6, (name, err)


def test_backward_delta_identity():
    q = RNG.standard_normal((10, 6))
    k = RNG.standard_normal((10, 6))
    v = RNG.standard_normal((10, 6))
    do = RNG.standard_normal((10, 6))
    p = oracle.attention_probs(q, k, 0.4)
    o, _ = oracle.attention_forward(q, k, v, 0.4)
    dp = do @ v.T
    assert np.allclose(np.sum(p * dp, axis=1), oracle.backward_delta(do, o), atol=1e-13)


def test_backward_single_key_closed_form():
    """One key: every query's softmax row is [1], so O = V, dV = Σ_i dO_i and
    dS = P∘(dP − D) vanishes, leaving dQ = dK = 0."""
    q = RNG.standard_normal((5, 4))
    k = RNG.standard_normal((1, 4))
    v = RNG.standard_normal((1, 4))
    do = RNG.standard_normal((5, 4))
    o, lse = oracle.attention_forward(q, k, v, 0.5)
    assert np.allclose(o, np.repeat(v, 5, axis=0), atol=1e-15)
    assert np.allclose(lse, 0.5 * (q @ k[0]), atol=1e-14)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5)
    assert np.abs(dq).max() <= 1e-14 and np.abs(dk).max() <= 1e-14
    assert np.allclose(dv, do.sum(axis=0, keepdims=True), atol=1e-14)


def test_backward_matches_torch_autograd_fp64():
    torch = pytest.importorskip("torch")
    q = RNG.standard_normal((2, 3, 17, 8))
    k = RNG.standard_normal((2, 3, 17, 8))
    v = RNG.standard_normal((2, 3, 17, 8))
    do = RNG.standard_normal((2, 3, 17, 8))
    scale = 0.3
    dq, dk, dv = oracle.attention_backward(q, k, v, do, scale)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    o = torch.softmax(scale * tq @ tk.transpose(-1, -2), dim=-1) @ tv
    o.backward(torch.tensor(do))
    assert np.allclose(tq.grad.numpy(), dq, atol=1e-12)
    assert np.allclose(tk.grad.numpy(), dk, atol=1e-12)
    assert np.allclose(tv.grad.numpy(), dv, atol=1e-12)


# ------------------------------------------------------------------ causal
# The causal mask follows the lesson's memory lab (§5, is_causal=True),
# bottom-right aligned: query i of Nq sees keys j <= i + Nk − Nq.


@pytest.mark.parametrize("nq,nk", [(9, 9), (5, 12), (1, 7), (16, 16)])
def test_causal_row_equals_unmasked_attention_over_its_prefix(nq, nk):
    """Independent route: the masked row is the plain definition on a truncated key set."""
    q = RNG.standard_normal((nq, 6))
    k = RNG.standard_normal((nk, 6))
    v = RNG.standard_normal((nk, 6))
    o, lse = oracle.attention_forward(q, k, v, 0.4, causal=True)
    for i in range(nq):
        n_vis = i + (nk - nq) + 1
        oi, li = oracle.attention_forward(q[i:i + 1], k[:n_vis], v[:n_vis], 0.4)
        assert np.allclose(o[i], oi[0], atol=1e-14)
        assert abs(lse[i] - li[0]) < 1e-13
        s = 0.4 * (k[:n_vis] @ q[i])
        assert abs(lse[i] - special.logsumexp(s)) < 1e-13


def test_causal_first_and_last_rows():
    n = 10
    q = RNG.standard_normal((n, 4))
    k = RNG.standard_normal((n, 4))
    v = RNG.standard_normal((n, 4))
    o, lse = oracle.attention_forward(q, k, v, 0.5, causal=True)
    full_o, full_lse = oracle.attention_forward(q, k, v, 0.5)
    assert np.allclose(o[0], v[0], atol=1e-15)            # row 0 sees key 0 only
    assert abs(lse[0] - 0.5 * q[0] @ k[0]) < 1e-15
    assert np.allclose(o[-1], full_o[-1], atol=1e-15)     # the last row sees every key
    assert abs(lse[-1] - full_lse[-1]) < 1e-15


def test_causal_rows_helper_and_row_blocks_agree():
    q = RNG.standard_normal((2, 2, 40, 8))
    k = RNG.standard_normal((2, 2, 55, 8))
    v = RNG.standard_normal((2, 2, 55, 8))
    ref = oracle.attention_forward(q, k, v, 0.3, row_block=None, causal=True)
    o, lse = oracle.attention_forward(q, k, v, 0.3, row_block=7, causal=True)
    assert np.max(np.abs(o - ref[0])) <= 1e-13
    rows = [0, 13, 39]
    o2, l2 = oracle.attention_rows(q[1, 0], k[1, 0], v[1, 0], 0.3, rows, causal=True)
    assert np.max(np.abs(o2 - ref[0][1, 0][rows])) <= 1e-14
    assert np.max(np.abs(l2 - ref[1][1, 0][rows])) <= 1e-14


def test_causal_backward_matches_finite_differences():
    rng = np.random.default_rng(77)
    n, d = 6, 3
    q, k, v, do = (rng.standard_normal((n, d)) for _ in range(4))
    scale = 0.6
    dq, dk, dv = oracle.attention_backward(q, k, v, do, scale, causal=True)

    def loss(qq, kk, vv):
        o, _ = oracle.attention_forward(qq, kk, vv, scale, causal=True)
        return float(np.sum(o * do))
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            args = {"q": q, "k": k, "v": v}
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            num[idx] = (loss(**{**{"qq": q, "kk": k, "vv": v}, **{name * 2: xp}})
                        - loss(**{**{"qq": q, "kk": k, "vv": v}, **{name * 2: xm}})) / (2 * h)
        assert np.linalg.norm(num - g) / np.linalg.norm(num) <= 1e-6, name
    # The last key only reaches the last query row.
    assert np.allclose(dv[-1], oracle.attention_probs(q, k, scale, True)[-1, -1] * do[-1], atol=1e-14)


# --------------------------------------------------------- grouped queries


def test_gqa_equals_standard_attention_on_repeated_heads():
    """Independent route: repeat each K/V head G times and use the plain path."""
    B, Hq, Hkv, N, d = 2, 6, 2, 9, 4
    q = RNG.standard_normal((B, Hq, 1, d))
    k = RNG.standard_normal((B, Hkv, N, d))
    v = RNG.standard_normal((B, Hkv, N, d))
    o, lse = oracle.attention_forward_gqa(q, k, v, 0.5)
    o2, lse2 = oracle.attention_forward(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), 0.5)
    assert np.allclose(o, o2, atol=1e-15) and np.allclose(lse, lse2, atol=1e-15)
    # Heads of one group differ only through their queries.
    o3, _ = oracle.attention_forward_gqa(np.repeat(q[:, :1], 6, axis=1), k, v, 0.5)
    assert np.allclose(o3[:, 0], o3[:, 2], atol=1e-15) and not np.allclose(o3[:, 0], o3[:, 3])


def test_gqa_with_one_group_is_standard():
    q = RNG.standard_normal((1, 3, 4, 5))
    k = RNG.standard_normal((1, 3, 7, 5))
    v = RNG.standard_normal((1, 3, 7, 5))
    assert np.allclose(oracle.attention_forward_gqa(q, k, v, 0.3)[0], oracle.attention_forward(q, k, v, 0.3)[0])


# ------------------------------------------------------------ paged cache


def _pack_pages(k, bs, order):
    """Contiguous [B, Hkv, N, d] cache -> pages [NB, Hkv, bs, d] placed at `order`."""
    B, Hkv, N, d = k.shape
    per = -(-N // bs)
    pages = np.zeros((B * per + 3, Hkv, bs, d))
    table = np.zeros((B, per), dtype=np.int32)
    for b in range(B):
        for i in range(per):
            pid = order[b * per + i]
            blk = k[b, :, i * bs:(i + 1) * bs]
            pages[pid, :, :blk.shape[1]] = blk
            table[b, i] = pid
    return pages, table


def test_paged_decode_equals_contiguous_decode_for_any_page_order():
    B, Hq, Hkv, N, d, bs = 2, 4, 2, 37, 8, 16
    q = RNG.standard_normal((B, Hq, d))
    k = RNG.standard_normal((B, Hkv, N, d))
    v = RNG.standard_normal((B, Hkv, N, d))
    lens = np.array([37, 21])
    per = -(-N // bs)
    for order in (np.arange(B * per), RNG.permutation(B * per + 3)[:B * per]):
        kc, table = _pack_pages(k, bs, order)
        vc, _ = _pack_pages(v, bs, order)
        o, lse = oracle.attention_decode_paged(q, kc, vc, table, lens, 0.35)
        for b in range(B):
            ref_o, ref_l = oracle.attention_forward_gqa(q[b][None, :, None, :], k[b:b + 1, :, :lens[b]],
                                                        v[b:b + 1, :, :lens[b]], 0.35)
            assert np.allclose(o[b], ref_o[0, :, 0], atol=1e-14)
            assert np.allclose(lse[b], ref_l[0, :, 0], atol=1e-14)


def test_gather_pages_follows_the_block_table():
    cache = np.arange(4 * 1 * 2 * 1, dtype=np.float64).reshape(4, 1, 2, 1)   # page p holds values 2p, 2p+1
    rows = oracle.gather_pages(cache, [3, 0, 2], 5, 0)
    assert rows[:, 0].tolist() == [6.0, 7.0, 0.0, 1.0, 4.0]
