"""GPU parity of split-KV decode over a paged key/value cache.

Pages are [num_blocks, H_kv, block_size, d]; logical key t of sequence b is
row t % bs of page block_table[b, t // bs].  The page pool is pre-filled with
NaN bit patterns and unused table entries are -1, so reading any slot past a
sequence's end, or any unused entry, would show up in the output.  Expected
values come from the oracle's gather + plain definition.  Tolerances as for
decode: O within 1e-2 max-abs, LSE within 1e-3.
"""

import math

import numpy as np
import pytest

import oracle
from io_aware_exact_11_gb300 import fa, inputs
from tests.gpu_helpers import cpu64, max_abs, to_device

pytestmark = pytest.mark.gpu
NAN_BF16 = np.uint16(0x7FC0)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.lib()
    yield
    fa.device_status()


def _paged(seed, B, Hq, Hkv, lens, bs, extra_pages=5, d=128):
    """Seeded contiguous K/V scattered into a shuffled, NaN-filled page pool."""
    maxlen = int(max(lens))
    per = -(-maxlen // bs)
    k = inputs.normal_tensor(seed, "k", B, Hkv, maxlen, d, "bf16")
    v = inputs.normal_tensor(seed, "v", B, Hkv, maxlen, d, "bf16")
    q = inputs.normal_tensor(seed, "q", B, Hq, 1, d, "bf16")[:, :, 0]
    used = [-(-int(n) // bs) for n in lens]
    nb = sum(used) + extra_pages
    order = np.random.default_rng(seed).permutation(nb)
    kc = np.full((nb, Hkv, bs, d), NAN_BF16, dtype=np.uint16)
    vc = np.full((nb, Hkv, bs, d), NAN_BF16, dtype=np.uint16)
    table = np.full((B, per + 2), -1, dtype=np.int32)
    nxt = 0
    for b in range(B):
        for i in range(used[b]):
            pid = int(order[nxt])
            nxt += 1
            r0, r1 = i * bs, min(int(lens[b]), (i + 1) * bs)
            kc[pid, :, :r1 - r0] = k[b, :, r0:r1]
            vc[pid, :, :r1 - r0] = v[b, :, r0:r1]
            table[b, i] = pid
    return q, kc, vc, table, np.asarray(lens, dtype=np.int32)


def _run(seed, B, Hq, Hkv, lens, bs, splits, heads=None, d=128):
    import torch
    q, kc, vc, table, lens = _paged(seed, B, Hq, Hkv, lens, bs, d=d)
    scale = 1 / math.sqrt(d)
    qd = to_device(q[:, :, None, :].copy(), "bf16")
    o, lse = fa.decode_paged(qd, to_device(kc, "bf16"), to_device(vc, "bf16"), torch.from_numpy(table).cuda(),
                             torch.from_numpy(lens).cuda(), n_splits=splits, scale=scale)
    fa.device_status()
    assert bool(torch.isfinite(o.float()).all()) and bool(torch.isfinite(lse).all())
    ro, rl = oracle.attention_decode_paged(inputs.as_f64(q, "bf16"), inputs.as_f64(kc, "bf16"),
                                           inputs.as_f64(vc, "bf16"), table, lens, scale) if heads is None else (None,
                                                                                                            None)
    if heads is None:
        assert max_abs(cpu64(o)[:, :, 0], ro) <= 1e-2
        assert max_abs(cpu64(lse), rl) <= 1e-3
    else:
        G = Hq // Hkv
        for b, h in heads:
            kk = oracle.gather_pages(inputs.as_f64(kc, "bf16"), table[b], lens[b], h // G)
            vv = oracle.gather_pages(inputs.as_f64(vc, "bf16"), table[b], lens[b], h // G)
            ob, lb = oracle.attention_forward(inputs.as_f64(q[b, h], "bf16")[None, :], kk, vv, scale)
            assert max_abs(cpu64(o[b, h, 0]), ob[0]) <= 1e-2, (b, h)
            assert abs(float(lse[b, h]) - lb[0]) <= 1e-3, (b, h)
    return o, lse


@pytest.mark.parametrize("B,Hq,Hkv,lens,bs,splits", [
    (3, 4, 4, [1000, 37, 2049], 16, 8),      # one query head per key/value head
    (3, 28, 4, [1000, 1, 300], 16, 4),       # groups of 7, a one-key sequence
    (2, 28, 4, [513, 777], 64, 4),
    (2, 8, 4, [128, 1200], 128, 16),         # groups of 2, one page per tile
    (1, 8, 1, [700], 32, 1),                 # one key/value head, one split
    (1, 8, 2, [17000], 16, 1),               # 1063 pages in one split: past the 1024 staged page ids
    (2, 32, 1, [900, 333], 16, 4),           # multi-query attention over 16-key pages
    (2, 32, 2, [640, 129], 64, 2),           # groups of 16 over 64-key pages
    (2, 64, 1, [900, 130], 16, 4),           # group of 64 (two softmax warps), partial last tiles
    (1, 96, 2, [1000], 32, 2),               # groups of 48
])
def test_paged_decode_matches_oracle(B, Hq, Hkv, lens, bs, splits):
    _run(41, B, Hq, Hkv, lens, bs, splits)


@pytest.mark.parametrize("B,Hq,Hkv,lens,bs,splits", [
    (3, 4, 4, [1000, 37, 2049], 16, 8),      # single-head kernel
    (3, 28, 4, [1000, 1, 300], 16, 4),       # grouped kernel, partial last tiles
    (2, 64, 1, [700, 130], 64, 2),           # group of 64
])
def test_paged_decode_head_dim_64_matches_oracle(B, Hq, Hkv, lens, bs, splits):
    _run(42, B, Hq, Hkv, lens, bs, splits, d=64)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 4)])   # single-head kernel; grouped tensor-core kernel
def test_paged_decode_flags_a_bad_page_id_without_faulting(Hq, Hkv):
    import torch
    q, kc, vc, table, lens = _paged(42, 1, Hq, Hkv, [300], 16)
    table[0, 3] = 10 ** 6
    with pytest.raises(fa.FAError) as ei:
        fa.decode_paged(to_device(q[:, :, None, :].copy(), "bf16"), to_device(kc, "bf16"), to_device(vc, "bf16"),
                        torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(), n_splits=4)
        fa.device_status()
    assert ei.value.status == fa.FA_ERR_INVALID_ARG
    fa.device_status()   # the flag was cleared and the context is healthy


@pytest.mark.slow
def test_paged_decode_qwen_shape_full_size_sampled():
    """B=64, 28 query / 4 key-value heads, 8192 keys each in 16-key pages, 4 splits."""
    _run(43, 64, 28, 4, [8192] * 64, 16, 4, heads=[(0, 0), (63, 27), (20, 9), (41, 16)])
