"""GPU parity of grouped-query split-KV decode against the float64 oracle.

Query head h reads key/value head h // G (G = Hq / Hkv); the oracle computes
that index map over the plain definition.  Tolerances as for decode: O within
1e-2 max-abs, LSE within 1e-3.
"""

import math

import numpy as np
import pytest

import oracle
from io_aware_exact_11_gb300 import fa, inputs
from tests.gpu_helpers import cpu64, max_abs, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.lib()
    yield
    fa.device_status()


def _run(seed, B, Hq, Hkv, N, splits, heads=None, d=128):
    hq = inputs.normal_tensor(seed, "q", B, Hq, 1, d, "bf16")
    hk = inputs.normal_tensor(seed, "k", B, Hkv, N, d, "bf16")
    hv = inputs.normal_tensor(seed, "v", B, Hkv, N, d, "bf16")
    q, k, v = to_device(hq, "bf16"), to_device(hk, "bf16"), to_device(hv, "bf16")
    scale = 1 / math.sqrt(d)
    o, lse = fa.decode_splitkv_gqa(q, k, v, n_splits=splits, scale=scale)
    fa.device_status()
    G = Hq // Hkv
    for b, h in heads or [(b, h) for b in range(B) for h in range(Hq)]:
        ro, rl = oracle.attention_forward(inputs.as_f64(hq[b, h], "bf16"), inputs.as_f64(hk[b, h // G], "bf16"),
                                          inputs.as_f64(hv[b, h // G], "bf16"), scale)
        assert max_abs(cpu64(o[b, h]), ro) <= 1e-2, (b, h)
        assert max_abs(cpu64(lse[b, h]), rl[0]) <= 1e-3, (b, h)
    return q, k, v, o, lse


@pytest.mark.parametrize("B,Hq,Hkv,N,splits", [
    (2, 28, 4, 1000, 32),    # group of 7 (the lab model's 28 query / 4 key-value heads)
    (1, 8, 1, 2048, 32),     # one key/value head for all (group of 8)
    (2, 6, 3, 777, 7),       # group of 2, ragged split
    (1, 4, 2, 20, 32),       # more splits than keys
    (2, 32, 2, 700, 4),      # group of 16
    (3, 32, 1, 1500, 8),     # multi-query attention: one key/value head for 32 query heads
    (2, 48, 1, 900, 4),      # group of 48: two softmax warps, the second half full
    (1, 71, 1, 1300, 8),     # group of 71: three softmax warps, a ragged last one
    (2, 128, 2, 640, 4),     # group of 64
    (1, 128, 1, 2000, 16),   # group of 128: all four TMEM lane quarters hold query rows
])
def test_gqa_decode_matches_oracle(B, Hq, Hkv, N, splits):
    _run(31, B, Hq, Hkv, N, splits)


@pytest.mark.parametrize("B,Hq,Hkv,N,splits", [(2, 28, 4, 1000, 32), (1, 64, 1, 1300, 8), (2, 6, 3, 777, 7)])
def test_gqa_decode_head_dim_64_matches_oracle(B, Hq, Hkv, N, splits):
    """d = 64: one 64-column block per tile, a ten-slot ring, N = 64 for P̃V."""
    _run(32, B, Hq, Hkv, N, splits, d=64)


def test_gqa_decode_with_group_one_equals_decode():
    import torch
    q, k, v, o, lse = _run(32, 2, 4, 4, 600, 32)
    o2, l2 = fa.decode_splitkv(q, k, v, n_splits=32)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


def test_gqa_decode_equals_decode_on_repeated_heads():
    """Same group computed two ways: shared K/V heads vs explicitly repeated ones."""
    import torch
    q, k, v, o, lse = _run(33, 1, 16, 2, 1500, 32, heads=[(0, 0)])
    o2, l2 = fa.decode_splitkv(q, k.repeat_interleave(8, dim=1).contiguous(), v.repeat_interleave(8, dim=1).contiguous(),
                               n_splits=32)
    assert float((o.float() - o2.float()).abs().max()) <= 2 ** -8
    assert float((lse - l2).abs().max()) <= 1e-5


@pytest.mark.slow
def test_gqa_decode_qwen_shape_full_size_sampled():
    """B=64, 28 query heads over 4 key/value heads, N_kv=8192, 32 splits."""
    _run(34, 64, 28, 4, 8192, 32, heads=[(0, 0), (0, 27), (63, 13), (31, 6), (17, 21)])
