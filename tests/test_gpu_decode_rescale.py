"""Decode with a rising running max: splits rescale mid-range.

Key magnitudes ramp from 1x to 9x along the sequence, so within each of two
splits a query row's tile maxima (nearly always) climb by more than 2^8 in
base 2, and the kernels rescale their partial (m, ℓ, o) on the way: the
single-head CUDA-core split kernel, the grouped tensor-core kernel, and both
over a paged cache (the grouped one in its one-box-per-page layout).  A CPU
check first confirms the rise in at least three of four (row, split) pairs.
Results are then held to the large-score bound: bf16 P̃ and bf16 O each round
with relative error <= 2^-8, so O is within 2^-7·max|V| plus fp32 noise; LSE
is within 1e-3 scaled by its magnitude.
"""

import math

import numpy as np
import pytest

import oracle
from io_aware_exact_11_gb300 import fa, inputs
from tests.gpu_helpers import cpu64, max_abs, to_device

pytestmark = pytest.mark.gpu

N, D, SPLITS = 2048, 128, 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.lib()
    yield
    fa.device_status()


def _inputs(seed, B, Hq, Hkv):
    """bf16 q [B,Hq,1,d], k and v [B,Hkv,N,d] with k ramped along the keys, as float64 and device tensors."""
    import torch
    q = to_device(inputs.normal_tensor(seed, "q", B, Hq, 1, D, "bf16"), "bf16")
    k0 = to_device(inputs.normal_tensor(seed, "k", B, Hkv, N, D, "bf16"), "bf16")
    v = to_device(inputs.normal_tensor(seed, "v", B, Hkv, N, D, "bf16"), "bf16")
    ramp = torch.linspace(1.0, 9.0, N, device="cuda").view(1, 1, N, 1)
    k = (k0.float() * ramp).to(torch.bfloat16)
    return q, k, v, cpu64(q), cpu64(k), cpu64(v)


def _assert_rises(q64, k64, G):
    """In most (row, split) pairs some 128-key tile max exceeds the split's first
    tile max by more than 8 (base 2), so the rescale path runs."""
    scale2 = math.log2(math.e) / math.sqrt(D)
    B, Hq = q64.shape[:2]
    per = N // SPLITS
    rising = 0
    for b in range(B):
        for h in range(Hq):
            s2 = scale2 * (k64[b, h // G] @ q64[b, h, 0])
            for c in range(SPLITS):
                t = s2[c * per:(c + 1) * per].reshape(-1, 128).max(axis=1)
                rising += int(t.max() > t[0] + 8.0)
    assert rising >= (3 * B * Hq * SPLITS) // 4, rising


def _check(o, lse, q64, k64, v64, G):
    scale = 1 / math.sqrt(D)
    B, Hq = q64.shape[:2]
    bound = 2.0 ** -7 * float(np.abs(v64).max()) + 1e-3
    for b in range(B):
        for h in range(Hq):
            ro, rl = oracle.attention_forward(q64[b, h], k64[b, h // G], v64[b, h // G], scale)
            assert max_abs(cpu64(o[b, h]), ro) <= bound, (b, h)
            assert abs(float(lse[b, h]) - float(rl[0])) <= 1e-3 * max(1.0, abs(float(rl[0])) / 8), (b, h)


def _pages(k, v, bs, seed):
    """Scatter contiguous [B,H,N,d] K/V into shuffled bs-key pages; returns caches, table, lengths."""
    import torch
    B, H = k.shape[:2]
    per = N // bs
    order = np.random.default_rng(seed).permutation(B * per).astype(np.int32).reshape(B, per)
    kc = torch.empty((B * per, H, bs, D), dtype=k.dtype, device="cuda")
    vc = torch.empty_like(kc)
    for b in range(B):
        for i in range(per):
            kc[int(order[b, i])] = k[b, :, i * bs:(i + 1) * bs]
            vc[int(order[b, i])] = v[b, :, i * bs:(i + 1) * bs]
    table = torch.from_numpy(order).cuda()
    lens = torch.full((B,), N, dtype=torch.int32, device="cuda")
    return kc, vc, table, lens


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
def test_decode_rising_scores_rescale(Hq, Hkv):
    q, k, v, q64, k64, v64 = _inputs(61, 2, Hq, Hkv)
    G = Hq // Hkv
    _assert_rises(q64, k64, G)
    dec = fa.decode_splitkv if G == 1 else fa.decode_splitkv_gqa
    o, lse = dec(q, k, v, n_splits=SPLITS)
    fa.device_status()
    _check(o, lse, q64, k64, v64, G)


@pytest.mark.parametrize("Hq,Hkv,bs", [(4, 4, 16), (8, 2, 16), (8, 2, 64)])
def test_paged_decode_rising_scores_rescale(Hq, Hkv, bs):
    q, k, v, q64, k64, v64 = _inputs(62, 2, Hq, Hkv)
    G = Hq // Hkv
    _assert_rises(q64, k64, G)
    kc, vc, table, lens = _pages(k, v, bs, 62)
    o, lse = fa.decode_paged(q, kc, vc, table, lens, n_splits=SPLITS)
    fa.device_status()
    _check(o, lse, q64, k64, v64, G)
