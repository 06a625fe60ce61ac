"""GPU parity on shapes drawn at random (from a fixed seed) against the float64
oracle: combinations of batch, heads, ragged query and key lengths, head dim,
causal mask, split counts, group sizes and page sizes that the hand-picked
cases elsewhere do not pin one by one.

Tolerances are the fixed ones: O within 1e-2 max-abs and LSE within 1e-3 for
bf16 inputs with fp32 accumulation, gradients within 2e-2 relative L2.  Causal
rows that see only a handful of keys can have |O| close to max|V|, where the
bf16 output's own rounding alone exceeds 1e-2; there each element takes the
larger of 1e-2 and the bound derived from the two bf16 roundings (P̃ entering
P̃·V: 2^-8·(P|V|); storing O: 2^-8·|O|), as in the causal tests.
"""

import math

import numpy as np
import pytest

import oracle
from io_aware_exact_11_gb300 import fa, inputs
from tests.gpu_helpers import cpu64, f64, make_qkv, max_abs, rel_l2, to_device

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE, TOL_GRAD = 1e-2, 1e-3, 2e-2


def _draw(seed, n, fn):
    rng = np.random.default_rng(seed)
    return [fn(rng) for _ in range(n)]


def _fwd_case(rng):
    causal = bool(rng.integers(2))
    d = int(rng.choice([64, 128]))
    nq = int(rng.integers(1, 700))
    nkv = int(rng.integers(nq, 900)) if causal else int(rng.integers(1, 900))
    return (int(rng.integers(1, 4)), int(rng.integers(1, 5)), nq, nkv, d, causal)


def _bwd_case(rng):
    return (int(rng.integers(1, 3)), int(rng.integers(1, 4)), int(rng.integers(1, 400)),
            int(rng.choice([64, 128])), bool(rng.integers(2)))


def _dec_case(rng):
    hkv = int(rng.integers(1, 5))
    g = int(rng.choice([1, 1, 2, 4, 7, 16]))
    n = int(rng.integers(1, 3000))
    return (int(rng.integers(1, 5)), g * hkv, hkv, n, int(rng.integers(1, 65)), int(rng.choice([64, 128])))


def _paged_case(rng):
    hkv = int(rng.integers(1, 4))
    g = int(rng.choice([1, 1, 4, 8]))
    bs = int(rng.choice([16, 32, 64, 128]))
    B = int(rng.integers(1, 4))
    lens = [int(x) for x in rng.integers(1, 1500, size=B)]
    return (B, g * hkv, hkv, tuple(lens), bs, int(rng.integers(1, 17)), int(rng.choice([64, 128])))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.lib()
    yield
    fa.device_status()


@pytest.mark.parametrize("case", _draw(101, 12, _fwd_case), ids=str)
def test_random_forward(case):
    B, H, Nq, Nkv, d, causal = case
    host, dev = make_qkv(61, B, H, Nq, Nkv, d, "bf16")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward(dev["q"], dev["k"], dev["v"], scale, causal=causal)
    fa.device_status()
    q64, k64, v64 = (f64(host[n], "bf16") for n in ("q", "k", "v"))
    ro, rl = oracle.attention_forward(q64, k64, v64, scale, causal=causal)
    pv = np.stack([np.stack([oracle.attention_probs(q64[b, h], k64[b, h], scale, causal=causal) @ np.abs(v64[b, h])
                             for h in range(H)]) for b in range(B)])
    bound = np.maximum(TOL_O, 2.0 ** -8 * (pv + np.abs(ro)) + 1e-4)
    err = np.abs(cpu64(o) - ro)
    assert np.all(err <= bound), float(np.max(err - bound))
    assert max_abs(cpu64(lse), rl) <= TOL_LSE


@pytest.mark.parametrize("case", _draw(102, 8, _bwd_case), ids=str)
def test_random_backward(case):
    B, H, N, d, causal = case
    host, dev = make_qkv(62, B, H, N, N, d, "bf16", with_do=True)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward(dev["q"], dev["k"], dev["v"], scale, causal=causal)
    dq, dk, dv = fa.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], scale, causal=causal)
    fa.device_status()
    for b in range(B):
        for h in range(H):
            rq, rk, rv = oracle.attention_backward(*(f64(host[n][b, h], "bf16") for n in ("q", "k", "v", "do")),
                                                   scale, causal=causal)
            if N == 1:  # one key: the exact dQ and dK are zero, so only dV has a relative error
                assert rel_l2(cpu64(dv[b, h]), rv) <= TOL_GRAD
                continue
            e = (rel_l2(cpu64(dq[b, h]), rq), rel_l2(cpu64(dk[b, h]), rk), rel_l2(cpu64(dv[b, h]), rv))
            assert max(e) <= TOL_GRAD, ((b, h), e)


@pytest.mark.parametrize("case", _draw(103, 10, _dec_case), ids=str)
def test_random_decode(case):
    B, Hq, Hkv, N, splits, d = case
    qh = inputs.normal_tensor(63, "q", B, Hq, 1, d, "bf16")
    kh = inputs.normal_tensor(63, "k", B, Hkv, N, d, "bf16")
    vh = inputs.normal_tensor(63, "v", B, Hkv, N, d, "bf16")
    q, k, v = (to_device(x, "bf16") for x in (qh, kh, vh))
    scale = 1.0 / math.sqrt(d)
    if Hq == Hkv:
        o, lse = fa.decode_splitkv(q, k, v, n_splits=splits, scale=scale)
    else:
        o, lse = fa.decode_splitkv_gqa(q, k, v, n_splits=splits, scale=scale)
    fa.device_status()
    G = Hq // Hkv
    q64, k64, v64 = (f64(x, "bf16") for x in (qh, kh, vh))
    for b in range(B):
        for h in range(Hq):
            ro, rl = oracle.attention_forward(q64[b, h], k64[b, h // G], v64[b, h // G], scale)
            assert max_abs(cpu64(o[b, h]), ro) <= TOL_O, (b, h)
            assert abs(float(lse[b, h]) - float(rl[0])) <= TOL_LSE, (b, h)


@pytest.mark.parametrize("case", _draw(104, 8, _paged_case), ids=str)
def test_random_paged_decode(case):
    import torch
    B, Hq, Hkv, lens, bs, splits, d = case
    G = Hq // Hkv
    max_blocks = (max(lens) + bs - 1) // bs
    nb = B * max_blocks + 3
    qh = inputs.normal_tensor(64, "q", B, Hq, 1, d, "bf16")
    kh = inputs.normal_tensor(64, "k", 1, nb, Hkv * bs, d, "bf16")[0].reshape(nb, Hkv, bs, d)
    vh = inputs.normal_tensor(64, "v", 1, nb, Hkv * bs, d, "bf16")[0].reshape(nb, Hkv, bs, d)
    rng = np.random.default_rng(65)
    table = rng.permutation(nb)[:B * max_blocks].reshape(B, max_blocks).astype(np.int32)
    for b in range(B):  # entries past a sequence's pages are never read
        table[b, (lens[b] + bs - 1) // bs:] = -1
    q, kc, vc = (to_device(x, "bf16") for x in (qh, kh, vh))
    o, lse = fa.decode_paged(q, kc, vc, torch.from_numpy(table).cuda(), torch.tensor(lens, dtype=torch.int32).cuda(),
                             n_splits=splits, scale=1.0 / math.sqrt(d))
    fa.device_status()
    q64, k64, v64 = (f64(x, "bf16") for x in (qh, kh, vh))
    scale = 1.0 / math.sqrt(d)
    for b in range(B):
        pages = table[b, :(lens[b] + bs - 1) // bs]
        for h in range(Hq):
            kk = np.concatenate([k64[p, h // G] for p in pages])[:lens[b]]
            vv = np.concatenate([v64[p, h // G] for p in pages])[:lens[b]]
            ro, rl = oracle.attention_forward(q64[b, h], kk, vv, scale)
            assert max_abs(cpu64(o[b, h]), ro) <= TOL_O, (b, h)
            assert abs(float(lse[b, h]) - float(rl[0])) <= TOL_LSE, (b, h)
