"""GPU parity: the CUDA kernels against the float64 oracle on seeded inputs.

Tolerances (fixed for this method): bf16 inputs with fp32 accumulation give
O within 1e-2 max-abs and LSE within 1e-3; the fp32 path gives both within
1e-5; gradients dQ, dK, dV within 2e-2 relative L2.
"""

import math

import numpy as np
import pytest

import oracle
from io_aware_exact_11_gb300 import fa, inputs
from tests.gpu_helpers import cpu64, f64, make_qkv, max_abs, rel_l2, to_device

pytestmark = pytest.mark.gpu

TOL_O_BF16, TOL_LSE_BF16 = 1e-2, 1e-3
TOL_FP32 = 1e-5
TOL_GRAD = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.lib()
    yield
    fa.device_status()


def _fwd_check(seed, B, H, Nq, Nkv, d, dtype, tol_o, tol_lse):
    host, dev = make_qkv(seed, B, H, Nq, Nkv, d, dtype)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward(dev["q"], dev["k"], dev["v"], scale)
    fa.device_status()
    ref_o, ref_lse = oracle.attention_forward(f64(host["q"], dtype), f64(host["k"], dtype),
                                              f64(host["v"], dtype), scale)
    eo, el = max_abs(cpu64(o), ref_o), max_abs(cpu64(lse), ref_lse)
    assert eo <= tol_o and el <= tol_lse, (eo, el)
    return eo, el


def test_tiny_fp32_exact():
    """B=1, H=1, N=256, d=64, fp32 N(0,1), scale 1/8, no mask."""
    _fwd_check(0, 1, 1, 256, 256, 64, "fp32", TOL_FP32, TOL_FP32)


@pytest.mark.parametrize("shape", [(2, 2, 100, 77, 128), (1, 1, 1, 1, 64), (1, 3, 33, 300, 128)])
def test_fp32_ragged(shape):
    B, H, Nq, Nkv, d = shape
    _fwd_check(11, B, H, Nq, Nkv, d, "fp32", TOL_FP32, TOL_FP32)


@pytest.mark.parametrize("shape", [
    (1, 2, 256, 256, 128),    # two full tiles each way
    (2, 3, 300, 277, 128),    # ragged query and key tails
    (1, 2, 384, 512, 128),    # N_q != N_kv
    (1, 1, 128, 1, 128),      # a single key: O = v
    (1, 2, 1, 130, 128),      # a single query row
    (1, 2, 640, 1000, 64),    # head dim 64
    (1, 1, 129, 129, 128),    # one row / one key past a tile boundary
])
def test_forward_bf16_matches_oracle(shape):
    B, H, Nq, Nkv, d = shape
    _fwd_check(1, B, H, Nq, Nkv, d, "bf16", TOL_O_BF16, TOL_LSE_BF16)


@pytest.mark.parametrize("shape", [
    (3, 70, 200, 300, 128),   # 210 work items: some CTAs run a second item; ragged rows and keys
    (2, 100, 600, 130, 64),   # 600 items of two key tiles each, head dim 64
    (4, 50, 256, 100, 128),   # 200 items of a single (ragged) key tile
])
def test_forward_bf16_many_blocks(shape):
    """More 256-row query blocks than SMs, so the grid runs in several waves
    (and, for the 200-row case, every block has a ragged row tail)."""
    B, H, Nq, Nkv, d = shape
    _fwd_check(3, B, H, Nq, Nkv, d, "bf16", TOL_O_BF16, TOL_LSE_BF16)


def test_forward_bf16_large_scores():
    """Scores with standard deviation ~6 exercise the running-max rescale.

    Bound derived from the arithmetic rather than the N(0,1) tolerance.  bf16
    keeps 8 significant bits, so one rounding has relative error <= 2^-8: the
    probabilities enter P·V rounded to bf16 (at most 2^-8·max|V| in O) and O is
    stored as bf16 (<= 2^-8·|O|).  With peaked rows |O| approaches max|V|, so the
    bound is 2^-7·max|V| plus fp32 noise.  LSE is fp32 throughout: its error
    scales with its magnitude (~1e-6 relative).
    """
    import torch
    B, H, N, d = 1, 2, 512, 128
    host, dev = make_qkv(5, B, H, N, N, d, "bf16")
    q = (dev["q"].float() * 6).to(torch.bfloat16)
    o, lse = fa.forward(q, dev["k"], dev["v"])
    v64 = f64(host["v"], "bf16")
    ref_o, ref_lse = oracle.attention_forward(cpu64(q), f64(host["k"], "bf16"), v64, 1 / math.sqrt(d))
    assert max_abs(cpu64(o), ref_o) <= 2.0 ** -7 * float(np.abs(v64).max()) + 1e-3
    assert max_abs(cpu64(lse), ref_lse) <= TOL_LSE_BF16 * max(1.0, float(np.abs(ref_lse).max()) / 8)


@pytest.mark.parametrize("d,causal", [(128, False), (64, False), (128, True)])
def test_forward_bf16_rising_scores_rescale_mid_sequence(d, causal):
    """Key magnitudes ramp from 1x to 5x along the sequence, so rows move their
    reference max (by more than 2^8 in base 2) in later key tiles and O is
    rescaled in TMEM mid-sequence.  A CPU check first confirms that the data
    triggers such rescales; the bound is the one derived for large scores."""
    import torch
    B, H, N = 1, 2, 1024
    host, dev = make_qkv(6, B, H, N, N, d, "bf16")
    ramp = torch.linspace(1.0, 5.0, N, device="cuda").view(1, 1, N, 1)
    k = (dev["k"].float() * ramp).to(torch.bfloat16)
    k64 = cpu64(k)
    q64 = f64(host["q"], "bf16")
    scale = 1 / math.sqrt(d)
    s2 = scale * math.log2(math.e) * np.einsum("bhqd,bhkd->bhqk", q64, k64)
    if causal:
        s2 = np.where(oracle.causal_visible(np.arange(N), N, N)[None, None], s2, -np.inf)
    tile_max = s2.reshape(B, H, N, N // 128, 128).max(axis=-1)
    m_ref = tile_max[..., 0]
    rescales = 0
    for j in range(1, N // 128):
        moved = tile_max[..., j] > m_ref + 8.0
        rescales += int(moved.sum())
        m_ref = np.where(moved, tile_max[..., j], m_ref)
    assert rescales >= N // 2, rescales
    o, lse = fa.forward(dev["q"], k, dev["v"], causal=causal)
    fa.device_status()
    v64 = f64(host["v"], "bf16")
    for h in range(H):
        ref_o, ref_lse = oracle.attention_rows(q64[0, h], k64[0, h], v64[0, h], scale, np.arange(N), causal=causal)
        assert max_abs(cpu64(o[0, h]), ref_o) <= 2.0 ** -7 * float(np.abs(v64).max()) + 1e-3, h
        assert max_abs(cpu64(lse[0, h]), ref_lse) <= TOL_LSE_BF16 * max(1.0, float(np.abs(ref_lse).max()) / 8), h


@pytest.mark.parametrize("d", [64, 128])
def test_forward_strided_inputs(d):
    """Q/K/V/O as [B, N, H, d] buffers viewed as [B, H, N, d] (at d = 64 the
    four-query-tile kernel, whose O leaves by direct stores through the strides)."""
    import torch
    B, H, N = 2, 3, 256
    host, dev = make_qkv(3, B, H, N, N, d, "bf16")
    qs, ks, vs = (dev[n].transpose(1, 2).contiguous().transpose(1, 2) for n in ("q", "k", "v"))
    assert not qs.is_contiguous()
    out = torch.empty((B, N, H, d), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    o, lse = fa.forward(qs, ks, vs, out=out)
    o_ref, lse_ref = fa.forward(dev["q"], dev["k"], dev["v"])
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


@pytest.mark.parametrize("d", [64, 128])
def test_forward_deterministic(d):
    import torch
    _, dev = make_qkv(2, 1, 4, 512, 512, d, "bf16")
    o1, l1 = fa.forward(dev["q"], dev["k"], dev["v"])
    o2, l2 = fa.forward(dev["q"], dev["k"], dev["v"])
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [64, 128])
def test_values_all_ones_give_ones(d):
    import torch
    B, H, N = 1, 2, 300
    _, dev = make_qkv(4, B, H, N, N, d, "bf16")
    ones = torch.ones_like(dev["v"])
    o, _ = fa.forward(dev["q"], dev["k"], ones)
    assert torch.all(o == 1)


@pytest.mark.slow
def test_prefill_full_size_sampled():
    """B=4, H=32, N=4096, d=128 bf16: two whole heads and 64 sampled rows of 8 more."""
    B, H, N, d = 4, 32, 4096, 128
    host, dev = make_qkv(1, B, H, N, N, d, "bf16")
    scale = 1 / math.sqrt(d)
    o, lse = fa.forward(dev["q"], dev["k"], dev["v"], scale)
    fa.device_status()
    rng = np.random.default_rng(7)
    heads = [(0, 0), (3, 31)] + [(int(rng.integers(B)), int(rng.integers(H))) for _ in range(8)]
    for n, (b, h) in enumerate(heads):
        rows = np.arange(N) if n < 2 else np.sort(rng.choice(N, 64, replace=False))
        ro, rl = oracle.attention_rows(f64(host["q"][b, h], "bf16"), f64(host["k"][b, h], "bf16"),
                                       f64(host["v"][b, h], "bf16"), scale, rows)
        assert max_abs(cpu64(o[b, h])[rows], ro) <= TOL_O_BF16
        assert max_abs(cpu64(lse[b, h])[rows], rl) <= TOL_LSE_BF16
    assert bool(o.isfinite().all()) and bool(lse.isfinite().all())


@pytest.mark.slow
def test_long_context_sampled_and_linear_memory():
    """B=1, H=32, N=32768, d=128: sampled rows, and no O(N²) buffer anywhere."""
    import torch
    B, H, N, d = 1, 32, 32768, 128
    host, dev = make_qkv(2, B, H, N, N, d, "bf16")
    o = torch.empty_like(dev["q"])
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    fa.forward(dev["q"], dev["k"], dev["v"], out=o, lse=lse)
    torch.cuda.synchronize()
    fa.device_status()
    assert torch.cuda.max_memory_allocated() - base == 0     # the library allocates nothing
    rng = np.random.default_rng(9)
    scale = 1 / math.sqrt(d)
    for h in (0, 17, 31):
        rows = np.concatenate([[0, N - 1], np.sort(rng.choice(N, 30, replace=False))])
        ro, rl = oracle.attention_rows(f64(host["q"][0, h], "bf16"), f64(host["k"][0, h], "bf16"),
                                       f64(host["v"][0, h], "bf16"), scale, rows)
        assert max_abs(cpu64(o[0, h])[rows], ro) <= TOL_O_BF16
        assert max_abs(cpu64(lse[0, h])[rows], rl) <= TOL_LSE_BF16


# ----------------------------------------------------------------- decode


def _decode_check(seed, B, H, N, n_splits, heads=None, d=128):
    host, dev = make_qkv(seed, B, H, 1, N, d, "bf16")
    scale = 1 / math.sqrt(d)
    o, lse = fa.decode_splitkv(dev["q"], dev["k"], dev["v"], n_splits=n_splits, scale=scale)
    fa.device_status()
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads:
        ro, rl = oracle.attention_forward(f64(host["q"][b, h], "bf16"), f64(host["k"][b, h], "bf16"),
                                          f64(host["v"][b, h], "bf16"), scale)
        assert max_abs(cpu64(o[b, h]), ro) <= TOL_O_BF16, (b, h)
        assert max_abs(cpu64(lse[b, h]), rl[0]) <= TOL_LSE_BF16, (b, h)
    return o, lse


@pytest.mark.parametrize("B,H,N,splits", [(2, 3, 1000, 32), (1, 2, 8192, 32), (2, 2, 777, 7), (1, 1, 300, 1),
                                          (1, 2, 20, 32), (1, 1, 1, 4), (1, 1, 4096, 256)])
def test_decode_matches_oracle(B, H, N, splits):
    _decode_check(3, B, H, N, splits)


@pytest.mark.parametrize("B,H,N,splits", [(2, 3, 1000, 32), (1, 2, 777, 7), (1, 1, 1, 4)])
def test_decode_head_dim_64_matches_oracle(B, H, N, splits):
    """d = 64: eight lanes per key, four keys per warp step, sixteen P·V groups."""
    _decode_check(4, B, H, N, splits, d=64)


def test_decode_matches_forward_kernel():
    """Decode and the prefill kernel with N_q = 1 compute the same function."""
    _, dev = make_qkv(8, 2, 4, 1, 2048, 128, "bf16")
    o1, l1 = fa.decode_splitkv(dev["q"], dev["k"], dev["v"], n_splits=32)
    o2, l2 = fa.forward(dev["q"], dev["k"], dev["v"])
    assert max_abs(cpu64(o1), cpu64(o2)) <= TOL_O_BF16
    assert max_abs(cpu64(l1), cpu64(l2)[..., 0]) <= TOL_LSE_BF16


@pytest.mark.slow
def test_decode_full_size_sampled():
    """B=64, H=32, one query row per head, N_kv=8192, d=128, 32 splits."""
    import torch
    o, lse = _decode_check(4, 64, 32, 8192, 32, heads=[(0, 0), (63, 31), (17, 5), (40, 20), (5, 30), (33, 1)])
    assert bool(o.isfinite().all()) and bool(lse.isfinite().all())
    del o, lse
    torch.cuda.empty_cache()


# --------------------------------------------------------------- backward


def _bwd_check(seed, B, H, N, heads=None, d=128):
    host, dev = make_qkv(seed, B, H, N, N, d, "bf16", with_do=True)
    scale = 1 / math.sqrt(d)
    o, lse = fa.forward(dev["q"], dev["k"], dev["v"], scale)
    dq, dk, dv = fa.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], scale)
    fa.device_status()
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    errs = []
    for b, h in heads:
        rq, rk, rv = oracle.attention_backward(*(f64(host[n][b, h], "bf16") for n in ("q", "k", "v", "do")),
                                               scale)
        e = (rel_l2(cpu64(dq[b, h]), rq), rel_l2(cpu64(dk[b, h]), rk), rel_l2(cpu64(dv[b, h]), rv))
        errs.append(e)
        assert max(e) <= TOL_GRAD, ((b, h), e)
    return errs


@pytest.mark.parametrize("B,H,N", [
    (1, 2, 128), (1, 2, 256), (2, 1, 640),
    (1, 2, 300),      # ragged last key and query tile
    (2, 1, 1000),
    (1, 3, 129),      # one key / query past a tile boundary
])
def test_backward_matches_oracle(B, H, N):
    _bwd_check(6, B, H, N)


@pytest.mark.parametrize("B,H,N", [(1, 2, 256), (1, 2, 300), (2, 1, 129)])
def test_backward_head_dim_64_matches_oracle(B, H, N):
    """d = 64: K's unused head-dim block is zeroed in shared memory so dQᵀ keeps
    its 128-row MMA; only the drain warps of head dims 0..63 reduce."""
    _bwd_check(7, B, H, N, d=64)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_single_key_degenerate(d):
    """N = 1: P = 1, so O = V, D = dO·V = dP and dS = P∘(dP − D) = 0 exactly;
    the exact dQ and dK are zero and dV = dO.  The kernel forms dP with the MMA
    and D with a separate fp32 sum of the same exact bf16 products, so dP − D
    is only summation-order rounding: at most d additions per side, each off by
    ≤ 2⁻²⁴ of the running magnitude (2⁻²³ allowed for the tensor core, whose
    accumulator may truncate), so |dP − D| ≤ 3·d·2⁻²⁴·Σ_t|dO_t V_t|.  Then
    |dQ_t| ≤ σ·|dS|·|K_t| (and |dK_t| likewise with Q_t) up to two bf16 roundings."""
    import torch
    B, H, N = 2, 3, 1
    host, dev = make_qkv(8, B, H, N, N, d, "bf16", with_do=True)
    scale = 1 / math.sqrt(d)
    o, lse = fa.forward(dev["q"], dev["k"], dev["v"], scale)
    dq, dk, dv = fa.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], scale)
    fa.device_status()
    assert torch.equal(dv, dev["do"])
    for b in range(B):
        for h in range(H):
            q, k, v, do = (f64(host[n][b, h], "bf16")[0] for n in ("q", "k", "v", "do"))
            gamma = 3 * d * 2.0 ** -24 * float(np.abs(do * v).sum())
            assert float(np.abs(cpu64(dq[b, h])).max()) <= 1.01 * scale * gamma * float(np.abs(k).max())
            assert float(np.abs(cpu64(dk[b, h])).max()) <= 1.01 * scale * gamma * float(np.abs(q).max())


@pytest.mark.slow
def test_backward_train_full_size_sampled():
    """B=2, H=16, N=8192, d=128: two whole heads against the oracle."""
    _bwd_check(5, 2, 16, 8192, heads=[(0, 0), (1, 15)])


# ------------------------------------------------------------ plumbing


def test_unsupported_shapes_raise_without_launching():
    import torch
    before = fa.launch_count()
    x = torch.zeros((1, 1, 16, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as ei:
        fa.forward(x, x, x)
    assert ei.value.status == fa.FA_ERR_UNSUPPORTED
    y = torch.zeros((1, 1, 200, 128), dtype=torch.float32, device="cuda")   # backward is built for bf16 only
    with pytest.raises(fa.FAError) as ei:
        fa.backward(y, y, y, y, torch.zeros((1, 1, 200), device="cuda"), y)
    assert ei.value.status == fa.FA_ERR_UNSUPPORTED
    assert fa.launch_count() == before


def test_launch_count_and_status():
    _, dev = make_qkv(0, 1, 1, 128, 128, 128, "bf16")
    before = fa.launch_count()
    fa.forward(dev["q"], dev["k"], dev["v"])
    fa.device_status()
    assert fa.launch_count() == before + 1
