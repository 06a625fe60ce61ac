"""fa_decode_splitkv_noalloc: the decode entry point that allocates nothing.

It exists for callers that cannot give the library device workspace when they
decode — a serving process whose KV cache already reserved the GPU's memory,
or a host program that only reaches this C function and has no device
allocator.  Its scratch is a fixed buffer compiled into libfa.so, shared by
every call.  These tests call it through the C ABI and through the Python
binding and check it three ways: against the float64 oracle within the decode
tolerance the other tests use, bit for bit against fa_decode_splitkv (caller
workspace; the same deterministic kernels run on the same inputs), and that
the device's free memory does not move across calls.  Calls come in a row with
different shapes, so stale scratch from one call cannot hide a fault in the
next, and the size limit is checked on both sides of its exact boundary.

This file is named to be collected last, so a fail-fast run has already run
every other test when it gets here; it also passes when run on its own.
"""

import ctypes
import math

import numpy as np
import pytest

import oracle
from io_aware_exact_11_gb300 import fa, inputs

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 1e-2, 1e-3


def _host(seed, name, B, H, N, d):
    return inputs.normal_tensor(seed, name, B, H, N, d, "bf16")


def _dev(x):
    import torch
    return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()


def _noalloc_fn():
    L = fa.lib()
    fn = L.fa_decode_splitkv_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp]
    fn.restype = i32
    return fn


def _call_noalloc(q, k, v, n_splits, o, lse):
    """The C entry point on caller-provided outputs (lse may be None)."""
    import torch
    B, H, _, d = q.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = _noalloc_fn()(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                       None if lse is None else lse.data_ptr(), B, H, k.shape[2], d, fa.FA_BF16,
                       1.0 / math.sqrt(d), n_splits, stream)
    assert rc == fa.FA_OK, fa.lib().fa_get_last_error()


def _oracle(qh, kh, vh, d):
    q, k, v = (inputs.as_f64(x, "bf16") for x in (qh, kh, vh))
    return oracle.attention_forward(q, k, v, 1.0 / math.sqrt(d))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.lib()


def test_noalloc_matches_oracle_and_workspace_path_on_calls_in_a_row():
    import torch
    # B, H, N_kv, n_splits, d, seed: different shapes back to back (the second
    # and third reuse the scratch the first one filled).
    cases = [(16, 32, 2048, 32, 128, 21), (2, 3, 1000, 7, 128, 22), (3, 5, 777, 9, 64, 23)]
    for n, (B, H, N, S, d, seed) in enumerate(cases):
        qh, kh, vh = _host(seed, "q", B, H, 1, d), _host(seed, "k", B, H, N, d), _host(seed, "v", B, H, N, d)
        q, k, v = _dev(qh), _dev(kh), _dev(vh)
        o_na = torch.empty_like(q)
        l_na = torch.empty((B, H), dtype=torch.float32, device="cuda")
        o_ws, l_ws = fa.decode_splitkv(q, k, v, n_splits=S)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        _call_noalloc(q, k, v, S, o_na, l_na)
        fa.device_status()
        free_after = torch.cuda.mem_get_info()[0]
        if n > 0:  # the first call may load the library's decode module (and its buffer)
            assert free_after == free_before, (free_before, free_after)
        # Bit for bit against the workspace entry point: same kernels, same inputs.
        assert torch.equal(o_na, o_ws) and torch.equal(l_na, l_ws), (B, H, N, S, d)
        ro, rl = _oracle(qh, kh, vh, d)
        eo = float(np.max(np.abs(o_na.float().cpu().numpy().astype(np.float64) - ro)))
        el = float(np.max(np.abs(l_na.cpu().numpy().astype(np.float64) - rl[..., 0])))
        assert eo <= TOL_O and el <= TOL_LSE, (B, H, N, S, d, eo, el)


def test_noalloc_python_binding_head_dim_64_and_without_lse():
    import torch
    B, H, N, S, d = 4, 6, 1500, 16, 64
    qh, kh, vh = _host(31, "q", B, H, 1, d), _host(31, "k", B, H, N, d), _host(31, "v", B, H, N, d)
    q, k, v = _dev(qh), _dev(kh), _dev(vh)
    o1, l1 = fa.decode_splitkv_noalloc(q, k, v, n_splits=S)
    o2, l2 = fa.decode_splitkv_noalloc(q, k, v, n_splits=S, return_lse=False)
    o_ws, l_ws = fa.decode_splitkv(q, k, v, n_splits=S)
    fa.device_status()
    assert l2 is None
    assert torch.equal(o1, o_ws) and torch.equal(l1, l_ws)
    assert torch.equal(o2, o_ws)
    ro, rl = _oracle(qh, kh, vh, d)
    assert float(np.max(np.abs(o2.float().cpu().numpy().astype(np.float64) - ro))) <= TOL_O


def test_noalloc_accepts_the_largest_request_and_rejects_one_more_head():
    import torch
    d, S = 128, 32
    limit = fa.DECODE_STATIC_SCRATCH_BYTES
    # B·H = 2268 heads with 32 splits is the largest head count that fits at d = 128.
    B, H, N = 84, 27, 256
    assert fa.decode_workspace_size(B, H, d, S) <= limit < fa.decode_workspace_size(1, B * H + 1, d, S)
    g = torch.Generator(device="cuda")
    g.manual_seed(41)
    q, k, v = (torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
               for s in ((B, H, 1, d), (B, H, N, d), (B, H, N, d)))
    o_na = torch.empty_like(q)
    l_na = torch.empty((B, H), dtype=torch.float32, device="cuda")
    _call_noalloc(q, k, v, S, o_na, l_na)
    o_ws, l_ws = fa.decode_splitkv(q, k, v, n_splits=S)
    fa.device_status()
    assert torch.equal(o_na, o_ws) and torch.equal(l_na, l_ws)
    del q, k, v, o_na, l_na, o_ws, l_ws
    # One more head: rejected before anything is enqueued.  The tensors have the
    # shape the call claims, so even a wrongly accepted call would stay in bounds.
    B2, H2, N2 = 1, B * H + 1, 16
    q = torch.zeros((B2, H2, 1, d), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((B2, H2, N2, d), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    before = fa.launch_count()
    rc = _noalloc_fn()(q.data_ptr(), kv.data_ptr(), kv.data_ptr(), o.data_ptr(), None, B2, H2, N2, d, fa.FA_BF16,
                       0.1, S, None)
    assert rc == fa.FA_ERR_UNSUPPORTED
    assert b"scratch" in fa.lib().fa_get_last_error()
    assert fa.launch_count() == before


def test_noalloc_rejects_sizes_far_beyond_its_buffer():
    import torch
    q = torch.zeros((512, 64, 1, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((512, 64, 16, 128), dtype=torch.bfloat16, device="cuda")
    need = fa.decode_workspace_size(512, 64, 128, 32)
    assert need > fa.DECODE_STATIC_SCRATCH_BYTES
    before = fa.launch_count()
    o = torch.empty_like(q)
    rc = _noalloc_fn()(q.data_ptr(), k.data_ptr(), k.data_ptr(), o.data_ptr(), None, 512, 64, 16, 128, fa.FA_BF16,
                       0.1, 32, None)
    assert rc == fa.FA_ERR_UNSUPPORTED
    assert b"scratch" in fa.lib().fa_get_last_error()
    assert fa.launch_count() == before
