"""fa_decode_splitkv_noalloc: the decode entry point that allocates nothing.

It exists for callers that cannot give the library device workspace when they
decode — a serving process whose KV cache already reserved the GPU's memory,
or a host program that only reaches this C function and has no device
allocator.  Its scratch is a fixed buffer compiled into libfa.so, shared by
every call.  These tests call it through the C ABI and compare it with
fa_decode_splitkv (caller workspace), within the decode tolerance used by the
other tests, on two calls in a row with different shapes so that stale scratch
from the first call cannot hide a fault in the second.

This file is named to be collected last, so a fail-fast run has already run
every other test when it gets here; it also passes when run on its own.
"""

import ctypes
import math

import numpy as np
import pytest

from io_aware_exact_11_gb300 import fa, inputs

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 1e-2, 1e-3


def _dev(seed, name, B, H, N, d):
    import torch
    x = inputs.normal_tensor(seed, name, B, H, N, d, "bf16")
    return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()


def _noalloc_fn():
    L = fa.lib()
    fn = L.fa_decode_splitkv_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp]
    fn.restype = i32
    return fn


def _call_noalloc(q, k, v, n_splits):
    import torch
    B, H, _, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = _noalloc_fn()(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, k.shape[2], d,
                       fa.FA_BF16, 1.0 / math.sqrt(d), n_splits, stream)
    assert rc == fa.FA_OK, fa.lib().fa_get_last_error()
    return o, lse


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.lib()


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import torch
    cases = [(16, 32, 2048, 32, 21), (2, 3, 1000, 7, 22)]   # B, H, N_kv, n_splits, seed
    for B, H, N, S, seed in cases:
        q = _dev(seed, "q", B, H, 1, 128)
        k = _dev(seed, "k", B, H, N, 128)
        v = _dev(seed, "v", B, H, N, 128)
        o_na, l_na = _call_noalloc(q, k, v, S)
        o_ws, l_ws = fa.decode_splitkv(q, k, v, n_splits=S)
        fa.device_status()
        eo = float((o_na.float() - o_ws.float()).abs().max())
        el = float((l_na - l_ws).abs().max())
        assert eo <= TOL_O and el <= TOL_LSE, (B, H, N, S, eo, el)
        assert bool(torch.isfinite(o_na.float()).all())


def test_noalloc_rejects_sizes_beyond_its_buffer():
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
