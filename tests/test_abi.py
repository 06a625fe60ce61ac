"""C-ABI checks that need no GPU: the library loads, exports every function
include/fa.h declares, and rejects bad arguments before touching CUDA."""

import ctypes
import os
import re

import pytest

from io_aware_exact_11_gb300 import fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(fa.LIB_PATH):
        from io_aware_exact_11_gb300 import build
        build.build()
    return fa.lib()


def test_header_declares_expected_entry_points():
    assert set(_declared()) == set(fa.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    assert L.fa_abi_version() == 1
    for s in range(5):
        assert L.fa_status_string(s)
    assert L.fa_status_string(99) == b"unknown status"


def test_workspace_sizes(L):
    assert L.fa_decode_workspace_size(64, 32, 128, 32) == 64 * 32 * 32 * 128 * 4 + 64 * 32 * 32 * 2 * 4
    assert L.fa_decode_workspace_size(1, 1, 128, 3) == 1536 + 256
    assert L.fa_decode_workspace_size(0, 1, 128, 3) == 0
    rows = 2 * 16 * 8192
    assert L.fa_backward_workspace_size(2, 16, 8192, 128) == rows * 128 * 4 + 2 * rows * 4
    assert L.fa_backward_workspace_size(1, 1, 5, 128) == 2560 + 2 * 256


FAKE = ctypes.c_void_p(1 << 20)        # never dereferenced: validation fails first
FAKE_BAD = ctypes.c_void_p((1 << 20) + 4)


def _fwd(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, H=1, Nq=128, Nkv=128, d=128, dt=fa.FA_BF16,
             scale=0.1, strides=None, stream=None)
    a.update(kw)
    return L.fa_forward(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nkv"], a["d"],
                        a["dt"], a["scale"], a["strides"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nkv=-3), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(dt=7), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(k=FAKE_BAD), fa.FA_ERR_INVALID_ARG),
    (dict(H=70000), fa.FA_ERR_UNSUPPORTED),
])
def test_forward_rejects_bad_arguments(L, kw, status):
    assert _fwd(L, **kw) == status
    assert L.fa_get_last_error()


def test_forward_rejects_bad_strides(L):
    st = (ctypes.c_int64 * 12)(*([128 * 128, 128 * 128, 128] * 3 + [128 * 128, 128 * 128, 100]))
    assert _fwd(L, strides=ctypes.cast(st, ctypes.c_void_p)) == fa.FA_ERR_INVALID_ARG
    assert b"stride" in L.fa_get_last_error()
    st2 = (ctypes.c_int64 * 12)(*([128 * 128, 128 * 128, 64] * 4))
    assert _fwd(L, strides=ctypes.cast(st2, ctypes.c_void_p)) == fa.FA_ERR_INVALID_ARG


def test_decode_rejects_bad_arguments(L):
    def dec(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=2, H=2, N=256, d=128, dt=fa.FA_BF16, scale=0.1,
                 ns=4, ws=FAKE, wsb=1 << 20, stream=None)
        a.update(kw)
        return L.fa_decode_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"],
                                   a["dt"], a["scale"], a["ns"], a["ws"], a["wsb"], a["stream"])
    assert dec(ws=None) == fa.FA_ERR_INVALID_ARG
    assert dec(wsb=100) == fa.FA_ERR_INVALID_ARG
    assert b"workspace" in L.fa_get_last_error()
    assert dec(d=96) == fa.FA_ERR_UNSUPPORTED
    assert dec(dt=fa.FA_FP32) == fa.FA_ERR_UNSUPPORTED
    assert dec(ns=0) == fa.FA_ERR_INVALID_ARG
    assert dec(ns=257) == fa.FA_ERR_UNSUPPORTED
    assert dec(N=0) == fa.FA_ERR_INVALID_ARG
    assert dec(q=FAKE_BAD) == fa.FA_ERR_INVALID_ARG


def test_backward_rejects_bad_arguments(L):
    def bwd(**kw):
        a = dict(B=1, H=1, N=256, d=128, dt=fa.FA_BF16, scale=0.1, ws=FAKE, wsb=1 << 24)
        a.update(kw)
        return L.fa_backward(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["B"], a["H"], a["N"], a["d"],
                             a["dt"], a["scale"], a["ws"], a["wsb"], None)
    assert bwd(N=0) == fa.FA_ERR_INVALID_ARG
    assert bwd(d=96) == fa.FA_ERR_UNSUPPORTED
    assert bwd(dt=fa.FA_FP32) == fa.FA_ERR_UNSUPPORTED
    assert bwd(wsb=10) == fa.FA_ERR_INVALID_ARG
    assert bwd(scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert bwd(ws=None) == fa.FA_ERR_INVALID_ARG


def test_masked_entry_points_validate_before_cuda(L):
    def fwdm(mask=fa.FA_MASK_CAUSAL, nq=128, nkv=128):
        return L.fa_forward_masked(FAKE, FAKE, FAKE, FAKE, None, 1, 1, nq, nkv, 128, fa.FA_BF16, 0.1, None, mask,
                                   None)
    assert fwdm(mask=5) == fa.FA_ERR_INVALID_ARG
    assert fwdm(nq=200, nkv=100) == fa.FA_ERR_INVALID_ARG      # causal needs N_q <= N_kv
    assert b"causal" in L.fa_get_last_error()
    # The causal grid holds at most 65535 blocks of 256 query rows.
    big = 65535 * 256 + 1
    assert fwdm(nq=big, nkv=big) == fa.FA_ERR_UNSUPPORTED

    def bwdm(mask=fa.FA_MASK_CAUSAL, n=200):
        return L.fa_backward_masked(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, n, 128, fa.FA_BF16,
                                    0.1, FAKE, 1 << 24, mask, None)
    assert bwdm(mask=-1) == fa.FA_ERR_INVALID_ARG
    assert bwdm(n=0) == fa.FA_ERR_INVALID_ARG
    assert bwdm(n=65535 * 128 + 1) == fa.FA_ERR_UNSUPPORTED   # the causal grid holds 65535 key tiles


def test_gqa_decode_validates_before_cuda(L):
    def dec(Hq=28, Hkv=4, d=128, wsb=1 << 24):
        return L.fa_decode_splitkv_gqa(FAKE, FAKE, FAKE, FAKE, None, 2, Hq, Hkv, 300, d, fa.FA_BF16, 0.1, 32, FAKE,
                                       wsb, None)
    assert dec(Hq=28, Hkv=5) == fa.FA_ERR_INVALID_ARG          # not a multiple
    assert dec(Hq=516, Hkv=4) == fa.FA_ERR_UNSUPPORTED         # group of 129
    assert dec(d=96) == fa.FA_ERR_UNSUPPORTED
    assert dec(wsb=64) == fa.FA_ERR_INVALID_ARG
    assert b"workspace" in L.fa_get_last_error()


def test_paged_decode_validates_before_cuda(L):
    def dec(bs=16, Hq=28, Hkv=4, d=128, wsb=1 << 24, table=FAKE, nb=100):
        return L.fa_decode_paged(FAKE, FAKE, FAKE, table, FAKE, FAKE, None, 2, Hq, Hkv, nb, bs, 64, d, fa.FA_BF16,
                                 0.1, 8, FAKE, wsb, None)
    assert dec(bs=24) == fa.FA_ERR_UNSUPPORTED
    assert dec(bs=256) == fa.FA_ERR_UNSUPPORTED
    assert dec(Hq=30) == fa.FA_ERR_INVALID_ARG
    assert dec(Hq=516) == fa.FA_ERR_UNSUPPORTED                # group of 129
    assert dec(table=None) == fa.FA_ERR_INVALID_ARG
    assert dec(wsb=16) == fa.FA_ERR_INVALID_ARG
    assert dec(d=96) == fa.FA_ERR_UNSUPPORTED
    assert dec(nb=1 << 30) == fa.FA_ERR_UNSUPPORTED              # page·H_kv + head past a 32-bit coordinate
    assert b"num_blocks" in L.fa_get_last_error()


def test_host_forward_workspace_size(L):
    # 3 heads of N_q=100, N_kv=300, d=128 bf16: q 76800 B, k and v 230400 B each, o 76800 B,
    # lse 1200 B -> 1280 B (each piece rounded up to 256 bytes); two chunk buffers.
    per_chunk = 76800 + 2 * 230400 + 76800 + 1280
    assert L.fa_forward_host_workspace_size(2, 4, 100, 300, 128, fa.FA_BF16, 3) == 2 * per_chunk
    # A chunk larger than B·H is clamped to B·H heads.
    assert (L.fa_forward_host_workspace_size(1, 2, 64, 64, 64, fa.FA_FP32, 50)
            == L.fa_forward_host_workspace_size(1, 2, 64, 64, 64, fa.FA_FP32, 2))
    assert L.fa_forward_host_workspace_size(0, 2, 64, 64, 64, fa.FA_BF16, 1) == 0
    assert L.fa_forward_host_workspace_size(1, 2, 64, 64, 64, 9, 1) == 0
    assert L.fa_forward_host_workspace_size(1, 2, 64, 64, 64, fa.FA_BF16, -1) == 0


def test_host_forward_validates_before_cuda(L):
    def fh(q=FAKE, ws=FAKE, B=2, H=3, nq=128, nkv=128, d=128, dt=fa.FA_BF16, scale=0.1, mask=fa.FA_MASK_NONE,
           hpc=2, wsb=1 << 30):
        return L.fa_forward_host(q, FAKE, FAKE, FAKE, None, B, H, nq, nkv, d, dt, scale, mask, hpc, ws, wsb, None)
    assert fh(q=None) == fa.FA_ERR_INVALID_ARG
    assert fh(ws=None) == fa.FA_ERR_INVALID_ARG
    assert fh(B=0) == fa.FA_ERR_INVALID_ARG
    assert fh(dt=7) == fa.FA_ERR_INVALID_ARG
    assert fh(mask=3) == fa.FA_ERR_INVALID_ARG
    assert fh(d=96) == fa.FA_ERR_UNSUPPORTED
    assert fh(scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert fh(mask=fa.FA_MASK_CAUSAL, nq=200, nkv=100) == fa.FA_ERR_INVALID_ARG
    assert fh(hpc=-1) == fa.FA_ERR_INVALID_ARG
    assert fh(ws=FAKE_BAD) == fa.FA_ERR_INVALID_ARG
    need = L.fa_forward_host_workspace_size(2, 3, 128, 128, 128, fa.FA_BF16, 2)
    assert fh(wsb=need - 1) == fa.FA_ERR_INVALID_ARG
    assert b"workspace" in L.fa_get_last_error()


def test_decode_split_choice(L):
    # No device here: the choice is made for 152 SMs.  Single-head decode aims at
    # ~27 CTAs per SM, grouped decode at ~1, with at least 256 keys per split.
    assert L.fa_decode_choose_splits(1, 32, 32, 8192) == 32      # capped by 8192 / 256 keys
    assert L.fa_decode_choose_splits(4, 32, 32, 8192) == 32
    assert L.fa_decode_choose_splits(64, 32, 32, 8192) == 2
    assert L.fa_decode_choose_splits(1, 28, 4, 32768) == 32
    assert L.fa_decode_choose_splits(8, 28, 4, 8192) == 4
    assert L.fa_decode_choose_splits(64, 28, 4, 8192) == 1
    assert L.fa_decode_choose_splits(1, 32, 32, 100) == 1         # a short sequence is not split
    assert L.fa_decode_choose_splits(0, 32, 32, 8192) == 0
    assert L.fa_decode_choose_splits(1, 30, 4, 8192) == 0         # H_q not a multiple of H_kv
    for B, Hq, Hkv, N in ((1, 1, 1, 1 << 20), (3, 64, 8, 5000)):
        s = L.fa_decode_choose_splits(B, Hq, Hkv, N)
        assert 1 <= s <= 256 and s & (s - 1) == 0
