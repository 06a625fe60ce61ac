"""Guard-band checks: no kernel writes outside the buffers it was given.

Every output and workspace below is a view into the middle of a larger
allocation whose bytes all start as a sentinel pattern; after the call the
bytes before and after the view must still hold the sentinel.  Shapes are
ragged (row counts that are not multiples of the tile sizes, one-key
sequences, pages past a sequence's end) so that every boundary guard in the
kernels is exercised.  Inputs come from the seeded generator; no result
values are compared here (the parity tests do that).
"""

import math

import numpy as np
import pytest

from io_aware_exact_11_gb300 import fa, inputs
from tests.gpu_helpers import Guarded, make_qkv, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.lib()
    yield
    fa.device_status()


def _check(*gs):
    fa.device_status()
    for g in gs:
        assert g.intact(), "a kernel wrote outside its buffer"


@pytest.mark.parametrize("B,H,Nq,Nkv,d,causal", [
    (1, 3, 300, 277, 128, False),
    (2, 2, 1, 129, 128, False),
    (1, 2, 200, 457, 128, True),
    (1, 5, 333, 333, 64, True),
    # head dim 64 without the mask (four 128-row query tiles per CTA, 64-key tiles):
    # a ragged last CTA, one with three query tiles wholly past N_q, exactly one key tile
    (1, 5, 333, 271, 64, False),
    (2, 3, 1, 1, 64, False),
    (2, 3, 700, 64, 64, False),
])
def test_forward_writes_stay_inside_o_and_lse(B, H, Nq, Nkv, d, causal):
    import torch
    _, dev = make_qkv(61, B, H, Nq, Nkv, d, "bf16")
    o = Guarded((B, H, Nq, d), torch.bfloat16)
    lse = Guarded((B, H, Nq), torch.float32)
    fa.forward(dev["q"], dev["k"], dev["v"], out=o.t, lse=lse.t, causal=causal)
    _check(o, lse)


@pytest.mark.parametrize("B,H,Nq,Nkv,causal", [(1, 3, 300, 300, True), (1, 3, 300, 577, False),
                                                (2, 1, 1, 1, False), (2, 2, 129, 700, True)])
def test_fp8_forward_writes_stay_inside(B, H, Nq, Nkv, causal):
    import torch
    q8, k8, v8 = (torch.randint(0, 120, (B, H, n, 128), dtype=torch.uint8, device="cuda") for n in (Nq, Nkv, Nkv))
    o = Guarded((B, H, Nq, 128), torch.bfloat16)
    lse = Guarded((B, H, Nq), torch.float32)
    fa.forward_fp8(q8, k8, v8, out=o.t, lse=lse.t, causal=causal)
    _check(o, lse)


def test_fp32_forward_writes_stay_inside():
    import torch
    _, dev = make_qkv(62, 1, 2, 77, 100, 64, "fp32")
    o32 = Guarded((1, 2, 77, 64), torch.float32)
    l32 = Guarded((1, 2, 77), torch.float32)
    fa.forward(dev["q"], dev["k"], dev["v"], out=o32.t, lse=l32.t)
    _check(o32, l32)


@pytest.mark.parametrize("B,H,N,d", [(1, 2, 300, 128), (2, 1, 129, 128), (1, 3, 200, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_writes_stay_inside_gradients_and_workspace(B, H, N, d, causal):
    import torch
    _, dev = make_qkv(63, B, H, N, N, d, "bf16", with_do=True)
    o, lse = fa.forward(dev["q"], dev["k"], dev["v"], causal=causal)
    grads = [Guarded((B, H, N, d), torch.bfloat16) for _ in range(3)]
    ws = Guarded((int(fa.lib().fa_backward_workspace_size(B, H, N, d)),), torch.uint8)
    fa.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], dq=grads[0].t, dk=grads[1].t, dv=grads[2].t,
                workspace=ws.t, causal=causal)
    _check(*grads, ws)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (28, 4), (32, 1), (128, 2), (71, 1)])
def test_decode_writes_stay_inside_output_and_workspace(Hq, Hkv):
    import torch
    B, N, S = 3, 777, 8
    q = to_device(inputs.normal_tensor(64, "q", B, Hq, 1, 128, "bf16"), "bf16")
    k = to_device(inputs.normal_tensor(64, "k", B, Hkv, N, 128, "bf16"), "bf16")
    v = to_device(inputs.normal_tensor(64, "v", B, Hkv, N, 128, "bf16"), "bf16")
    o = Guarded((B, Hq, 1, 128), torch.bfloat16)
    lse = Guarded((B, Hq), torch.float32)
    ws = Guarded((int(fa.lib().fa_decode_workspace_size(B, Hq, 128, S)),), torch.uint8)
    if Hq == Hkv:
        fa.decode_splitkv(q, k, v, n_splits=S, out=o.t, lse=lse.t, workspace=ws.t)
    else:
        fa.decode_splitkv_gqa(q, k, v, n_splits=S, out=o.t, lse=lse.t, workspace=ws.t)
    _check(o, lse, ws)


@pytest.mark.parametrize("Hq,Hkv,bs", [(4, 4, 16), (28, 4, 16), (8, 2, 64), (32, 1, 32), (96, 1, 16)])
def test_paged_decode_writes_stay_inside_output_and_workspace(Hq, Hkv, bs):
    import torch
    B, S = 3, 4
    lens = np.array([1000, 1, 300], dtype=np.int32)
    per = -(-int(lens.max()) // bs)
    nb = B * per + 3
    kc = to_device(inputs.normal_tensor(65, "k", nb, Hkv, bs, 128, "bf16"), "bf16")
    vc = to_device(inputs.normal_tensor(65, "v", nb, Hkv, bs, 128, "bf16"), "bf16")
    q = to_device(inputs.normal_tensor(65, "q", B, Hq, 1, 128, "bf16"), "bf16")
    order = np.random.default_rng(65).permutation(nb)[: B * per].astype(np.int32).reshape(B, per)
    table = torch.from_numpy(order).cuda()
    seq = torch.from_numpy(lens).cuda()
    o = Guarded((B, Hq, 1, 128), torch.bfloat16)
    lse = Guarded((B, Hq), torch.float32)
    ws = Guarded((int(fa.lib().fa_decode_workspace_size(B, Hq, 128, S)),), torch.uint8)
    fa.decode_paged(q, kc, vc, table, seq, n_splits=S, out=o.t, lse=lse.t, workspace=ws.t)
    _check(o, lse, ws)


def test_host_forward_writes_stay_inside_workspace():
    import torch
    B, H, N, d = 2, 3, 300, 128
    _, dev = make_qkv(66, B, H, N, N, d, "bf16")
    need = int(fa.lib().fa_forward_host_workspace_size(B, H, N, N, d, fa.FA_BF16, 2))
    ws = Guarded((need,), torch.uint8)
    qh, kh, vh = (dev[n].cpu().pin_memory() for n in ("q", "k", "v"))
    oh = torch.empty((B, H, N, d), dtype=torch.bfloat16, pin_memory=True)
    lh = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
    st = torch.cuda.current_stream()
    fa._check(fa.lib().fa_forward_host(fa._ptr(qh), fa._ptr(kh), fa._ptr(vh), fa._ptr(oh), fa._ptr(lh), B, H, N, N,
                                       d, fa.FA_BF16, 1.0 / math.sqrt(d), fa.FA_MASK_NONE, 2, fa._ptr(ws.t), need,
                                       fa._stream_ptr(st)))
    _check(ws)
