"""CUDA graph capture: every device entry point only enqueues work on the
caller's stream (the host-buffer forward also forks onto its copy streams
with events), so it can be captured once and replayed.  Each test captures
a call, overwrites the inputs in place, replays, and compares with an eager
call on the new inputs: results must be identical bit for bit (dQ, summed
with reductions in a varying order, to one bf16 ulp per element)."""

import numpy as np
import pytest

from io_aware_exact_11_gb300 import fa, inputs
from tests.gpu_helpers import make_qkv, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.lib()
    yield
    fa.device_status()


def _capture(fn):
    """Warm up on a side stream (first calls set kernel attributes), then capture."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _refill(dst, seed, name, dtype="bf16"):
    src = to_device(inputs.normal_tensor(seed, name, *dst.shape, dtype), dtype)
    dst.copy_(src)


@pytest.mark.parametrize("d,causal", [(128, False), (128, True), (64, False)])
def test_forward_replay_matches_eager(d, causal):
    import torch
    B, H, N = 2, 3, 300
    _, dev = make_qkv(71, B, H, N, N, d, "bf16")
    q, k, v = dev["q"], dev["k"], dev["v"]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device="cuda")
    g = _capture(lambda: fa.forward(q, k, v, out=o, lse=lse, causal=causal))
    for name, t in (("q", q), ("k", k), ("v", v)):
        _refill(t[:, :, :, :], 72, name)
    g.replay()
    torch.cuda.synchronize()
    ro, rl = fa.forward(q, k, v, causal=causal)
    torch.cuda.synchronize()
    fa.device_status()
    assert torch.equal(o, ro) and torch.equal(lse, rl)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (28, 4)])
def test_decode_replay_matches_eager(Hq, Hkv):
    import torch
    B, N, d, S = 2, 1000, 128, 8
    q = to_device(inputs.normal_tensor(73, "q", B, Hq, 1, d, "bf16"), "bf16")
    k = to_device(inputs.normal_tensor(73, "k", B, Hkv, N, d, "bf16"), "bf16")
    v = to_device(inputs.normal_tensor(73, "v", B, Hkv, N, d, "bf16"), "bf16")
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), device="cuda")
    ws = torch.empty(int(fa.lib().fa_decode_workspace_size(B, Hq, d, S)), dtype=torch.uint8, device="cuda")
    dec = fa.decode_splitkv if Hq == Hkv else fa.decode_splitkv_gqa
    g = _capture(lambda: dec(q, k, v, n_splits=S, out=o, lse=lse, workspace=ws))
    _refill(q, 74, "q")
    g.replay()
    torch.cuda.synchronize()
    ro, rl = dec(q, k, v, n_splits=S)
    torch.cuda.synchronize()
    fa.device_status()
    assert torch.equal(o, ro) and torch.equal(lse, rl)


def test_paged_decode_replay_follows_table_and_length_updates():
    """The block table and sequence lengths live in device memory, so a
    captured decode step picks up a grown sequence on replay."""
    import torch
    B, Hq, Hkv, bs, d, S = 2, 8, 2, 16, 128, 4
    per, nb = 40, 2 * 40 + 4
    kc = to_device(inputs.normal_tensor(75, "k", nb, Hkv, bs, d, "bf16"), "bf16")
    vc = to_device(inputs.normal_tensor(75, "v", nb, Hkv, bs, d, "bf16"), "bf16")
    q = to_device(inputs.normal_tensor(75, "q", B, Hq, 1, d, "bf16"), "bf16")
    order = np.random.default_rng(75).permutation(nb)[: B * per].astype(np.int32).reshape(B, per)
    table = torch.from_numpy(order).cuda()
    lens = torch.tensor([300, 17], dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), device="cuda")
    ws = torch.empty(int(fa.lib().fa_decode_workspace_size(B, Hq, d, S)), dtype=torch.uint8, device="cuda")
    g = _capture(lambda: fa.decode_paged(q, kc, vc, table, lens, n_splits=S, out=o, lse=lse, workspace=ws))
    lens.copy_(torch.tensor([639, 18], dtype=torch.int32))   # the table holds 40 pages = 640 keys
    table[1, 1] = int(order[0, 39])          # sequence 1's second page moves
    _refill(q, 76, "q")
    g.replay()
    torch.cuda.synchronize()
    ro, rl = fa.decode_paged(q, kc, vc, table, lens, n_splits=S)
    torch.cuda.synchronize()
    fa.device_status()
    assert torch.equal(o, ro) and torch.equal(lse, rl)


def test_backward_replay_matches_eager():
    import torch
    B, H, N, d = 1, 2, 300, 128
    _, dev = make_qkv(77, B, H, N, N, d, "bf16", with_do=True)
    q, k, v, do = dev["q"], dev["k"], dev["v"], dev["do"]
    o, lse = fa.forward(q, k, v)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(int(fa.lib().fa_backward_workspace_size(B, H, N, d)), dtype=torch.uint8, device="cuda")
    g = _capture(lambda: fa.backward(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, workspace=ws))
    _refill(do, 78, "do")
    g.replay()
    torch.cuda.synchronize()
    rq, rk, rv = fa.backward(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    fa.device_status()
    # dK and dV are accumulated in TMEM in a fixed order; dQ is summed with fp32
    # reductions whose order varies from run to run.  Those fp32 sums differ by a
    # few fp32 ulps at most, far below a bf16 ulp, so after rounding to bf16 each
    # element may differ by at most one bf16 ulp (8 significant bits).
    assert torch.equal(dk, rk) and torch.equal(dv, rv)
    a, b = dq.float(), rq.float()
    _, e = torch.frexp(torch.maximum(a.abs(), b.abs()))
    ulp = torch.ldexp(torch.ones_like(a), e - 8)
    assert bool(((a - b).abs() <= ulp).all())


def test_host_forward_replay_matches_eager():
    """Graph capture across the host-buffer forward's copy streams (forked and
    joined with events) and its host↔device copies."""
    import torch
    B, H, N, d = 2, 3, 256, 128
    _, dev = make_qkv(79, B, H, N, N, d, "bf16")
    qh, kh, vh = (dev[n].cpu().pin_memory() for n in ("q", "k", "v"))
    oh = torch.empty((B, H, N, d), dtype=torch.bfloat16, pin_memory=True)
    lh = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
    g = _capture(lambda: fa.forward_host(qh, kh, vh, out=oh, lse=lh, heads_per_chunk=2))
    _, dev2 = make_qkv(80, B, H, N, N, d, "bf16")
    for src, dst in ((dev2["q"], qh), (dev2["k"], kh), (dev2["v"], vh)):
        dst.copy_(src.cpu())
    g.replay()
    torch.cuda.synchronize()
    ro, rl = fa.forward(dev2["q"], dev2["k"], dev2["v"])
    torch.cuda.synchronize()
    fa.device_status()
    assert torch.equal(oh, ro.cpu()) and torch.equal(lh, rl.cpu())
