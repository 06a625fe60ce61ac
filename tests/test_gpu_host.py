"""GPU checks of the host-buffer forward (fa_forward_host): the chunked,
pipelined copies must give exactly the device forward's results on the same
data, and those match the float64 oracle within the usual bounds (bf16 O
within 1e-2 max-abs and LSE within 1e-3; fp32 within 1e-5)."""

import math

import pytest

import oracle
from io_aware_exact_11_gb300 import fa
from tests.gpu_helpers import cpu64, f64, make_qkv, max_abs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.lib()
    yield
    fa.device_status()


def _host(t, pinned=True):
    h = t.cpu()
    return h.pin_memory() if pinned else h


@pytest.mark.parametrize("shape,dtype,causal,hpc", [
    ((2, 3, 300, 277, 128), "bf16", False, 4),   # 6 heads in chunks of 4 and 2, ragged rows and keys
    ((1, 5, 256, 256, 64), "bf16", False, 1),    # five one-head chunks, head dim 64
    ((2, 2, 200, 457, 128), "bf16", True, 3),    # causal, N_q < N_kv, chunks of 3 and 1
    ((1, 3, 100, 130, 128), "fp32", False, 2),   # fp32 path
])
def test_host_forward_equals_device_forward(shape, dtype, causal, hpc):
    import torch
    B, H, Nq, Nkv, d = shape
    _, dev = make_qkv(31, B, H, Nq, Nkv, d, dtype)
    o_dev, l_dev = fa.forward(dev["q"], dev["k"], dev["v"], causal=causal)
    qh, kh, vh = (_host(dev[n]) for n in ("q", "k", "v"))
    o_h, l_h = fa.forward_host(qh, kh, vh, causal=causal, heads_per_chunk=hpc)
    torch.cuda.synchronize()
    fa.device_status()
    assert torch.equal(o_h, o_dev.cpu()) and torch.equal(l_h, l_dev.cpu())


def test_host_forward_matches_oracle_with_default_chunks():
    """B=4, H=24, N=384: the library picks the chunking (several chunks)."""
    import torch
    B, H, N, d = 4, 24, 384, 128
    host, dev = make_qkv(32, B, H, N, N, d, "bf16")
    o_h, l_h = fa.forward_host(*(_host(dev[n]) for n in ("q", "k", "v")))
    torch.cuda.synchronize()
    fa.device_status()
    scale = 1.0 / math.sqrt(d)
    ro, rl = oracle.attention_forward(f64(host["q"], "bf16"), f64(host["k"], "bf16"), f64(host["v"], "bf16"), scale)
    assert max_abs(cpu64(o_h), ro) <= 1e-2 and max_abs(cpu64(l_h), rl) <= 1e-3


def test_host_forward_pageable_inputs_and_reuse():
    """Pageable host tensors are copied correctly too, and two calls in a row
    on the same stream (sharing the library's workspace and events) both land."""
    import torch
    B, H, N, d = 1, 4, 256, 128
    _, d1 = make_qkv(33, B, H, N, N, d, "bf16")
    _, d2 = make_qkv(34, B, H, N, N, d, "bf16")
    r1 = fa.forward(d1["q"], d1["k"], d1["v"])
    r2 = fa.forward(d2["q"], d2["k"], d2["v"])
    a = fa.forward_host(*(_host(d1[n], pinned=False) for n in ("q", "k", "v")), heads_per_chunk=1)
    b = fa.forward_host(*(_host(d2[n]) for n in ("q", "k", "v")), heads_per_chunk=3)
    torch.cuda.synchronize()
    fa.device_status()
    for got, ref in ((a, r1), (b, r2)):
        assert torch.equal(got[0], ref[0].cpu()) and torch.equal(got[1], ref[1].cpu())


def test_host_forward_from_two_threads():
    """Two host threads call the host-buffer forward at once, each on its own
    stream: the library serialises them on its per-device copy streams and
    workspace bookkeeping, and both results are exact."""
    import threading

    import torch
    B, H, N, d = 2, 4, 256, 128
    data = [make_qkv(40 + t, B, H, N, N, d, "bf16")[1] for t in range(2)]
    refs = [fa.forward(dv["q"], dv["k"], dv["v"]) for dv in data]
    torch.cuda.synchronize()
    results = [None, None]
    errors = []

    def run(t):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                hq, hk, hv = (_host(data[t][n]) for n in ("q", "k", "v"))
                for _ in range(3):
                    results[t] = fa.forward_host(hq, hk, hv, heads_per_chunk=3, stream=st)
            st.synchronize()
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    fa.device_status()
    for t in range(2):
        assert torch.equal(results[t][0], refs[t][0].cpu()) and torch.equal(results[t][1], refs[t][1].cpu())

