"""The failure path of the bounded pipeline waits, on the device.

fa_watchdog_selftest enqueues a kernel whose thread waits, with the same
bounded wait every pipeline kernel uses, on a barrier that nothing completes.
The wait gives up after its limit (1 s) and records its site; nothing faults
or hangs.  fa_device_status must then report FA_ERR_DEVICE_TIMEOUT naming the
kernel and site, clear the flag, and leave a context that still computes
correct results."""

import math
import time

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
    fa.device_status()  # start from a clear watchdog word
    yield
    fa.device_status()


def test_wait_that_runs_out_is_reported_and_the_context_survives():
    t0 = time.monotonic()
    fa.watchdog_selftest()
    with pytest.raises(fa.FAError) as ei:
        fa.device_status()
    elapsed = time.monotonic() - t0
    assert ei.value.status == fa.FA_ERR_DEVICE_TIMEOUT
    msg = fa.lib().fa_get_last_error()
    assert b"kernel 15" in msg and b"site 1" in msg, msg
    assert 0.5 <= elapsed < 60.0, elapsed  # the wait limit is 1 s of device time
    fa.device_status()  # the flag was cleared by the report

    B, H, Nq, Nkv, d = 1, 2, 200, 300, 128
    host, dev = make_qkv(90, B, H, Nq, Nkv, d, "bf16")
    o, lse = fa.forward(dev["q"], dev["k"], dev["v"])
    fa.device_status()
    for h in range(H):
        ro, rl = oracle.attention_forward(f64(host["q"][0, h], "bf16"), f64(host["k"][0, h], "bf16"),
                                          f64(host["v"][0, h], "bf16"), 1.0 / math.sqrt(d))
        assert max_abs(cpu64(o[0, h]), ro) <= 1e-2 and max_abs(cpu64(lse[0, h]), rl) <= 1e-3
