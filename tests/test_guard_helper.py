"""The guard-band detector used by the GPU write-bounds tests, checked on
the CPU: writes inside the view leave it intact, a single byte written just
before or just after the view is caught."""

import pytest

from tests.gpu_helpers import Guarded


def test_writes_inside_the_view_leave_the_guards_intact():
    torch = pytest.importorskip("torch")
    g = Guarded((3, 5, 7), torch.float32, device="cpu")
    g.t.fill_(1.5)
    assert g.intact()


@pytest.mark.parametrize("where", ["before", "after"])
def test_one_stray_byte_is_caught(where):
    torch = pytest.importorskip("torch")
    g = Guarded((3, 5, 7), torch.bfloat16, device="cpu")
    g.t.fill_(2.0)
    idx = Guarded.GUARD - 1 if where == "before" else Guarded.GUARD + g.nbytes
    g.raw[idx] = 0
    assert not g.intact()


def test_view_keeps_256_byte_alignment():
    torch = pytest.importorskip("torch")
    g = Guarded((100,), torch.float32, device="cpu")
    assert (g.t.data_ptr() - g.raw.data_ptr()) % 256 == 0
