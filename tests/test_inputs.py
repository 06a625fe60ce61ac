"""The seeded input generator: determinism, slicing and bf16 rounding."""

import numpy as np
import pytest

from io_aware_exact_11_gb300 import inputs


def test_slices_are_deterministic_and_distinct():
    a = inputs.normal_slice(3, "q", 1, 2, 16, 8)
    b = inputs.normal_slice(3, "q", 1, 2, 16, 8)
    c = inputs.normal_slice(3, "k", 1, 2, 16, 8)
    d = inputs.normal_slice(4, "q", 1, 2, 16, 8)
    assert a.dtype == np.float32 and np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)


def test_full_tensor_is_stack_of_slices():
    t = inputs.normal_tensor(7, "v", 2, 3, 33, 8, dtype="fp32")
    for b in range(2):
        for h in range(3):
            assert np.array_equal(t[b, h], inputs.normal_slice(7, "v", b, h, 33, 8))
    tb = inputs.normal_tensor(7, "v", 2, 3, 33, 8, dtype="bf16")
    assert np.array_equal(inputs.as_f64(tb, "bf16")[1, 2], inputs.head_as_f64(7, "v", 1, 2, 33, 8))


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.concatenate([
        np.random.default_rng(0).standard_normal(100000).astype(np.float32),
        np.array([1.0, -2.5, 3.0039062, 1.00390625, 1.01171875, 0.0, -0.0], dtype=np.float32),
    ])
    ours = inputs.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = inputs.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_distribution_is_standard_normal():
    x = inputs.normal_slice(0, "q", 0, 0, 4096, 64)
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01


def test_e4m3_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8")
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32) * s for s in (1.0, 0.01, 30.0)] +
                       [np.array([0.0, -0.0, 448.0, 460.0, 1e6, -1e6, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10,
                                  0.0625, 0.06640625, 1.0625, 1.1875], dtype=np.float32)])
    ours = inputs.f32_to_e4m3_bits(x)
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    back = inputs.e4m3_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(ref).view(torch.float8_e4m3fn).float().numpy())
