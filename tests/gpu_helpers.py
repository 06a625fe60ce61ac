"""Shared helpers for the GPU parity tests: seeded inputs on the device and
error metrics.  Inputs come from the seeded generator only; expected values
come from the float64 oracle only."""

from __future__ import annotations

import numpy as np

from io_aware_exact_11_gb300 import inputs


def to_device(host: np.ndarray, dtype: str):
    """Host tensor from ``inputs.normal_tensor`` -> CUDA tensor (bf16 or fp32)."""
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(host).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(host))
    return t.cuda()


def make_qkv(seed: int, B: int, H: int, Nq: int, Nkv: int, d: int, dtype: str, with_do: bool = False):
    """Host arrays (storage type) and device tensors for Q, K, V (and dO)."""
    host = {
        "q": inputs.normal_tensor(seed, "q", B, H, Nq, d, dtype),
        "k": inputs.normal_tensor(seed, "k", B, H, Nkv, d, dtype),
        "v": inputs.normal_tensor(seed, "v", B, H, Nkv, d, dtype),
    }
    if with_do:
        host["do"] = inputs.normal_tensor(seed, "do", B, H, Nq, d, dtype)
    dev = {k: to_device(v, dtype) for k, v in host.items()}
    return host, dev


def f64(host: np.ndarray, dtype: str) -> np.ndarray:
    return inputs.as_f64(host, dtype)


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64))))


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def cpu64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class Guarded:
    """A tensor of the given shape and dtype placed in the middle of a larger
    byte buffer whose every byte starts as SENTINEL; ``intact()`` says whether
    the GUARD bytes before and after the tensor still hold it.  GUARD is a
    multiple of 256, so the tensor keeps the allocation's alignment."""

    GUARD = 4096
    SENTINEL = 0x5A

    def __init__(self, shape, dtype, device="cuda"):
        import torch
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.nbytes = n
        self.raw = torch.full((self.GUARD + n + self.GUARD,), self.SENTINEL, dtype=torch.uint8, device=device)
        self.t = self.raw[self.GUARD:self.GUARD + n].view(dtype).view(shape)

    def intact(self) -> bool:
        import torch
        if self.raw.is_cuda:
            torch.cuda.synchronize()
        head = self.raw[:self.GUARD].cpu().numpy()
        tail = self.raw[self.GUARD + self.nbytes:].cpu().numpy()
        return bool(np.all(head == self.SENTINEL) and np.all(tail == self.SENTINEL))
