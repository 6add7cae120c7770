"""Helpers of the GPU tests: host <-> device copies of bit patterns, and
outputs fenced by canary bytes so that out-of-bounds writes show up."""

import numpy as np
import torch

CANARY = 0xA5
GUARD = 4096


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def dev_input(a: np.ndarray) -> torch.Tensor:
    return dev_bf16(a) if a.dtype == np.uint16 else dev_f32(a)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a device tensor: uint16 for bf16, uint32 for fp32, uint8 for bytes."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    if t.dtype in (torch.uint8, torch.float8_e4m3fn, torch.float8_e5m2):
        return t.view(torch.uint8).numpy()
    raise TypeError(t.dtype)


def oracle_bits(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.float32:
        return a.view(np.uint32)
    return a


class Guarded:
    """A device buffer of `shape`/`dtype` with CANARY bytes on both sides."""

    def __init__(self, shape, dtype, offset: int = 0):
        es = torch.empty((), dtype=dtype).element_size()
        n = 1
        for d in shape:
            n *= d
        self.nbytes = n * es
        self.head = GUARD + offset
        self.raw = torch.full((self.nbytes + 2 * GUARD + offset,), CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.raw[self.head:self.head + self.nbytes].view(dtype).view(shape)

    def intact(self) -> bool:
        r = self.raw
        return bool((r[:self.head] == CANARY).all()) and bool((r[self.head + self.nbytes:] == CANARY).all())
