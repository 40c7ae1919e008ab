"""Helpers for the GPU parity tests: move synthetic BF16 bit patterns to the device and back."""
import numpy as np
import torch

DEV = "cuda:0"


def bf16_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def to_np_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def first_mismatch(a: np.ndarray, b: np.ndarray) -> str:
    bad = np.argwhere(a != b)
    if bad.size == 0:
        return "equal"
    i = tuple(bad[0])
    return f"{len(bad)} mismatches; first at {i}: got {a[i]} want {b[i]}"
