"""Copy a generated case to the GPU as torch tensors (plumbing only: no arithmetic)."""
from __future__ import annotations

from types import SimpleNamespace

import numpy as np
import torch

from .gen import Case


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bit patterns -> a bf16 torch tensor on `device` (same bits)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def bf16_bits_of(t: torch.Tensor) -> np.ndarray:
    """A bf16 tensor -> its uint16 bit patterns on the host."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def i32_tensor(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def to_device(case: Case, device="cuda") -> SimpleNamespace:
    return SimpleNamespace(
        q=bf16_tensor(case.q, device),
        k_new=bf16_tensor(case.k_new, device),
        v_new=bf16_tensor(case.v_new, device),
        k_pool=bf16_tensor(case.k_pool, device),
        v_pool=bf16_tensor(case.v_pool, device),
        block_table=i32_tensor(case.block_table, device),
        context_lens=i32_tensor(case.context_lens, device),
        q_indptr=i32_tensor(case.q_indptr, device),
    )
