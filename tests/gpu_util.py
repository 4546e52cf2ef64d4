"""Helpers for the GPU tests: device tensors from seeded numpy draws, fp64 views.

Device memory comes from torch; every pass runs in the CUDA library through
its C ABI.  bf16 conversion is torch's round-to-nearest-even cast, done once
on the host so the oracle sees the same input bits.
"""

import numpy as np
import torch


def have_gpu() -> bool:
    return torch.cuda.is_available()


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def empty_bf16(*shape) -> torch.Tensor:
    # NaN-filled so that an unwritten element fails every comparison
    return torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")


def empty_f32(*shape) -> torch.Tensor:
    return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")


def sync(zb):
    torch.cuda.synchronize()
    zb.zb_sync_status()
