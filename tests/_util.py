"""Small conversions shared by the tests (no layer arithmetic here)."""
import numpy as np
import torch

from oracle import moe_ref as ref


def bf16_to_np64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a bf16 tensor."""
    return ref.bf16_to_f64(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def f32_bits(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def sync_status(status: torch.Tensor) -> int:
    torch.cuda.synchronize()
    return int(status.item())
