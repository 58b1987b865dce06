"""numpy storage arrays <-> torch device tensors (bf16 carried as uint16 bit patterns)."""
import numpy as np
import torch


def to_dev(a, dev, bf16=False):
    a = np.ascontiguousarray(a)
    if bf16 or a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def to_np(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def widen(a):
    """storage array (float32 or bf16 bits) -> float64 values."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)
