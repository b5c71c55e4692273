"""Helpers for the GPU parity tests: move seeded host inputs to the device."""
import numpy as np
import torch


def dev(a, dtype=None):
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.to(dtype) if dtype is not None else t).cuda()


def host(t):
    return t.detach().cpu().numpy()


def as_f32(a):
    """Host float32 view of bf16 bits or float arrays."""
    import dspark_inputs as di
    return di.bf16_bits_to_f32(a) if a.dtype == np.uint16 else np.asarray(a, dtype=np.float32)
