"""Helpers for the GPU parity tests: host <-> device marshalling only."""
import numpy as np
import torch


def dev_bf16(bits):
    """uint16 bf16 bit patterns (numpy) -> CUDA bf16 tensor (same bits)."""
    a = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host_bf16_bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def host(t):
    return t.detach().cpu().numpy()


def bf16_ulp_diff(a_bits, b_bits):
    """Distance in bf16 ulps between two arrays of finite bf16 bit patterns."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + (x & 0x7FFF))
    return np.abs(ordered(a_bits) - ordered(b_bits))
