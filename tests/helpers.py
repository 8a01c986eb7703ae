"""Shared helpers of the GPU parity tests (marshalling only)."""
import numpy as np


def dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t) -> np.ndarray:
    import torch
    t = t.detach()
    if t.dtype == torch.bfloat16:          # numpy has no bf16: return the bit patterns
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def f32_bits(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def stratified(n: int, block: int, rng, extra=()):
    """One random index per block of `block`, plus the first/last and extras."""
    idx = [min(n - 1, b + int(rng.integers(0, block))) for b in range(0, n, block)]
    idx += [0, n - 1] + [e for e in extra if 0 <= e < n]
    return np.unique(np.array(idx, dtype=np.int64))
