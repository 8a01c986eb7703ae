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


# ------------------------------------------------ the oracle on many host cores
# The oracle's C routines are called through ctypes, which releases the GIL,
# so row chunks run on separate cores.  Splitting is by definition exact: the
# 1x128 rule is per row, the 128x128 rule per 128-row block, the per-tensor
# rule elementwise (its amax is the max of the chunks' amaxes), and every
# output element of a product is its own sum.
def host_threads() -> int:
    import os
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _chunks(n, parts, align=1):
    step = max(align, -(-n // max(1, parts)) // align * align)
    return [(i, min(n, i + step)) for i in range(0, n, step)]


def par_map(fn, jobs, threads=None):
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=threads or host_threads()) as ex:
        return list(ex.map(fn, jobs))


def par_quantize_1x128(orc, x, fmt, mode):
    parts = par_map(lambda c: orc.quantize_1x128(x[c[0]:c[1]], fmt, mode), _chunks(x.shape[0], host_threads()))
    return np.concatenate([q for q, _ in parts], 0), np.ascontiguousarray(np.concatenate([s for _, s in parts], 1))


def par_quantize_128x128(orc, w, fmt, mode):
    parts = par_map(lambda c: orc.quantize_128x128(w[c[0]:c[1]], fmt, mode),
                    _chunks(w.shape[0], host_threads(), 128))
    return np.concatenate([q for q, _ in parts], 0), np.concatenate([s for _, s in parts], 0)


def par_quantize_tensor(orc, x, fmt, scale):
    """Per-tensor quantization with a given scale -> (q, amax)."""
    flat = x.reshape(-1)
    parts = par_map(lambda c: orc.quantize_tensor(flat[c[0]:c[1]], fmt, scale), _chunks(flat.size, host_threads()))
    return np.concatenate([q for q, _ in parts]).reshape(x.shape), max(a for _, a in parts)


def par_gemm(orc, M, N, K, A, B, rows, cols):
    rows = np.asarray(rows)
    parts = par_map(lambda c: orc.gemm(M, N, K, A, B, rows=rows[c[0]:c[1]], cols=cols),
                    _chunks(rows.size, 4 * host_threads()))
    return np.concatenate([y for y, _ in parts], 0), np.concatenate([a for _, a in parts], 0)


def par_grouped_gemm(orc, off, a_rows, N, K, A, B, rows, cols):
    rows = np.asarray(rows)
    parts = par_map(lambda c: orc.grouped_gemm(off, a_rows, N, K, A, B, rows=rows[c[0]:c[1]], cols=cols),
                    _chunks(rows.size, 4 * host_threads()))
    return np.concatenate([y for y, _ in parts], 0), np.concatenate([a for _, a in parts], 0)
