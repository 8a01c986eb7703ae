"""Python binding of libfp8bs, the GB300 FP8 linear-layer library.

Thin marshalling over the C ABI declared in ``include/fp8bs.h``: every
function here checks tensor devices/dtypes, allocates outputs with PyTorch
when the caller does not pass them, and calls the C entry point of the same
name on the current CUDA stream.  All arithmetic runs in the library's
CUDA kernels; there is no CPU path -- a missing library or a CPU tensor is
an error.

Method (three web pages on FP8 training): block-wise E4M3 quantization with
1x128 activation tiles and 128x128 weight tiles, a block-scaled FP8 GEMM with
fp32 accumulation ("NVIDIA NeMo RL logra una aceleracion del 48%...",
"El avance tecnico"), and per-tensor delayed scaling with an amax history
and E5M2 gradients ("Infraestructura de Entrenamiento FP8", "Transformer
Engine: la base de software").
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB as _LIB_PATH

E4M3, E5M2 = 0, 1
SCALE_FP32, SCALE_POW2 = 0, 1
OUT_F32, OUT_BF16 = 0, 1
GRAN_1x128, GRAN_128x128, GRAN_TENSOR, GRAN_1x32 = 0, 1, 2, 3
EPI_NONE, EPI_SWIGLU = 0, 1

STATUS = {0: "OK", -1: "INVALID_ARG", -2: "UNSUPPORTED", -3: "MISALIGNED", -4: "CUDA",
          -5: "DEVICE_TIMEOUT"}


class Fp8bsError(RuntimeError):
    def __init__(self, code: int, fn: str, msg: str):
        super().__init__(f"{fn} -> {STATUS.get(code, code)}: {msg}")
        self.code = code


class AttnInput(ctypes.Structure):
    """fp8bs_attn_input: FP8 codes [tokens, heads*128] + scale table."""
    _fields_ = [("data", ctypes.c_void_p), ("ld", ctypes.c_int64), ("fmt", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("scales", ctypes.c_void_p)]


class Operand(ctypes.Structure):
    """fp8bs_operand: FP8 data + scale table of one GEMM operand."""
    _fields_ = [("data", ctypes.c_void_p), ("ld", ctypes.c_int64),
                ("transposed", ctypes.c_int32), ("fmt", ctypes.c_int32),
                ("gran", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("scales", ctypes.c_void_p)]


_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libfp8bs (built by ``python -m block_scaled_gemm_quantize_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libfp8bs is not built ({_LIB_PATH} missing); run "
                               "`python -m block_scaled_gemm_quantize_gb300.build`")
        L = ctypes.CDLL(_LIB_PATH)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        op = ctypes.POINTER(Operand)
        sig = {
            "fp8_quantize_1x128": [vp, i64, i64, i64, i32, i32, vp, i64, vp, vp],
            "fp8_quantize_128x128": [vp, i64, i64, i64, i32, i32, vp, i64, vp, vp],
            "fp8_quantize_tensor_delayed": [vp, i64, i32, vp, vp, vp, vp],
            "fp8_quantize_mx": [vp, i64, i64, i64, i32, vp, i64, vp, vp],
            "fp8_quantize_linear": [vp, i64, i64, vp, i64, vp, vp, i64, i64, vp, i64, vp, i64, i32, i32, vp],
            "fp8_quantize_1x128_colwise": [vp, i64, i64, i64, i32, i32, vp, i64, vp, vp, i64, vp, vp],
            "fp8_amax_history_update": [vp, vp, i32, vp, i32, i32, vp, vp],
            "fp8_block_gemm": [i64, i64, i64, op, op, i32, vp, i64, i32, vp],
            "fp8_grouped_block_gemm": [i32, vp, i64, i64, i64, op, op, i32, vp, i64, i32, vp],
            "fp8_block_gemm_quant": [i64, i64, i64, op, op, i32, i32, i32, i32, vp, i64, vp, vp],
            "fp8_grouped_block_gemm_quant": [i32, vp, i64, i64, i64, op, op, i32, i32, i32, i32, vp, i64,
                                             vp, vp],
            "fp8_attention_fwd": [i64, i64, i32, i32, i32, i32, ctypes.c_float,
                                  ctypes.POINTER(AttnInput), ctypes.POINTER(AttnInput),
                                  ctypes.POINTER(AttnInput), vp, i64, vp],
            "fp8bs_device_status": [vp],
            "fp8bs_selftest_wait_timeout": [i32, vp, vp],
            "fp8bs_version": [],
            "fp8bs_last_error": [],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.fp8bs_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _call(name: str, *args) -> None:
    L = lib()
    rc = getattr(L, name)(*args)
    if rc != 0:
        raise Fp8bsError(rc, name, L.fp8bs_last_error().decode(errors="replace"))


def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t, name, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _rowmajor(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with unit column stride")
    return t


# ----------------------------------------------------------- quantizers
def fp8_quantize_1x128(x, fmt=E4M3, mode=SCALE_FP32, q=None, scales=None, stream=None):
    """x [rows, cols] bf16 -> (q [rows, cols] uint8 codes, scales [cols/128, rows] fp32)."""
    torch = _torch()
    _rowmajor(_dev(x, "x", torch.bfloat16), "x")
    rows, cols = x.shape
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((cols // 128, rows), dtype=torch.float32, device=x.device)
    _rowmajor(_dev(q, "q", torch.uint8), "q")
    _dev(scales, "scales", torch.float32)
    _call("fp8_quantize_1x128", x.data_ptr(), rows, cols, x.stride(0), fmt, mode,
          q.data_ptr(), q.stride(0), scales.data_ptr(), _stream(stream))
    return q, scales


def fp8_quantize_128x128(w, fmt=E4M3, mode=SCALE_FP32, q=None, scales=None, stream=None):
    """w [rows, cols] bf16 -> (q, scales [ceil(rows/128), cols/128] fp32)."""
    torch = _torch()
    _rowmajor(_dev(w, "w", torch.bfloat16), "w")
    rows, cols = w.shape
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty(((rows + 127) // 128, cols // 128), dtype=torch.float32, device=w.device)
    _rowmajor(_dev(q, "q", torch.uint8), "q")
    _dev(scales, "scales", torch.float32)
    _call("fp8_quantize_128x128", w.data_ptr(), rows, cols, w.stride(0), fmt, mode,
          q.data_ptr(), q.stride(0), scales.data_ptr(), _stream(stream))
    return q, scales


def fp8_quantize_linear(x, w, fmt=E4M3, mode=SCALE_FP32, qx=None, sx=None, qw=None, sw=None, stream=None):
    """Both operands of a linear layer in one launch: x [m, k] per 1x128 tile,
    w [n, k] per 128x128 tile.  Returns (qx, sx, qw, sw) exactly as
    fp8_quantize_1x128(x) and fp8_quantize_128x128(w) return them."""
    torch = _torch()
    _rowmajor(_dev(x, "x", torch.bfloat16), "x")
    _rowmajor(_dev(w, "w", torch.bfloat16), "w")
    m, k = x.shape
    n, kw = w.shape
    if kw != k:
        raise ValueError(f"x has {k} columns, w has {kw}")
    if qx is None:
        qx = torch.empty((m, k), dtype=torch.uint8, device=x.device)
    if sx is None:
        sx = torch.empty((k // 128, m), dtype=torch.float32, device=x.device)
    if qw is None:
        qw = torch.empty((n, k), dtype=torch.uint8, device=w.device)
    if sw is None:
        sw = torch.empty(((n + 127) // 128, k // 128), dtype=torch.float32, device=w.device)
    for t, nm in ((qx, "qx"), (qw, "qw")):
        _rowmajor(_dev(t, nm, torch.uint8), nm)
    _dev(sx, "sx", torch.float32)
    _dev(sw, "sw", torch.float32)
    _call("fp8_quantize_linear", x.data_ptr(), m, x.stride(0), qx.data_ptr(), qx.stride(0), sx.data_ptr(),
          w.data_ptr(), n, w.stride(0), qw.data_ptr(), qw.stride(0), sw.data_ptr(), k, fmt, mode, _stream(stream))
    return qx, sx, qw, sw


def fp8_quantize_mx(x, fmt=E4M3, q=None, scales=None, stream=None):
    """MXFP8: one E8M0 scale per 32 elements of a row.  Returns (q [rows, cols]
    uint8, scales [cols/128, rows, 4] uint8)."""
    torch = _torch()
    _rowmajor(_dev(x, "x", torch.bfloat16), "x")
    rows, cols = x.shape
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((cols // 128, rows, 4), dtype=torch.uint8, device=x.device)
    _rowmajor(_dev(q, "q", torch.uint8), "q")
    _dev(scales, "scales", torch.uint8)
    _call("fp8_quantize_mx", x.data_ptr(), rows, cols, x.stride(0), fmt, q.data_ptr(), q.stride(0),
          scales.data_ptr(), _stream(stream))
    return q, scales


def fp8_quantize_1x128_colwise(x, fmt=E4M3, mode=SCALE_FP32, rowwise=False, qt=None, scales_t=None,
                               q=None, scales=None, stream=None):
    """Column-wise 1x128 tiles (128 rows of one column), written transposed:
    returns (qt [cols, rows] uint8, scales_t [rows/128, cols] fp32) and, with
    rowwise=True (or q/scales given), also the row-wise (q, scales) from the
    same read of x."""
    torch = _torch()
    _rowmajor(_dev(x, "x", torch.bfloat16), "x")
    rows, cols = x.shape
    if qt is None:
        qt = torch.empty((cols, rows), dtype=torch.uint8, device=x.device)
    if scales_t is None:
        scales_t = torch.empty((rows // 128, cols), dtype=torch.float32, device=x.device)
    _rowmajor(_dev(qt, "qt", torch.uint8), "qt")
    _dev(scales_t, "scales_t", torch.float32)
    if rowwise or q is not None:
        if q is None:
            q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
        if scales is None:
            scales = torch.empty((cols // 128, rows), dtype=torch.float32, device=x.device)
        _rowmajor(_dev(q, "q", torch.uint8), "q")
        _dev(scales, "scales", torch.float32)
    _call("fp8_quantize_1x128_colwise", x.data_ptr(), rows, cols, x.stride(0), fmt, mode, qt.data_ptr(),
          qt.stride(0), scales_t.data_ptr(), q.data_ptr() if q is not None else None,
          q.stride(0) if q is not None else 0, scales.data_ptr() if scales is not None else None,
          _stream(stream))
    if q is not None:
        return qt, scales_t, q, scales
    return qt, scales_t


def fp8_quantize_tensor_delayed(x, fmt, scale, q=None, amax=None, stream=None):
    """Per-tensor quantization with the scale in use (device scalar); returns (q, amax)."""
    torch = _torch()
    _dev(x, "x", torch.bfloat16)
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    _dev(scale, "scale", torch.float32)
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=x.device)
    _call("fp8_quantize_tensor_delayed", x.data_ptr(), x.numel(), fmt, scale.data_ptr(),
          q.data_ptr(), amax.data_ptr(), _stream(stream))
    return q, amax


def fp8_amax_history_update(history, head, amax, fmt, margin, scale, stream=None):
    torch = _torch()
    _dev(history, "history", torch.float32)
    _dev(head, "head", torch.int32)
    _dev(amax, "amax", torch.float32)
    _dev(scale, "scale", torch.float32)
    _call("fp8_amax_history_update", history.data_ptr(), head.data_ptr(), history.numel(),
          amax.data_ptr(), fmt, margin, scale.data_ptr(), _stream(stream))


class DelayedScaling:
    """Per-tensor delayed-scaling state on the device: amax history, head,
    dequantization scale in use (fresh state: zeros, 0, 1.0)."""

    def __init__(self, history_len: int, fmt: int, margin: int = 0, device="cuda"):
        torch = _torch()
        self.fmt, self.margin = fmt, margin
        self.history = torch.zeros(history_len, dtype=torch.float32, device=device)
        self.head = torch.zeros(1, dtype=torch.int32, device=device)
        self.scale = torch.ones(1, dtype=torch.float32, device=device)
        self.amax = torch.zeros(1, dtype=torch.float32, device=device)

    def quantize(self, x, q=None, stream=None, update=False):
        """Quantize x with the scale in use (`self.scale`, built from earlier
        steps) and record its amax in `self.amax`.  The products that read these
        codes must dequantize with that same `self.scale`, so the state is
        advanced separately, by update(), once they have been enqueued;
        update=True advances it right away (for callers that read no product
        from `self.scale` in between)."""
        q, _ = fp8_quantize_tensor_delayed(x, self.fmt, self.scale, q=q, amax=self.amax, stream=stream)
        if update:
            self.update(stream=stream)
        return q

    def update(self, stream=None, group=None):
        """Push this step's amax into the history and compute the next scale.
        With a process group, the amax is first reduced (MAX) over its ranks,
        so every data-parallel replica advances the same history."""
        if group is not None:
            reduce_amax(self.amax, group)
        fp8_amax_history_update(self.history, self.head, self.amax, self.fmt, self.margin,
                                self.scale, stream=stream)

    def state_dict(self):
        return {"history": self.history.cpu(), "head": self.head.cpu(), "scale": self.scale.cpu(),
                "fmt": self.fmt, "margin": self.margin}

    def load_state_dict(self, sd):
        self.history.copy_(sd["history"])
        self.head.copy_(sd["head"])
        self.scale.copy_(sd["scale"])
        self.fmt, self.margin = sd["fmt"], sd["margin"]


# ---------------------------------------------------------------- GEMM
def operand(q, scales, fmt=E4M3, gran=GRAN_1x128, transposed=False) -> Operand:
    """Describe an FP8 operand.  q is the stored matrix: [rows, K] or, when
    transposed, [K, rows]; scales follow the table layouts of fp8bs.h."""
    torch = _torch()
    _rowmajor(_dev(q, "q", torch.uint8), "q")
    _dev(scales, "scales", torch.uint8 if gran == GRAN_1x32 else torch.float32)
    op = Operand(data=q.data_ptr(), ld=q.stride(0), transposed=int(bool(transposed)), fmt=fmt,
                 gran=gran, reserved=0, scales=scales.data_ptr())
    op._keep = (q, scales)
    return op


def fp8_block_gemm(A: Operand, B: Operand, M: int, N: int, K: int, out_dtype=OUT_BF16,
                   mode=SCALE_FP32, y=None, stream=None, device=None):
    """Y [M, N] = deq(A) deq(B)^T (fp32 accumulation), bf16 or fp32 output."""
    torch = _torch()
    dt = torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32
    if y is None:
        dev = device if device is not None else A._keep[0].device
        y = torch.empty((M, N), dtype=dt, device=dev)
    _rowmajor(_dev(y, "y", dt), "y")
    _call("fp8_block_gemm", M, N, K, ctypes.byref(A), ctypes.byref(B), mode, y.data_ptr(),
          y.stride(0), out_dtype, _stream(stream))
    return y


def fp8_grouped_block_gemm(offsets, A: Operand, B: Operand, a_rows: int, N: int, K: int,
                           out_dtype=OUT_BF16, mode=SCALE_FP32, y=None, stream=None):
    """Grouped product: rows [offsets[g], offsets[g+1]) of A times expert g's
    weights (B stored [G*N, K]).  offsets: int32 device tensor [G+1]."""
    torch = _torch()
    _dev(offsets, "offsets", torch.int32)
    dt = torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32
    if y is None:
        y = torch.empty((a_rows, N), dtype=dt, device=offsets.device)
    _rowmajor(_dev(y, "y", dt), "y")
    _call("fp8_grouped_block_gemm", offsets.numel() - 1, offsets.data_ptr(), a_rows, N, K,
          ctypes.byref(A), ctypes.byref(B), mode, y.data_ptr(), y.stride(0), out_dtype,
          _stream(stream))
    return y


def _quant_out(rows, n_out, q, q_scales, device):
    torch = _torch()
    if q is None:
        q = torch.empty((rows, n_out), dtype=torch.uint8, device=device)
    if q_scales is None:
        q_scales = torch.empty((n_out // 128, rows), dtype=torch.float32, device=device)
    _rowmajor(_dev(q, "q", torch.uint8), "q")
    _dev(q_scales, "q_scales", torch.float32)
    return q, q_scales


def fp8_block_gemm_quant(A: Operand, B: Operand, M: int, N: int, K: int, epilogue=EPI_NONE,
                         q_fmt=E4M3, q_mode=SCALE_FP32, mode=SCALE_FP32, q=None, q_scales=None,
                         stream=None):
    """Product whose epilogue emits the next linear's FP8 operand: Z = Y or
    (SwiGLU) silu(Y[:, :N/2]) * Y[:, N/2:], quantized per 1x128 tile.
    Returns (q [M, cols(Z)] uint8, q_scales [cols(Z)/128, M] fp32)."""
    n_out = N // 2 if epilogue == EPI_SWIGLU else N
    q, q_scales = _quant_out(M, n_out, q, q_scales, A._keep[0].device)
    _call("fp8_block_gemm_quant", M, N, K, ctypes.byref(A), ctypes.byref(B), mode, epilogue, q_fmt,
          q_mode, q.data_ptr(), q.stride(0), q_scales.data_ptr(), _stream(stream))
    return q, q_scales


def fp8_grouped_block_gemm_quant(offsets, A: Operand, B: Operand, a_rows: int, N: int, K: int,
                                 epilogue=EPI_NONE, q_fmt=E4M3, q_mode=SCALE_FP32, mode=SCALE_FP32,
                                 q=None, q_scales=None, stream=None):
    """Grouped form of fp8_block_gemm_quant (expert layers)."""
    torch = _torch()
    _dev(offsets, "offsets", torch.int32)
    n_out = N // 2 if epilogue == EPI_SWIGLU else N
    q, q_scales = _quant_out(a_rows, n_out, q, q_scales, offsets.device)
    _call("fp8_grouped_block_gemm_quant", offsets.numel() - 1, offsets.data_ptr(), a_rows, N, K,
          ctypes.byref(A), ctypes.byref(B), mode, epilogue, q_fmt, q_mode, q.data_ptr(), q.stride(0),
          q_scales.data_ptr(), _stream(stream))
    return q, q_scales


def linear_fprop(x, w, mode=SCALE_FP32, out_dtype=OUT_BF16, stream=None):
    """FP8 linear layer forward: Y = X W^T with X quantized per 1x128 tile and
    W per 128x128 tile (E4M3), block-scaled FP8 GEMM, fp32 accumulation."""
    qx, sx, qw, sw = fp8_quantize_linear(x, w, E4M3, mode, stream=stream)
    A = operand(qx, sx, E4M3, GRAN_1x128)
    B = operand(qw, sw, E4M3, GRAN_128x128)
    return fp8_block_gemm(A, B, x.shape[0], w.shape[0], x.shape[1], out_dtype, mode, stream=stream)


def attn_input(q, scales, fmt=E4M3) -> AttnInput:
    """Describe an attention input: codes [tokens, heads*128] (uint8), scales
    (Q: [heads, tokens]; K, V: [ceil(tokens/128), heads])."""
    torch = _torch()
    _rowmajor(_dev(q, "q", torch.uint8), "q")
    _dev(scales, "scales", torch.float32)
    a = AttnInput(data=q.data_ptr(), ld=q.stride(0), fmt=fmt, reserved=0, scales=scales.data_ptr())
    a._keep = (q, scales)
    return a


def fp8_attention_fwd(Q: AttnInput, K: AttnInput, V: AttnInput, seq_q: int, seq_k: int, heads_q: int,
                      heads_kv: int, causal=True, softmax_scale=None, o=None, stream=None):
    """FP8 attention forward over an FP8 KV cache; returns O bf16 [seq_q, heads_q*128]."""
    torch = _torch()
    if softmax_scale is None:
        softmax_scale = 128 ** -0.5
    if o is None:
        o = torch.empty((seq_q, heads_q * 128), dtype=torch.bfloat16, device=Q._keep[0].device)
    _rowmajor(_dev(o, "o", torch.bfloat16), "o")
    _call("fp8_attention_fwd", seq_q, seq_k, heads_q, heads_kv, 128, int(bool(causal)), float(softmax_scale),
          ctypes.byref(Q), ctypes.byref(K), ctypes.byref(V), o.data_ptr(), o.stride(0), _stream(stream))
    return o


def device_status(stream=None) -> None:
    """Raise if a kernel gave up on a bounded device wait (synchronizes)."""
    _call("fp8bs_device_status", _stream(stream))


def selftest_wait_timeout(limit_ms: int = 200, stream=None) -> bool:
    """Run the bounded-wait self-test; returns True if the wait gave up (and
    leaves the timeout recorded for device_status())."""
    torch = _torch()
    out = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _call("fp8bs_selftest_wait_timeout", limit_ms, out.data_ptr(), _stream(stream))
    torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
    return int(out.item()) == 0


def reduce_amax(amax, group=None):
    """Data-parallel exchange of delayed scaling: element-wise MAX of this
    step's amax over the ranks of `group` (torch.distributed), in place."""
    import torch.distributed as dist
    dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    return amax


def version() -> int:
    return lib().fp8bs_version()
