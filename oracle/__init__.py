"""CPU oracle for the FP8 linear layer -- test infrastructure only.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never does, and this package never imports the product.

The arithmetic lives in ``fp8_oracle.c`` (plain loops, fp64 where a sum is
formed); this module only compiles it with ``gcc`` and marshals numpy arrays.
Every function cites the passage of the FP8-training pages it restates in the
C source.

Pins (what ties each part to something other than itself) are the
``-m "not gpu"`` tests ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

E4M3, E5M2 = 0, 1
SCALE_FP32, SCALE_POW2 = 0, 1
GRAN_1x128, GRAN_128x128, GRAN_TENSOR, GRAN_1x32 = 0, 1, 2, 3

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, f"liboracle_{platform.machine()}.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class Operand(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("ld", ctypes.c_int64),
                ("transposed", ctypes.c_int32), ("fmt", ctypes.c_int32),
                ("gran", ctypes.c_int32), ("pad_", ctypes.c_int32),
                ("scales", ctypes.c_void_p)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    i64, i32, vp, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_float
    lib.fp8o_decode.argtypes = [ctypes.c_uint32, ctypes.c_int]
    lib.fp8o_decode.restype = ctypes.c_double
    lib.fp8o_fmax.argtypes = [ctypes.c_int]
    lib.fp8o_fmax.restype = ctypes.c_double
    lib.fp8o_encode.argtypes = [f32, ctypes.c_int]
    lib.fp8o_encode.restype = ctypes.c_uint32
    lib.fp8o_encode_array.argtypes = [vp, i64, ctypes.c_int, vp]
    lib.fp8o_encode_array.restype = None
    lib.fp8o_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.fp8o_bf16_to_f32.restype = f32
    lib.fp8o_block_scale.argtypes = [f32, ctypes.c_int, ctypes.c_int]
    lib.fp8o_block_scale.restype = f32
    lib.fp8o_quantize_1x128.argtypes = [vp, i64, i64, i64, ctypes.c_int, ctypes.c_int, vp, i64, vp]
    lib.fp8o_quantize_1x128.restype = None
    lib.fp8o_quantize_1x128_f32.argtypes = [vp, i64, i64, i64, ctypes.c_int, ctypes.c_int, vp, i64,
                                            vp]
    lib.fp8o_quantize_1x128_f32.restype = None
    lib.fp8o_mx_scale_code.argtypes = [f32, ctypes.c_int]
    lib.fp8o_mx_scale_code.restype = ctypes.c_uint8
    lib.fp8o_quantize_mx.argtypes = [vp, i64, i64, i64, ctypes.c_int, vp, i64, vp]
    lib.fp8o_quantize_mx.restype = None
    lib.fp8o_quantize_128x128.argtypes = [vp, i64, i64, i64, ctypes.c_int, ctypes.c_int, vp, i64, vp]
    lib.fp8o_quantize_128x128.restype = None
    lib.fp8o_quantize_tensor.argtypes = [vp, i64, ctypes.c_int, f32, vp, vp]
    lib.fp8o_quantize_tensor.restype = None
    lib.fp8o_amax_history_update.argtypes = [vp, vp, i32, f32, ctypes.c_int, i32, vp]
    lib.fp8o_amax_history_update.restype = None
    lib.fp8o_gemm.argtypes = [i64, i64, i64, ctypes.POINTER(Operand), ctypes.POINTER(Operand),
                              i64, vp, i64, vp, vp, vp]
    lib.fp8o_gemm.restype = ctypes.c_int
    lib.fp8o_grouped_gemm.argtypes = [i32, vp, i64, i64, i64, ctypes.POINTER(Operand),
                                      ctypes.POINTER(Operand), i64, vp, i64, vp, vp, vp]
    lib.fp8o_grouped_gemm.restype = ctypes.c_int
    lib.fp8o_attention.argtypes = [i64, i64, i32, i32, ctypes.c_int, ctypes.c_double,
                                   vp, vp, ctypes.c_int, vp, vp, ctypes.c_int, vp, vp, ctypes.c_int,
                                   i64, vp, vp, vp, vp, vp]
    lib.fp8o_attention.restype = ctypes.c_int
    return lib


def build_variant(source: str, name: str) -> str:
    """Compile a modified copy of the oracle source (tests that plant a
    mistake in the oracle use this to show that the pins catch it)."""
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_BUILD, f"{name}.c")
    out = os.path.join(_BUILD, f"{name}_{platform.machine()}.so")
    with open(src, "w") as f:
        f.write(source)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", out, src, "-lm"], check=True)
    return out


class using_library:
    """Context manager: route every oracle call through another compiled
    oracle (a planted-mistake variant) and restore the real one on exit."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self._old = _lib
        _lib = _bind(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._old
        return False


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"] or a.ndim == 0
    return a.ctypes.data


def _bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (numpy uint16)")
    return x


# ------------------------------------------------------------------ formats
def decode(code: int, fmt: int) -> float:
    return _load().fp8o_decode(int(code) & 0xFF, fmt)


def decode_table(fmt: int) -> np.ndarray:
    """fp64 value of each of the 256 codes (NaN for NaN codes)."""
    return np.array([decode(c, fmt) for c in range(256)], dtype=np.float64)


def fmax(fmt: int) -> float:
    return _load().fp8o_fmax(fmt)


def encode(v: float, fmt: int) -> int:
    return int(_load().fp8o_encode(ctypes.c_float(v), fmt))


def encode_array(v: np.ndarray, fmt: int) -> np.ndarray:
    """Element-wise encoder over an fp32 array."""
    flat = np.ascontiguousarray(np.asarray(v, dtype=np.float32).ravel())
    out = np.empty(flat.shape, dtype=np.uint8)
    _load().fp8o_encode_array(_ptr(flat), flat.size, fmt, _ptr(out))
    return out.reshape(np.shape(v))


def bf16_to_f32(h: int) -> float:
    return _load().fp8o_bf16_to_f32(int(h))


def block_scale(amax: float, fmt: int, mode: int) -> float:
    return float(_load().fp8o_block_scale(ctypes.c_float(amax), fmt, mode))


# ------------------------------------------------------------- quantizers
def quantize_1x128(x: np.ndarray, fmt: int = E4M3, mode: int = SCALE_FP32):
    """x: [rows, cols] bf16 bits -> (q [rows, cols] u8, scales [ceil(cols/128), rows] f32)."""
    x = _bf16(x)
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.empty(((cols + 127) // 128, rows), dtype=np.float32)
    _load().fp8o_quantize_1x128(_ptr(x), rows, cols, cols, fmt, mode, _ptr(q), cols, _ptr(s))
    return q, s


def quantize_1x128_f32(y: np.ndarray, fmt: int = E4M3, mode: int = SCALE_FP32):
    """The 1x128 rule on an fp32 matrix (a product's own result, quantized for
    the next linear layer) -> (q [rows, cols] u8, scales [ceil(cols/128), rows])."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    rows, cols = y.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.empty(((cols + 127) // 128, rows), dtype=np.float32)
    _load().fp8o_quantize_1x128_f32(_ptr(y), rows, cols, cols, fmt, mode, _ptr(q), cols, _ptr(s))
    return q, s


def quantize_1x128_colwise(x: np.ndarray, fmt: int = E4M3, mode: int = SCALE_FP32):
    """Column-wise 1x128 tiles (128 consecutive rows of one column), kept as
    the transposed copy: by definition the 1x128 rule applied to x^T.
    x: [rows, cols] bf16 bits -> (qt [cols, rows] u8, scales_t [ceil(rows/128), cols])."""
    return quantize_1x128(np.ascontiguousarray(_bf16(x).T), fmt, mode)


def mx_scale_code(amax: float, fmt: int) -> int:
    """MXFP8 scale code (E8M0) of a 32-element block with this amax."""
    return int(_load().fp8o_mx_scale_code(ctypes.c_float(amax), fmt))


def quantize_mx(x: np.ndarray, fmt: int = E4M3):
    """MXFP8: 32-element blocks along rows, E8M0 scale codes.
    x: [rows, cols] bf16 bits -> (q [rows, cols] u8, scales [ceil(cols/128), rows, 4] u8)."""
    x = _bf16(x)
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.empty(((cols + 127) // 128, rows, 4), dtype=np.uint8)
    _load().fp8o_quantize_mx(_ptr(x), rows, cols, cols, fmt, _ptr(q), cols, _ptr(s))
    return q, s


def quantize_128x128(w: np.ndarray, fmt: int = E4M3, mode: int = SCALE_FP32):
    """w: [rows, cols] bf16 bits -> (q, scales [ceil(rows/128), ceil(cols/128)] f32)."""
    w = _bf16(w)
    rows, cols = w.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.empty(((rows + 127) // 128, (cols + 127) // 128), dtype=np.float32)
    _load().fp8o_quantize_128x128(_ptr(w), rows, cols, cols, fmt, mode, _ptr(q), cols, _ptr(s))
    return q, s


def quantize_tensor(x: np.ndarray, fmt: int, scale: float):
    """Per-tensor quantization with a given dequant scale -> (q, amax)."""
    x = _bf16(x)
    q = np.empty(x.shape, dtype=np.uint8)
    amax = np.zeros(1, dtype=np.float32)
    _load().fp8o_quantize_tensor(_ptr(x), x.size, fmt, ctypes.c_float(scale), _ptr(q), _ptr(amax))
    return q, float(amax[0])


class DelayedState:
    """Per-tensor delayed-scaling state: amax history, head, scale in use."""

    def __init__(self, history_len: int, fmt: int, margin: int = 0):
        self.history = np.zeros(history_len, dtype=np.float32)
        self.head = np.zeros(1, dtype=np.int32)
        self.scale = np.ones(1, dtype=np.float32)
        self.fmt, self.margin = fmt, margin

    def update(self, amax: float) -> float:
        _load().fp8o_amax_history_update(_ptr(self.history), _ptr(self.head), len(self.history),
                                         ctypes.c_float(amax), self.fmt, self.margin, _ptr(self.scale))
        return float(self.scale[0])

    def step(self, x: np.ndarray):
        """Quantize with the scale in use, then fold this step's amax in."""
        q, amax = quantize_tensor(x, self.fmt, float(self.scale[0]))
        self.update(amax)
        return q, amax


# ------------------------------------------------------------------- GEMM
def operand(data: np.ndarray, fmt: int, gran: int, scales: np.ndarray, transposed: bool = False):
    data = np.ascontiguousarray(data, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8 if gran == GRAN_1x32 else np.float32)
    op = Operand(data=_ptr(data), ld=data.shape[-1], transposed=int(transposed), fmt=fmt,
                 gran=gran, pad_=0, scales=_ptr(scales))
    op._keep = (data, scales)
    return op


def _sel(sel, n):
    if sel is None:
        return n, None, None
    a = np.ascontiguousarray(sel, dtype=np.int64)
    return a.size, a, _ptr(a)


def gemm(M: int, N: int, K: int, A: Operand, B: Operand, rows=None, cols=None):
    """fp64 y and sum|terms| for the selected outputs of deq(A) deq(B)^T."""
    nr, r_arr, r_p = _sel(rows, M)
    nc, c_arr, c_p = _sel(cols, N)
    y = np.empty((nr, nc), dtype=np.float64)
    ya = np.empty((nr, nc), dtype=np.float64)
    rc = _load().fp8o_gemm(M, N, K, ctypes.byref(A), ctypes.byref(B), nr, r_p, nc, c_p,
                           _ptr(y), _ptr(ya))
    if rc:
        raise ValueError("oracle gemm: unsupported operand combination or index out of range")
    return y, ya


def grouped_gemm(offsets: np.ndarray, a_rows: int, N: int, K: int, A: Operand, B: Operand,
                 rows=None, cols=None):
    """Grouped product; a_rows = rows of A as stored (>= offsets[-1])."""
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    G = off.size - 1
    nr, r_arr, r_p = _sel(rows, int(off[-1]))
    nc, c_arr, c_p = _sel(cols, N)
    y = np.empty((nr, nc), dtype=np.float64)
    ya = np.empty((nr, nc), dtype=np.float64)
    rc = _load().fp8o_grouped_gemm(G, _ptr(off), a_rows, N, K, ctypes.byref(A), ctypes.byref(B),
                                   nr, r_p, nc, c_p, _ptr(y), _ptr(ya))
    if rc:
        raise ValueError("oracle grouped gemm: unsupported operand combination")
    return y, ya


# ------------------------------------------------------- acceptance rules
def check_f32(y: np.ndarray, y_ref: np.ndarray, yabs: np.ndarray, rel: float = 1e-5):
    """fp32 output bound: |y - y_ref| <= rel * sum|terms| (sum 0 -> y must be 0).
    Returns a boolean mask of elements that FAIL."""
    y = np.asarray(y, dtype=np.float64)
    return ~(np.abs(y - y_ref) <= rel * yabs)


def _bf16_round(v: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 (via fp32, both nearest-even), as bit patterns."""
    import torch
    t = torch.from_numpy(np.asarray(v, dtype=np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _ordinal(b: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> integer that is monotone in the value (+0 and -0 both 0)."""
    b = b.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def check_bf16(y_bits: np.ndarray, y_ref: np.ndarray, yabs: np.ndarray, rel: float = 1e-5):
    """bf16 output: within one bf16 ordinal step of the bf16 rounding of any
    value inside the fp32 bound [y_ref - rel*abs, y_ref + rel*abs].  Away from
    cancellation this is "within 1 ulp of bf16(y_ref)".  Returns FAIL mask."""
    tol = rel * yabs
    lo = _ordinal(_bf16_round(y_ref - tol)) - 1
    hi = _ordinal(_bf16_round(y_ref + tol)) + 1
    o = _ordinal(np.asarray(y_bits, dtype=np.uint16))
    return ~((o >= lo) & (o <= hi))


# ------------------------------------------------------------ SwiGLU
def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """silu(g) * u in fp64 with silu(g) = g / (1 + e^-g): the gated activation
    between an MLP's gate/up product and its down product.  It is one of the
    non-linear functions the NeMo RL page keeps out of FP8 math ("El avance
    tecnico"); here it sits between two FP8 products."""
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def _silu_argmin() -> float:
    """Where silu has its minimum: the root of silu'(x) = s(x) (1 + x (1 - s(x)))
    with s the logistic function, i.e. of 1 + x (1 - s(x)), found by bisection
    on [-2, -1] (the root is near -1.2785)."""
    lo, hi = -2.0, -1.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        f = 1.0 + mid * (1.0 - 1.0 / (1.0 + np.exp(-mid)))
        if f > 0:
            hi = mid
        else:
            lo = mid
    return 0.5 * (lo + hi)


SILU_ARGMIN = _silu_argmin()


def silu_range(lo: np.ndarray, hi: np.ndarray):
    """Element-wise (min, max) of silu over the intervals [lo, hi]: silu falls
    on (-inf, SILU_ARGMIN] and rises after it."""
    lo = np.asarray(lo, dtype=np.float64)
    hi = np.asarray(hi, dtype=np.float64)
    one = np.ones_like(lo)
    a, b = swiglu(lo, one), swiglu(hi, one)
    inside = (lo <= SILU_ARGMIN) & (hi >= SILU_ARGMIN)
    mn = np.where(inside, swiglu(np.float64(SILU_ARGMIN), 1.0), np.minimum(a, b))
    return mn, np.maximum(a, b)


def swiglu_bounds(g, g_tol, u, u_tol, rel: float = 1e-6, rel_g: float = 1e-7):
    """Interval [lo, hi] holding silu(g') * u' for every g' within g_tol of g
    and u' within u_tol of u, widened by (rel + rel_g |g'|) of its magnitude
    for an fp32 evaluation of silu and of the product.  The default slack is
    twice the error of the fast exponential / division forms: the argument
    -g log2(e) is rounded to fp32 (relative error of e^-g up to
    |g| log2(e) 2^-24 ln 2, about 4e-8 |g|) and the base-2 exponential,
    the reciprocal and three roundings add about 5e-7."""
    g = np.asarray(g, dtype=np.float64)
    s_lo, s_hi = silu_range(g - g_tol, g + g_tol)
    u_lo, u_hi = np.asarray(u) - u_tol, np.asarray(u) + u_tol
    prods = np.stack([s_lo * u_lo, s_lo * u_hi, s_hi * u_lo, s_hi * u_hi])
    lo, hi = prods.min(axis=0), prods.max(axis=0)
    slack = (rel + rel_g * (np.abs(g) + g_tol)) * np.maximum(np.abs(lo), np.abs(hi)) + 1e-37
    return lo - slack, hi + slack


# ---------------------------------------------- quantized-output acceptance
def _code_ordinal(c: np.ndarray) -> np.ndarray:
    """8-bit code -> integer monotone in the encoded value (+0 and -0 both 0)."""
    c = np.asarray(c).astype(np.int64)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


def _block_scale_vec(amax: np.ndarray, fmt: int, mode: int) -> np.ndarray:
    flat = np.asarray(amax, dtype=np.float32).ravel()
    out = np.array([block_scale(float(a), fmt, mode) for a in flat], dtype=np.float32)
    return out.reshape(np.shape(amax))


def check_quantized_1x128(q: np.ndarray, s: np.ndarray, lo: np.ndarray, hi: np.ndarray,
                          fmt: int, mode: int):
    """Accept a 1x128 quantization (codes q [rows, cols], scales s [cols/128,
    rows]) of fp32 values that are only known to lie in [lo, hi] (fp64,
    element-wise): a product's result inside its tolerance.
      scale: between the scale rule applied to the smallest and to the largest
             block amax the intervals allow (1 also allowed when the amax can
             be 0: the zero-block rule);
      code:  between enc(fl32(lo32 * r)) and enc(fl32(hi32 * r)) in value
             order, r = fl32(1 / s) the reciprocal of the scale the kernel
             chose, lo32/hi32 the intervals rounded outward to fp32 (the
             encoder and fl32(x * r) are both monotone).
    With lo == hi == an fp32 matrix this is exactly quantize_1x128_f32.
    Returns (bad_scale [cols/128, rows], bad_code [rows, cols]) masks."""
    lo = np.asarray(lo, dtype=np.float64)
    hi = np.asarray(hi, dtype=np.float64)
    rows, cols = lo.shape
    nb = cols // 128
    lo32 = lo.astype(np.float32)
    lo32 = np.where(lo32.astype(np.float64) > lo, np.nextafter(lo32, np.float32(-np.inf)), lo32)
    hi32 = hi.astype(np.float32)
    hi32 = np.where(hi32.astype(np.float64) < hi, np.nextafter(hi32, np.float32(np.inf)), hi32)
    amin = np.where((lo32 <= 0) & (hi32 >= 0), np.float32(0),
                    np.minimum(np.abs(lo32), np.abs(hi32)))
    amaxe = np.maximum(np.abs(lo32), np.abs(hi32))
    blk_lo = amin.reshape(rows, nb, 128).max(axis=2)
    blk_hi = amaxe.reshape(rows, nb, 128).max(axis=2)
    tiny = np.float32(np.finfo(np.float32).smallest_subnormal)
    s_lo = _block_scale_vec(np.maximum(blk_lo, tiny), fmt, mode)
    s_hi = _block_scale_vec(np.maximum(blk_hi, tiny), fmt, mode)
    sg = np.asarray(s, dtype=np.float32).T                       # [rows, nb]
    ok_s = ((sg >= s_lo) & (sg <= s_hi)) | ((blk_lo == 0) & (sg == np.float32(1.0)))
    r = (np.float32(1.0) / sg).astype(np.float32)
    r_e = np.repeat(r, 128, axis=1)
    v_lo = (lo32 * r_e).astype(np.float32)
    v_hi = (hi32 * r_e).astype(np.float32)
    o_lo = _code_ordinal(encode_array(v_lo, fmt))
    o_hi = _code_ordinal(encode_array(v_hi, fmt))
    o = _code_ordinal(q)
    ok_c = (o >= o_lo) & (o <= o_hi)
    return ~ok_s.T, ~ok_c


# ------------------------------------------------------------ attention
def attention(seq_q: int, seq_k: int, hq: int, hkv: int, causal: bool, scale: float,
              q, sq, k, sk, v, sv, rows=None, heads=None, fmts=(E4M3, E4M3, E4M3)):
    """FP8 attention over an FP8 KV cache (fp64 definition, see fp8o_attention).
    q: [seq_q, hq*128] codes, sq: [hq, seq_q] (1x128 scales); k, v: [seq_k, hkv*128]
    codes, sk, sv: [ceil(seq_k/128), hkv] (128x128 scales).  rows/heads select
    (row, head) pairs (default: all).  Returns (o, oap, oav) of shape [n, 128]:
    the output, sum_j P|V|/l and sum_j |V code| svm / l (svm: the head's
    largest V tile scale; see the acceptance rule below)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    k = np.ascontiguousarray(k, dtype=np.uint8)
    v = np.ascontiguousarray(v, dtype=np.uint8)
    sq = np.ascontiguousarray(sq, dtype=np.float32)
    sk = np.ascontiguousarray(sk, dtype=np.float32)
    sv = np.ascontiguousarray(sv, dtype=np.float32)
    if rows is None:
        rr, hh = np.meshgrid(np.arange(seq_q), np.arange(hq), indexing="ij")
        rows, heads = rr.ravel(), hh.ravel()
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    heads = np.ascontiguousarray(heads, dtype=np.int32)
    n = rows.size
    o = np.empty((n, 128), np.float64)
    oap = np.empty((n, 128), np.float64)
    oav = np.empty((n, 128), np.float64)
    rc = _load().fp8o_attention(seq_q, seq_k, hq, hkv, int(causal), float(scale),
                                _ptr(q), _ptr(sq), fmts[0], _ptr(k), _ptr(sk), fmts[1], _ptr(v), _ptr(sv),
                                fmts[2], n, _ptr(rows), _ptr(heads), _ptr(o), _ptr(oap), _ptr(oav))
    if rc:
        raise ValueError("oracle attention: bad arguments")
    return o, oap, oav


# Acceptance rule of the FP8 attention output.  The kernel quantizes the
# softmax numerators P (in [0, 1] after the running-max subtraction), each
# times sv_t / svm (its key tile's V scale over the head's largest, at most
# 1), to E4M3 with the scale 1/448, so each carries a rounding error of at
# most 2^-4 P (normal range) or 2^-10 / 448 * svm / sv_t in P units
# (subnormal range); the row sum l uses the unrounded values.  Hence per
# output element
#   |o - o_ref| <= (2^-4 + 1e-4) sum_j P_j |V_j| / l
#                  + (2^-10 / 448) sum_j |V_j| (svm / sv_t(j)) / l
#                  + 1e-5 |o_ref|   (fp32 scores, exp2, accumulation)
# plus half a bf16 unit of the stored value; the attention oracle returns the
# second sum as oav.
ATTN_P_REL = 2.0 ** -4 + 1e-4
ATTN_P_ABS = 2.0 ** -10 / 448.0


def check_attention_bf16(o_bits: np.ndarray, o_ref: np.ndarray, oap: np.ndarray, oav: np.ndarray):
    """FAIL mask for a bf16 attention output (bit patterns) under the rule above."""
    import torch
    o = torch.from_numpy(np.ascontiguousarray(o_bits, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()
    tol = ATTN_P_REL * oap + ATTN_P_ABS * oav + 1e-5 * np.abs(o_ref) + 2.0 ** -8 * np.abs(o_ref) + 1e-30
    return ~(np.abs(o - o_ref) <= tol)
