"""C-ABI checks that need no GPU: the library loads, exports every function
include/fp8bs.h declares, and rejects bad arguments on the host (status
codes, message) before anything is launched."""
import ctypes
import os
import re

import pytest

import block_scaled_gemm_quantize_gb300 as fp8
from block_scaled_gemm_quantize_gb300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bs.h")


@pytest.fixture(scope="module")
def L():
    fbuild.build()
    return fp8.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fp8\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_six_entry_points():
    names = _declared()
    for n in ["fp8_quantize_1x128", "fp8_quantize_128x128", "fp8_quantize_tensor_delayed",
              "fp8_amax_history_update", "fp8_block_gemm", "fp8_grouped_block_gemm"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    assert L.fp8bs_version() == 1


FAKE = 0x10000000  # aligned, never dereferenced: every call below fails validation first


def _err(L):
    return L.fp8bs_last_error().decode()


def test_quantize_validation(L):
    f = L.fp8_quantize_1x128
    assert f(None, 4, 256, 256, 0, 0, FAKE, 256, FAKE, None) == -1          # null x
    assert "null" in _err(L)
    assert f(FAKE, 4, 200, 200, 0, 0, FAKE, 208, FAKE, None) == -2          # cols % 128
    assert f(FAKE + 2, 4, 256, 256, 0, 0, FAKE, 256, FAKE, None) == -3      # misaligned x
    assert f(FAKE, 4, 256, 260, 0, 0, FAKE, 256, FAKE, None) == -3         # ld_x*2 % 16
    assert f(FAKE, 4, 256, 256, 7, 0, FAKE, 256, FAKE, None) == -1          # bad format
    assert f(FAKE, 4, 256, 128, 0, 0, FAKE, 256, FAKE, None) == -1          # ld < cols
    assert f(FAKE, 0, 256, 256, 0, 0, FAKE, 256, FAKE, None) == 0           # empty: no launch
    assert f(FAKE, -1, 256, 256, 0, 0, FAKE, 256, FAKE, None) == -1
    g = L.fp8_quantize_128x128
    assert g(FAKE, 4, 384, 384, 1, 3, FAKE, 384, FAKE, None) == -1          # bad mode
    assert g(FAKE, 4, 384, 384, 1, 1, FAKE + 8, 384, FAKE, None) == -3
    assert g(FAKE, 5, 0, 0, 1, 1, FAKE, 0, FAKE, None) == 0


def test_delayed_validation(L):
    f = L.fp8_quantize_tensor_delayed
    assert f(FAKE, 100, 1, None, FAKE, FAKE, None) == -1
    assert f(FAKE, -3, 1, FAKE, FAKE, FAKE, None) == -1
    assert f(FAKE + 4, 64, 1, FAKE, FAKE, FAKE, None) == -3
    h = L.fp8_amax_history_update
    assert h(FAKE, FAKE, 0, FAKE, 0, 0, FAKE, None) == -1                   # history_len < 1
    assert h(FAKE, FAKE, 16, FAKE, 0, 200, FAKE, None) == -1                # margin range
    assert h(None, FAKE, 16, FAKE, 0, 0, FAKE, None) == -1


def _op(data=FAKE, ld=512, transposed=0, fmt=0, gran=0, scales=FAKE):
    return fp8.Operand(data=data, ld=ld, transposed=transposed, fmt=fmt, gran=gran, reserved=0,
                       scales=scales)


def test_gemm_validation(L):
    g = L.fp8_block_gemm
    A, B = _op(gran=0), _op(gran=1)
    by = ctypes.byref
    assert g(256, 256, 500, by(A), by(B), 0, FAKE, 256, 1, None) == -2      # K % 128
    assert g(256, 250, 512, by(A), by(B), 0, FAKE, 256, 1, None) == -2      # N % 8
    assert g(256, 256, 512, by(A), by(_op(gran=0, transposed=1, ld=256)), 0, FAKE, 256, 1, None) == -2
    assert g(256, 256, 512, by(_op(gran=1, transposed=1, ld=256)), by(_op(gran=0)), 0, FAKE, 256, 1,
             None) == -2                                                    # 1x128 B, A^T
    assert g(256, 256, 512, by(_op(gran=0, transposed=1, ld=256)), by(B), 0, FAKE, 256, 1, None) == -2
    assert g(256, 256, 512, by(A), by(B), 0, FAKE + 8, 256, 1, None) == -3  # Y alignment
    assert g(256, 256, 512, by(A), by(B), 0, FAKE, 260, 1, None) == -3      # ld_y pitch
    assert g(256, 256, 512, by(_op(data=FAKE + 16, ld=520)), by(B), 0, FAKE, 256, 1, None) == -3
    assert g(256, 256, 512, by(A), by(B), 0, None, 256, 1, None) == -1
    assert g(256, 256, 512, by(A), by(B), 5, FAKE, 256, 1, None) == -1      # bad mode
    assert g(256, 256, 512, by(A), by(B), 0, FAKE, 256, 9, None) == -1      # bad out dtype
    assert g(256, 256, 512, by(_op(fmt=3)), by(B), 0, FAKE, 256, 1, None) == -1
    assert g(0, 256, 512, by(A), by(B), 0, FAKE, 256, 1, None) == 0        # empty
    assert g(256, 0, 512, by(A), by(B), 0, FAKE, 256, 1, None) == 0
    Bc = _op(gran=0)                                                        # 1x128 B (per-column scales)
    assert g(254, 256, 512, by(A), by(Bc), 0, FAKE, 256, 1, None) == -2     # rows of A % 4
    assert g(256, 256, 512, by(A), by(_op(gran=0, scales=FAKE + 4)), 0, FAKE, 256, 1, None) == -3
    assert L.fp8_block_gemm_quant(256, 256, 512, by(A), by(Bc), 0, 0, 0, 0, FAKE, 256, FAKE, None) == -2
    gg = L.fp8_grouped_block_gemm
    assert gg(0, FAKE, 1024, 256, 512, by(A), by(B), 0, FAKE, 256, 1, None) == -1   # G < 1
    assert gg(2000, FAKE, 1024, 256, 512, by(A), by(B), 0, FAKE, 256, 1, None) == -1
    assert gg(8, None, 1024, 256, 512, by(A), by(B), 0, FAKE, 256, 1, None) == -1
    assert gg(8, FAKE, 1024, 256, 512, by(A), by(_op(transposed=1, gran=1, ld=256)), 0, FAKE, 256, 1,
              None) == -2
    assert gg(8, FAKE, 1024, 256, 512, by(_op(gran=1)), by(B), 0, FAKE, 256, 1, None) == -2
    assert gg(8, FAKE, 1024, 256, 512, by(A), by(_op(gran=0)), 0, FAKE, 256, 1, None) == -2


def test_quantized_output_validation(L):
    g = L.fp8_block_gemm_quant
    A, B = _op(gran=0), _op(gran=1)
    by = ctypes.byref
    #        M    N    K    A      B      mode epi fmt qmode Q     ld_q  scales
    assert g(256, 640, 512, by(A), by(B), 0, 1, 0, 0, FAKE, 320, FAKE, None) == -2  # SwiGLU N % 256
    assert g(256, 200, 512, by(A), by(B), 0, 0, 0, 0, FAKE, 208, FAKE, None) == -2  # N % 128
    assert g(256, 512, 512, by(A), by(B), 0, 7, 0, 0, FAKE, 512, FAKE, None) == -1  # bad epilogue
    assert g(256, 512, 512, by(A), by(B), 0, 0, 4, 0, FAKE, 512, FAKE, None) == -1  # bad q format
    assert g(256, 512, 512, by(A), by(B), 0, 0, 0, 9, FAKE, 512, FAKE, None) == -1  # bad q mode
    assert g(256, 512, 512, by(A), by(B), 0, 0, 0, 0, None, 512, FAKE, None) == -1  # null Q
    assert g(256, 512, 512, by(A), by(B), 0, 0, 0, 0, FAKE, 512, None, None) == -1  # null scales
    assert g(256, 512, 512, by(A), by(B), 0, 0, 0, 0, FAKE + 8, 512, FAKE, None) == -3
    assert g(256, 512, 512, by(A), by(B), 0, 0, 0, 0, FAKE, 520, FAKE, None) == -3  # ld_q % 16
    assert g(256, 512, 512, by(A), by(B), 0, 0, 0, 0, FAKE, 512, FAKE + 2, None) == -3
    assert g(256, 512, 512, by(A), by(B), 0, 1, 0, 0, FAKE, 128, FAKE, None) == -1  # ld_q < N/2
    assert g(256, 512, 512, by(A), by(_op(gran=1, transposed=1, ld=512)), 0, 1, 0, 0, FAKE, 256, FAKE,
             None) == -2                                                            # SwiGLU, B^T
    assert g(0, 512, 512, by(A), by(B), 0, 1, 0, 0, FAKE, 256, FAKE, None) == 0     # empty
    gg = L.fp8_grouped_block_gemm_quant
    assert gg(4, None, 1024, 512, 512, by(A), by(B), 0, 1, 0, 0, FAKE, 256, FAKE, None) == -1
    assert gg(0, FAKE, 1024, 512, 512, by(A), by(B), 0, 1, 0, 0, FAKE, 256, FAKE, None) == -1


def test_colwise_quantizer_validation(L):
    f = L.fp8_quantize_1x128_colwise
    #        x     rows cols ld   fmt mode qt    ld_qt st    q     ld_q sc
    assert f(FAKE, 200, 384, 384, 0, 0, FAKE, 208, FAKE, None, 0, None, None) == -2   # rows % 128
    assert f(FAKE, 256, 200, 200, 0, 0, FAKE, 256, FAKE, None, 0, None, None) == -2   # cols % 128
    assert f(FAKE, 256, 384, 384, 0, 0, None, 256, FAKE, None, 0, None, None) == -1   # null qt
    assert f(FAKE, 256, 384, 384, 0, 0, FAKE, 256, FAKE, FAKE, 384, None, None) == -1  # q without scales
    assert f(FAKE, 256, 384, 384, 0, 0, FAKE, 128, FAKE, None, 0, None, None) == -1   # ld_qt < rows
    assert f(FAKE, 256, 384, 384, 0, 0, FAKE + 8, 256, FAKE, None, 0, None, None) == -3
    assert f(FAKE, 256, 384, 384, 0, 2, FAKE, 256, FAKE, None, 0, None, None) == -1   # bad mode
    assert f(FAKE, 0, 384, 384, 0, 0, FAKE, 0, FAKE, None, 0, None, None) == 0        # empty


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 128, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        fp8.fp8_quantize_1x128(x)


def test_quantize_linear_validation(L):
    f = L.fp8_quantize_linear
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p]
    ok = (FAKE, 4, 256, FAKE, 256, FAKE)
    assert f(None, 4, 256, FAKE, 256, FAKE, *ok, 256, 0, 0, None) == -1    # null x
    assert f(*ok, FAKE, 4, 256, None, 256, FAKE, 256, 0, 0, None) == -1    # null qw
    assert f(*ok, FAKE + 2, 4, 256, FAKE, 256, FAKE, 256, 0, 0, None) == -3  # misaligned w
    assert f(*ok, *ok, 200, 0, 0, None) == -2                              # k % 128
    assert f(*ok, *ok, 256, 0, 5, None) == -1                              # bad mode
    assert f(*ok, *ok, -1, 0, 0, None) == -1                               # negative size
    assert f(FAKE, 0, 256, FAKE, 256, FAKE, FAKE, 0, 256, FAKE, 256, FAKE, 256, 0, 0, None) == 0  # empty
