"""Plain CPU oracle for the FP8-blk decode GEMV, fused argmax and NVFP4 experts.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``fp8_block_scaled_fp8blk_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``fp8blk_oracle.c`` (plain C, double precision, decode
by table built from the format bit fields).  This module compiles it with gcc on
first use and wraps it with ctypes; it adds no arithmetic of its own.

Every function here is pinned by ``tests/test_oracle_pins.py`` against facts
that do not come from the oracle itself: torch's independent float8 decoders,
the OCP format tables, closed forms, brute force and numpy float64 matmul.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8blk_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (IEEE semantics, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-std=c11", "-Wall", _SRC, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint]
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_e2m1_value.argtypes = [ctypes.c_uint]
        lib.oracle_e8m0_value.restype = ctypes.c_int
        lib.oracle_e8m0_value.argtypes = [ctypes.c_uint, ctypes.POINTER(ctypes.c_double)]
        lib.oracle_e4m3_table.argtypes = [P]
        lib.oracle_e2m1_table.argtypes = [P]
        lib.oracle_bf16_value.restype = ctypes.c_double
        lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_bf16_rne.argtypes = [ctypes.c_double, ctypes.POINTER(ctypes.c_int)]
        lib.oracle_fp8blk_gemv.restype = ctypes.c_int
        lib.oracle_fp8blk_gemv.argtypes = [P, P, P, P, P, ctypes.c_int, I64, I64, ctypes.c_int]
        lib.oracle_argmax.restype = I64
        lib.oracle_argmax.argtypes = [P, I64]
        lib.oracle_nvfp4_dequant_bf16.restype = ctypes.c_int
        lib.oracle_nvfp4_dequant_bf16.argtypes = [P, P, ctypes.c_double, I64, I64, P,
                                                  ctypes.POINTER(I64)]
        lib.oracle_bf16_gemv.restype = ctypes.c_int
        lib.oracle_bf16_gemv.argtypes = [P, P, P, P, ctypes.c_int, I64, I64, ctypes.c_int]
        lib.oracle_nvfp4_expert_dequant_gemv.restype = ctypes.c_int
        lib.oracle_nvfp4_expert_dequant_gemv.argtypes = [P, P, P, ctypes.c_int, P, ctypes.c_int,
                                                         P, P, P, P, I64, I64, ctypes.c_int]
        lib.oracle_mxfp4_expert_gemv.restype = ctypes.c_int
        lib.oracle_mxfp4_expert_gemv.argtypes = [P, P, ctypes.c_int, P, ctypes.c_int, P, P, P, I64, I64,
                                                 ctypes.c_int]
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


class OracleError(ValueError):
    pass


# ---------------------------------------------------------------- decoders
def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(code)


def e4m3_table() -> np.ndarray:
    t = np.empty(256, dtype=np.float64)
    _load().oracle_e4m3_table(_ptr(t))
    return t


def e2m1_value(nibble: int) -> float:
    return _load().oracle_e2m1_value(nibble)


def e2m1_table() -> np.ndarray:
    t = np.empty(16, dtype=np.float64)
    _load().oracle_e2m1_table(_ptr(t))
    return t


def e8m0_value(code: int) -> float:
    """2^(code-127); raises OracleError for the refused code 0xFF."""
    out = ctypes.c_double()
    if _load().oracle_e8m0_value(code, ctypes.byref(out)) != 0:
        raise OracleError(f"e8m0 code {code:#x} is refused")
    return out.value


def bf16_value(bits: int) -> float:
    return _load().oracle_bf16_value(bits)


def bf16_rne(v: float) -> tuple[int, bool]:
    """(bf16 bits nearest to v, ties to even; whether rounding changed v)."""
    inexact = ctypes.c_int()
    bits = _load().oracle_bf16_rne(float(v), ctypes.byref(inexact))
    return int(bits), bool(inexact.value)


# ---------------------------------------------------------------- GEMV
def fp8blk_gemv(codes: np.ndarray, scale_e8m0: np.ndarray, x: np.ndarray,
                nthreads: int = 1) -> tuple[np.ndarray, np.ndarray]:
    """Return (y [m, rows] float64, sum_c |w x| [m, rows] float64).

    codes: uint8 [rows, cols] e4m3; scale_e8m0: uint8 [ceil(rows/128),
    ceil(cols/128)]; x: float32 [m, cols].
    """
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scale_e8m0 = np.ascontiguousarray(scale_e8m0, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    rows, cols = codes.shape
    m = x.shape[0]
    assert x.shape[1] == cols
    assert scale_e8m0.shape == ((rows + 127) // 128, (cols + 127) // 128)
    y = np.zeros((m, rows), dtype=np.float64)
    a = np.zeros((m, rows), dtype=np.float64)
    rc = _load().oracle_fp8blk_gemv(_ptr(codes), _ptr(scale_e8m0), _ptr(x), _ptr(y), _ptr(a),
                                   m, rows, cols, nthreads)
    if rc == -1:
        raise OracleError("e8m0 scale code 0xFF is refused")
    if rc != 0:
        raise OracleError(f"oracle_fp8blk_gemv failed ({rc})")
    return y, a


def argmax(v: np.ndarray) -> int:
    """Lowest index of the maximum; NaN never wins; all -inf/NaN gives 0."""
    v = np.ascontiguousarray(v, dtype=np.float64).ravel()
    return int(_load().oracle_argmax(_ptr(v), v.size))


# ---------------------------------------------------------------- NVFP4
def nvfp4_dequant_bf16(codes: np.ndarray, scales: np.ndarray, g: float) -> tuple[np.ndarray, int]:
    """(bf16 bits uint16 [rows, cols], number of values rounding changed)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, half = codes.shape
    cols = 2 * half
    assert scales.shape == (rows, cols // 16)
    out = np.zeros((rows, cols), dtype=np.uint16)
    nin = ctypes.c_int64()
    rc = _load().oracle_nvfp4_dequant_bf16(_ptr(codes), _ptr(scales), float(g), rows, cols,
                                          _ptr(out), ctypes.byref(nin))
    if rc != 0:
        raise OracleError(f"oracle_nvfp4_dequant_bf16 failed ({rc})")
    return out, int(nin.value)


def bf16_gemv(b: np.ndarray, x: np.ndarray, nthreads: int = 1) -> tuple[np.ndarray, np.ndarray]:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    rows, cols = b.shape
    m = x.shape[0]
    y = np.zeros((m, rows), dtype=np.float64)
    a = np.zeros((m, rows), dtype=np.float64)
    rc = _load().oracle_bf16_gemv(_ptr(b), _ptr(x), _ptr(y), _ptr(a), m, rows, cols, nthreads)
    if rc != 0:
        raise OracleError(f"oracle_bf16_gemv failed ({rc})")
    return y, a


def nvfp4_expert_dequant_gemv(codes: np.ndarray, scales: np.ndarray, gscale: np.ndarray,
                              ids: np.ndarray, x: np.ndarray, nthreads: int = 1,
                              want_scratch: bool = False):
    """(y [n_active, rows], sum|w x| [n_active, rows], last expert's bf16 or None)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    gscale = np.ascontiguousarray(gscale, dtype=np.float32)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    n_experts, rows, half = codes.shape
    cols = 2 * half
    n_active = ids.size
    y = np.zeros((n_active, rows), dtype=np.float64)
    a = np.zeros((n_active, rows), dtype=np.float64)
    scratch = np.zeros((rows, cols), dtype=np.uint16) if want_scratch else None
    rc = _load().oracle_nvfp4_expert_dequant_gemv(
        _ptr(codes), _ptr(scales), _ptr(gscale), n_experts, _ptr(ids), n_active, _ptr(x),
        _ptr(y), _ptr(a), _ptr(scratch) if scratch is not None else None, rows, cols, nthreads)
    if rc == -4:
        raise OracleError("expert id out of range or repeated")
    if rc != 0:
        raise OracleError(f"oracle_nvfp4_expert_dequant_gemv failed ({rc})")
    return y, a, scratch


def mxfp4_expert_gemv(codes: np.ndarray, scales: np.ndarray, ids: np.ndarray, x: np.ndarray,
                      nthreads: int = 1) -> tuple[np.ndarray, np.ndarray]:
    """OCP MXFP4 experts: (y [n_active, rows], sum|w x| [n_active, rows]) with
    y[k][r] = sum_c e2m1(codes[ids[k]][r][c]) * 2^(scales[ids[k]][r][c/32] - 127) * x[c]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    n_experts, rows, half = codes.shape
    cols = 2 * half
    assert scales.shape == (n_experts, rows, cols // 32) and x.size == cols
    y = np.zeros((ids.size, rows), dtype=np.float64)
    a = np.zeros((ids.size, rows), dtype=np.float64)
    rc = _load().oracle_mxfp4_expert_gemv(_ptr(codes), _ptr(scales), n_experts, _ptr(ids), ids.size, _ptr(x),
                                          _ptr(y), _ptr(a), rows, cols, nthreads)
    if rc == -4:
        raise OracleError("expert id out of range")
    if rc != 0:
        raise OracleError(f"oracle_mxfp4_expert_gemv failed ({rc})")
    return y, a
