"""Thin ctypes binding of libfp8blk (C ABI in ``include/fp8blk.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of the library.  Tensors are torch CUDA tensors (torch is used for
device memory and streams); each call enqueues on the current torch stream of
the tensors' device and returns without synchronizing.  Importing this module
loads the library and raises ``ImportError`` if it has not been built, so the
product path can never run without its kernels.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from .build import LIB as _LIB_PATH

library_path = _LIB_PATH

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"libfp8blk is not built ({_LIB_PATH} missing); run "
        "`python -m fp8_block_scaled_fp8blk_gb300.build` (or __graft_entry__.build())")

_lib = ctypes.CDLL(_LIB_PATH)

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int

_lib.fp8blk_abi_version.restype = _INT
_lib.fp8blk_strerror.restype = ctypes.c_char_p
_lib.fp8blk_strerror.argtypes = [_INT]
_lib.fp8blk_scales_from_e8m0.restype = _INT
_lib.fp8blk_scales_from_e8m0.argtypes = [_P, ctypes.c_size_t, _P, ctypes.POINTER(ctypes.c_size_t)]
_lib.fp8blk_gemv.restype = _INT
_lib.fp8blk_gemv.argtypes = [_P, _P, _P, _P, _INT, _I64, _I64, _P]
_lib.fp8blk_gemv_argmax_ws_bytes.restype = ctypes.c_size_t
_lib.fp8blk_gemv_argmax_ws_bytes.argtypes = [_INT, _I64, _I64]
_lib.fp8blk_gemv_argmax.restype = _INT
_lib.fp8blk_gemv_argmax.argtypes = [_P, _P, _P, _P, _P, _P, ctypes.c_size_t, _INT, _I64, _I64, _P]
_lib.fp8blk_gemv_argmax_noalloc.restype = _INT
_lib.fp8blk_gemv_argmax_noalloc.argtypes = [_P, _P, _P, _P, _P, _INT, _I64, _I64, _P]
_lib.fp8blk_noalloc_scratch_bytes.restype = ctypes.c_size_t
_lib.fp8blk_bf16_gemv.restype = _INT
_lib.fp8blk_bf16_gemv.argtypes = [_P, _P, _P, _INT, _I64, _I64, _P]
_lib.nvfp4_expert_dequant.restype = _INT
_lib.nvfp4_expert_dequant.argtypes = [_P, _P, _P, _INT, _INT, _P, _I64, _I64, _P]
_lib.nvfp4_expert_dequant_gemv.restype = _INT
_lib.nvfp4_expert_dequant_gemv.argtypes = [_P, _P, _P, _INT, _P, _INT, _P, _P, _P, _I64, _I64, _P]
_lib.nvfp4_expert_gemv.restype = _INT
_lib.nvfp4_expert_gemv.argtypes = [_P, _P, _P, _INT, _P, _INT, _P, _P, _I64, _I64, _P]
_lib.mxfp4_expert_gemv.restype = _INT
_lib.mxfp4_expert_gemv.argtypes = [_P, _P, _INT, _P, _INT, _P, _P, _I64, _I64, _P]
_lib.fp8blk_set_launch_tuning.restype = _INT
_lib.fp8blk_set_launch_tuning.argtypes = [_INT, _INT, _INT, _INT, _INT]
_lib.fp8blk_set_m1_kernel.restype = _INT
_lib.fp8blk_set_m1_kernel.argtypes = [_INT, _I64]
_lib.fp8blk_set_fp4_kernel.restype = _INT
_lib.fp8blk_set_fp4_kernel.argtypes = [_INT]
_lib.fp8blk_set_wait_limit.restype = _INT
_lib.fp8blk_set_wait_limit.argtypes = [_I64]
_lib.fp8blk_set_tensor_core_min_m.restype = _INT
_lib.fp8blk_set_tensor_core_min_m.argtypes = [_INT, _I64]
_lib.fp8blk_plan_query.restype = _INT
_lib.fp8blk_plan_query.argtypes = [_INT, _I64, _I64, _INT, _INT, _INT, _INT, _P]
_lib.fp8blk_device_status.restype = _INT
_lib.fp8blk_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), _INT]

# Return codes (include/fp8blk.h)
OK, EINVAL, EALIGN, ESCALE, EWS, ECUDA, ERANGE = 0, 1, 2, 3, 4, 5, 6
STATUS_WAIT_TIMEOUT = 1
STATUS_BAD_EXPERT = 2


class Fp8BlkError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {_lib.fp8blk_strerror(code).decode()} (code {code})")


def _check(rc: int, where: str) -> None:
    if rc != OK:
        raise Fp8BlkError(rc, where)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(t: torch.Tensor) -> int:
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    return torch.cuda.current_stream(t.device).cuda_stream


def abi_version() -> int:
    return _lib.fp8blk_abi_version()


# ---------------------------------------------------------------- host helper
def fp8blk_scales_from_e8m0(codes: np.ndarray | torch.Tensor) -> np.ndarray:
    """Decode an e8m0 scale grid on the host (same shape, float32)."""
    if isinstance(codes, torch.Tensor):
        codes = codes.cpu().numpy()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float32)
    bad = ctypes.c_size_t(0)
    rc = _lib.fp8blk_scales_from_e8m0(codes.ctypes.data, codes.size, out.ctypes.data,
                                      ctypes.byref(bad))
    if rc == ESCALE:
        raise Fp8BlkError(rc, f"fp8blk_scales_from_e8m0 (flat index {bad.value})")
    _check(rc, "fp8blk_scales_from_e8m0")
    return out


# ---------------------------------------------------------------- GEMV
def fp8blk_gemv(w_codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor,
                y: torch.Tensor | None = None) -> torch.Tensor:
    """y [m, rows] = decode(w_codes [rows, cols] e4m3 x scales [rows/128, cols/128]) @ x.T."""
    rows, cols = w_codes.shape
    x2 = x if x.dim() == 2 else x.view(1, -1)
    m = x2.shape[0]
    if y is None:
        y = torch.empty((m, rows), dtype=torch.float32, device=x.device)
    _check(_lib.fp8blk_gemv(_ptr(w_codes), _ptr(scales), _ptr(x2), _ptr(y), m, rows, cols,
                            _stream(x)), "fp8blk_gemv")
    return y


def fp8blk_gemv_argmax_ws_bytes(m: int, rows: int, cols: int) -> int:
    return int(_lib.fp8blk_gemv_argmax_ws_bytes(m, rows, cols))


def argmax_workspace(m: int, rows: int, cols: int, device) -> torch.Tensor:
    """A zero-filled workspace of the size fp8blk_gemv_argmax needs."""
    n = fp8blk_gemv_argmax_ws_bytes(m, rows, cols)
    if n == 0:
        raise Fp8BlkError(EINVAL, "fp8blk_gemv_argmax_ws_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def fp8blk_gemv_argmax(w_codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor,
                       ws: torch.Tensor, tokens: torch.Tensor | None = None,
                       logits: torch.Tensor | None = None) -> torch.Tensor:
    """Greedy tokens [m] (uint32 as int32 storage) of decode(W) @ x.T; logits optional."""
    rows, cols = w_codes.shape
    x2 = x if x.dim() == 2 else x.view(1, -1)
    m = x2.shape[0]
    if tokens is None:
        tokens = torch.empty(m, dtype=torch.int32, device=x.device)
    _check(_lib.fp8blk_gemv_argmax(_ptr(w_codes), _ptr(scales), _ptr(x2), _ptr(logits),
                                   _ptr(tokens), _ptr(ws), ws.numel() * ws.element_size(), m,
                                   rows, cols, _stream(x)), "fp8blk_gemv_argmax")
    return tokens


def fp8blk_gemv_argmax_noalloc(w_codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor,
                               tokens: torch.Tensor | None = None,
                               logits: torch.Tensor | None = None) -> torch.Tensor:
    """fp8blk_gemv_argmax with the library's own fixed device scratch (no workspace).

    For callers that cannot allocate device memory; calls must not overlap on the GPU.
    """
    rows, cols = w_codes.shape
    x2 = x if x.dim() == 2 else x.view(1, -1)
    m = x2.shape[0]
    if tokens is None:
        tokens = torch.empty(m, dtype=torch.int32, device=x.device)
    _check(_lib.fp8blk_gemv_argmax_noalloc(_ptr(w_codes), _ptr(scales), _ptr(x2), _ptr(logits),
                                           _ptr(tokens), m, rows, cols, _stream(x)),
           "fp8blk_gemv_argmax_noalloc")
    return tokens


def fp8blk_bf16_gemv(w_bf16: torch.Tensor, x: torch.Tensor,
                     y: torch.Tensor | None = None) -> torch.Tensor:
    rows, cols = w_bf16.shape
    x2 = x if x.dim() == 2 else x.view(1, -1)
    m = x2.shape[0]
    if y is None:
        y = torch.empty((m, rows), dtype=torch.float32, device=x.device)
    _check(_lib.fp8blk_bf16_gemv(_ptr(w_bf16), _ptr(x2), _ptr(y), m, rows, cols, _stream(x)),
           "fp8blk_bf16_gemv")
    return y


# ---------------------------------------------------------------- NVFP4 experts
def _host_f32(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def _host_i32(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def nvfp4_expert_dequant(codes: torch.Tensor, scales: torch.Tensor, gscale, expert_id: int,
                         out: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 bits (int16 storage) [rows, cols] of expert `expert_id`."""
    n_experts, rows, half = codes.shape
    cols = 2 * half
    g = _host_f32(gscale)
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.int16, device=codes.device)
    _check(_lib.nvfp4_expert_dequant(_ptr(codes), _ptr(scales), g.ctypes.data, n_experts,
                                     int(expert_id), _ptr(out), rows, cols, _stream(codes)),
           "nvfp4_expert_dequant")
    return out


def nvfp4_expert_dequant_gemv(codes: torch.Tensor, scales: torch.Tensor, gscale, ids,
                              x: torch.Tensor, scratch: torch.Tensor,
                              y: torch.Tensor | None = None) -> torch.Tensor:
    """y [n_active, rows]: each active expert dequantised into `scratch`, then GEMV'd."""
    n_experts, rows, half = codes.shape
    cols = 2 * half
    g = _host_f32(gscale)
    ids_h = _host_i32(ids)
    if y is None:
        y = torch.empty((ids_h.size, rows), dtype=torch.float32, device=x.device)
    _check(_lib.nvfp4_expert_dequant_gemv(_ptr(codes), _ptr(scales), g.ctypes.data, n_experts,
                                          ids_h.ctypes.data, ids_h.size, _ptr(x), _ptr(y),
                                          _ptr(scratch), rows, cols, _stream(x)),
           "nvfp4_expert_dequant_gemv")
    return y


def nvfp4_expert_gemv(codes: torch.Tensor, scales: torch.Tensor, gscale: torch.Tensor, ids: torch.Tensor,
                      x: torch.Tensor, y: torch.Tensor | None = None) -> torch.Tensor:
    """y [n_active, rows] = W(ids[k]) x in one launch (CUDA cores or tensor
    cores, see set_fp4_kernel); `gscale` (f32 [n_experts]) and `ids` (int32
    [n_active]) stay on the device."""
    n_experts, rows, half = codes.shape
    cols = 2 * half
    if gscale.dtype != torch.float32 or ids.dtype != torch.int32:
        raise TypeError("gscale must be float32 and ids int32 device tensors")
    n_active = ids.numel()
    if y is None:
        y = torch.empty((n_active, rows), dtype=torch.float32, device=x.device)
    _check(_lib.nvfp4_expert_gemv(_ptr(codes), _ptr(scales), _ptr(gscale), n_experts, _ptr(ids), n_active,
                                  _ptr(x), _ptr(y), rows, cols, _stream(x)), "nvfp4_expert_gemv")
    return y


def mxfp4_expert_gemv(codes: torch.Tensor, scales: torch.Tensor, ids: torch.Tensor, x: torch.Tensor,
                      y: torch.Tensor | None = None) -> torch.Tensor:
    """OCP MXFP4 experts: y [n_active, rows] = W(ids[k]) x in one launch
    (e8m0 scale per 32 columns; CUDA cores or tensor cores, see
    set_fp4_kernel; `ids` int32 on the device)."""
    n_experts, rows, half = codes.shape
    cols = 2 * half
    if ids.dtype != torch.int32:
        raise TypeError("ids must be an int32 device tensor")
    n_active = ids.numel()
    if y is None:
        y = torch.empty((n_active, rows), dtype=torch.float32, device=x.device)
    _check(_lib.mxfp4_expert_gemv(_ptr(codes), _ptr(scales), n_experts, _ptr(ids), n_active, _ptr(x), _ptr(y),
                                  rows, cols, _stream(x)), "mxfp4_expert_gemv")
    return y


# ---------------------------------------------------------------- control
def set_launch_tuning(target_stage_bytes: int = 0, ctas_per_sm: int = 0, use_pdl: int = 1,
                      l2_prefetch: int = 1, max_stages: int = 0) -> None:
    _check(_lib.fp8blk_set_launch_tuning(target_stage_bytes, ctas_per_sm, use_pdl, l2_prefetch,
                                         max_stages), "fp8blk_set_launch_tuning")


PLAN_FIELDS = ("panels", "panel_cols", "team_warps", "teams", "row_batches", "rows_per_batch",
               "stage_rows", "stage_bytes", "stages", "ctas_per_sm", "n_groups",
               "dynamic_smem_bytes", "kernel")


def plan_query(m: int, rows: int, cols: int, bytes_per_weight: int = 1, sms: int = 152,
               smem_per_sm: int = 233472, smem_per_block: int = 232448) -> dict:
    """Launch geometry for a shape on a device with the given facts (host only)."""
    out = np.zeros(13, dtype=np.int64)
    _check(_lib.fp8blk_plan_query(m, rows, cols, bytes_per_weight, sms, smem_per_sm,
                                  smem_per_block, out.ctypes.data), "fp8blk_plan_query")
    return dict(zip(PLAN_FIELDS, (int(v) for v in out)))


def set_m1_kernel(choice: int = 0, rowwarp_min_bytes: int = 0) -> None:
    """m = 1 kernel: 0 by size, 1 row-per-warp, 2 team (speed only)."""
    _check(_lib.fp8blk_set_m1_kernel(choice, rowwarp_min_bytes), "fp8blk_set_m1_kernel")


def set_fp4_kernel(choice: int = 0) -> None:
    """NVFP4 and MXFP4 expert GEMV kernel: 0 by shape (tensor cores from
    12288 active rows on), 1 CUDA cores, 2 tensor cores."""
    _check(_lib.fp8blk_set_fp4_kernel(choice), "fp8blk_set_fp4_kernel")


def set_tensor_core_min_m(min_m: int = 0, min_bytes: int = 0) -> None:
    """e4m3 GEMVs with m >= min_m (2..8; 9 = never) and at least min_bytes of
    weights (1 = any) run on the tensor cores; 0 restores a default."""
    _check(_lib.fp8blk_set_tensor_core_min_m(min_m, min_bytes), "fp8blk_set_tensor_core_min_m")


WAIT_LIMIT_DEFAULT_NS = 1_000_000_000


def set_wait_limit(limit_ns: int = WAIT_LIMIT_DEFAULT_NS) -> None:
    """How long a CUDA-core GEMV thread waits for a weight tile before giving
    up (status FP8BLK_STATUS_WAIT_TIMEOUT); the default is about one second."""
    _check(_lib.fp8blk_set_wait_limit(int(limit_ns)), "fp8blk_set_wait_limit")


def fp8blk_device_status(clear: bool = False) -> int:
    """Device status word (0 = healthy).  Synchronizes the current device."""
    v = ctypes.c_uint32(0)
    _check(_lib.fp8blk_device_status(ctypes.byref(v), int(clear)), "fp8blk_device_status")
    return int(v.value)


def raw_library() -> ctypes.CDLL:
    """The loaded ctypes library, for callers that pass raw pointers."""
    return _lib
