"""Seeded synthetic inputs for the FP8-blk GEMV, head argmax and NVFP4 experts.

This module only draws random codes and activations with the distributions of
the workloads below.  It holds none of the method's arithmetic (no decoding,
no scaling, no dot products), so both the CUDA path and the CPU oracle can be
fed from it without sharing any computation.

Distributions (numpy ``default_rng(seed)``):
  * e4m3 weight codes: uniform over the 254 finite codes 0x00..0x7E, 0x80..0xFE
    (the two NaN codes 0x7F and 0xFF are never drawn).
  * e8m0 block-scale codes: 127 + e, e uniform integer in [-8, 0].
  * activations: float32 N(0, 1).
  * NVFP4 codes: both nibbles of every byte uniform over the 16 e2m1 codes.
  * NVFP4 block scales (one e4m3 per 16 columns): sign 0, biased exponent
    e + 7 with e uniform in [-6, 2], mantissa uniform in 0..7 (normal values).
  * NVFP4 global scale: 2^-4 for every expert.
  * active expert ids: ``rng.choice(n_experts, n_active, replace=False)``.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# Named workloads: (rows, cols, m) for the FP8-blk GEMV family.
WORKLOADS = {
    "gemv_512x1024_m1": dict(rows=512, cols=1024, m=1, seed=0),
    "gemv_4096x4096_m1": dict(rows=4096, cols=4096, m=1, seed=1),
    "head_argmax_131072x4096_m1": dict(rows=131072, cols=4096, m=1, seed=2),
    "verify_16384x4096_m8": dict(rows=16384, cols=4096, m=8, seed=3),
}
NVFP4_WORKLOAD = dict(n_experts=64, rows=2048, cols=4096, n_active=6, seed=4)
# The MTP block's routed experts (OCP MXFP4), same expert geometry as the trunk's.
MXFP4_WORKLOAD = dict(n_experts=64, rows=2048, cols=4096, n_active=6, seed=5)


@dataclass
class Mxfp4Case:
    codes: np.ndarray    # uint8 [n_experts, rows, cols/2], column 2j in the low nibble
    scales: np.ndarray   # uint8 e8m0 [n_experts, rows, cols/32]
    ids: np.ndarray      # int32 [n_active]
    x: np.ndarray        # float32 [cols]


@dataclass
class Fp8BlkCase:
    codes: np.ndarray       # uint8 [rows, cols]
    scale_e8m0: np.ndarray  # uint8 [ceil(rows/128), ceil(cols/128)]
    x: np.ndarray           # float32 [m, cols]


@dataclass
class Nvfp4Case:
    codes: np.ndarray    # uint8 [n_experts, rows, cols/2]
    scales: np.ndarray   # uint8 e4m3 [n_experts, rows, cols/16]
    gscale: np.ndarray   # float32 [n_experts]
    ids: np.ndarray      # int32 [n_active]
    x: np.ndarray        # float32 [cols]


def finite_e4m3_codes(rng: np.random.Generator, shape) -> np.ndarray:
    k = rng.integers(0, 254, size=shape, dtype=np.uint8)
    # 0..126 stay, 127..253 move up by one: 0x7F is skipped and 0xFF unreachable.
    return np.where(k >= 127, k + np.uint8(1), k).astype(np.uint8)


def e8m0_codes(rng: np.random.Generator, shape, lo: int = -8, hi: int = 0) -> np.ndarray:
    return (127 + rng.integers(lo, hi + 1, size=shape)).astype(np.uint8)


def fp8blk_case(rows: int, cols: int, m: int, seed: int) -> Fp8BlkCase:
    rng = np.random.default_rng(seed)
    codes = finite_e4m3_codes(rng, (rows, cols))
    scale = e8m0_codes(rng, ((rows + 127) // 128, (cols + 127) // 128))
    x = rng.standard_normal((m, cols), dtype=np.float32)
    return Fp8BlkCase(codes, scale, x)


def workload_case(name: str) -> Fp8BlkCase:
    w = WORKLOADS[name]
    return fp8blk_case(w["rows"], w["cols"], w["m"], w["seed"])


def nvfp4_scale_codes(rng: np.random.Generator, shape) -> np.ndarray:
    e = rng.integers(-6, 3, size=shape)
    mant = rng.integers(0, 8, size=shape)
    return (((e + 7) << 3) | mant).astype(np.uint8)


def nvfp4_case(n_experts: int, rows: int, cols: int, n_active: int, seed: int,
               gscale: float = 2.0 ** -4) -> Nvfp4Case:
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=(n_experts, rows, cols // 2), dtype=np.uint8)
    scales = nvfp4_scale_codes(rng, (n_experts, rows, cols // 16))
    g = np.full(n_experts, gscale, dtype=np.float32)
    ids = rng.choice(n_experts, n_active, replace=False).astype(np.int32)
    x = rng.standard_normal(cols, dtype=np.float32)
    return Nvfp4Case(codes, scales, g, ids, x)


def mxfp4_case(n_experts: int, rows: int, cols: int, n_active: int, seed: int) -> Mxfp4Case:
    """e2m1 codes uniform over all 16; e8m0 block scales 2^[-8, 0] (codes 119..127)."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=(n_experts, rows, cols // 2), dtype=np.uint8)
    scales = e8m0_codes(rng, (n_experts, rows, cols // 32))
    ids = rng.choice(n_experts, n_active, replace=False).astype(np.int32)
    x = rng.standard_normal(cols, dtype=np.float32)
    return Mxfp4Case(codes, scales, ids, x)
