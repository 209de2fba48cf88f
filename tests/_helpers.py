"""Shared helpers for the GPU parity tests (tolerance, uploads, sampling)."""
import numpy as np

# Per-element bound: |gpu - oracle| <= REL * sum_c |w x| + ABS.
REL = 1e-5
ABS = 1e-6


def within_tolerance(gpu: np.ndarray, ref: np.ndarray, abs_sum: np.ndarray):
    """(ok, worst ratio err / bound) for f32 GPU outputs against double oracle."""
    gpu = np.asarray(gpu, dtype=np.float64)
    bound = REL * abs_sum + ABS
    err = np.abs(gpu - ref)
    ratio = err / bound
    ok = bool(np.all(err <= bound)) and not np.isnan(gpu).any()
    return ok, float(np.nanmax(ratio)) if ratio.size else 0.0


def assert_close(gpu, ref, abs_sum, what=""):
    ok, worst = within_tolerance(gpu, ref, abs_sum)
    assert ok, f"{what}: worst err/bound = {worst:.3g}"
    return worst


def to_dev(a: np.ndarray, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to("cuda:0")


def scales_dev(scale_e8m0: np.ndarray):
    from fp8_block_scaled_fp8blk_gb300 import ops
    return to_dev(ops.fp8blk_scales_from_e8m0(scale_e8m0))
