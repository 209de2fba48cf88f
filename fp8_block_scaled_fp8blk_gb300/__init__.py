"""GB300-native FP8 block-scaled decode GEMV, fused greedy argmax and NVFP4
routed-expert dequant + GEMV.

The compute lives in ``libfp8blk.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/fp8blk.h``).  ``fp8_block_scaled_fp8blk_gb300.ops``
is the thin ctypes binding; importing any of its names loads the library and
raises if it has not been built.  ``synth`` (seeded inputs) imports without it.
"""
_BINDING_NAMES = (
    "fp8blk_gemv", "fp8blk_gemv_argmax", "fp8blk_gemv_argmax_ws_bytes", "fp8blk_bf16_gemv",
    "nvfp4_expert_dequant", "nvfp4_expert_dequant_gemv", "nvfp4_expert_gemv", "mxfp4_expert_gemv",
    "fp8blk_scales_from_e8m0",
    "fp8blk_device_status", "Fp8BlkError", "library_path", "argmax_workspace",
    "set_launch_tuning", "abi_version",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import ops
        return getattr(ops, name)
    raise AttributeError(name)
