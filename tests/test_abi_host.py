"""Host-side checks of the C ABI, runnable without a GPU: the library loads,
exports every entry point the header declares, and refuses bad arguments on
the host before touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8blk.h")


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_fp8blk_gb300 import build
    build.build()
    from fp8_block_scaled_fp8blk_gb300 import ops as o
    return o


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^(?:const\s+)?\w+[\s*]+(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary_calls():
    names = set(declared_functions())
    for n in ("fp8blk_gemv", "fp8blk_gemv_argmax", "fp8blk_gemv_argmax_ws_bytes",
              "nvfp4_expert_dequant_gemv", "nvfp4_expert_dequant", "nvfp4_expert_gemv", "mxfp4_expert_gemv",
              "fp8blk_scales_from_e8m0",
              "fp8blk_strerror", "fp8blk_bf16_gemv", "fp8blk_device_status"):
        assert n in names, n


def test_library_exports_every_declared_symbol(ops):
    lib = ops.raw_library()
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in fp8blk.h but not exported"


def test_strerror_and_version(ops):
    lib = ops.raw_library()
    assert ops.abi_version() == 1
    for code in range(0, 8):
        assert lib.fp8blk_strerror(code)


def test_scales_from_e8m0_matches_oracle_and_refuses_ff(ops):
    codes = np.arange(255, dtype=np.uint8)
    got = ops.fp8blk_scales_from_e8m0(codes)
    for c in range(255):
        assert float(got[c]) == oracle.e8m0_value(c)
    bad = np.array([[127, 3], [0xFF, 1]], dtype=np.uint8)
    with pytest.raises(ops.Fp8BlkError) as ei:
        ops.fp8blk_scales_from_e8m0(bad)
    assert ei.value.code == ops.ESCALE and "flat index 2" in str(ei.value)


A16 = 0x10000  # fake, never-dereferenced device addresses with known alignment
A4 = 0x10004
A1 = 0x10001


def test_gemv_host_validation(ops):
    lib = ops.raw_library()
    ok = dict(w=A16, s=A16, x=A16, y=A16, m=1, rows=128, cols=256)

    def call(**kw):
        a = {**ok, **kw}
        return lib.fp8blk_gemv(a["w"], a["s"], a["x"], a["y"], a["m"], a["rows"], a["cols"], None)

    assert call(w=None) == ops.EINVAL
    assert call(y=None) == ops.EINVAL
    assert call(m=0) == ops.EINVAL
    assert call(m=9) == ops.EINVAL
    assert call(rows=0) == ops.EINVAL
    assert call(cols=8) == ops.EINVAL
    assert call(cols=264) == ops.EINVAL  # not a multiple of 16
    assert call(rows=1 << 31) == ops.ERANGE
    assert call(w=A4) == ops.EALIGN
    assert call(x=A4) == ops.EALIGN
    assert call(s=A1) == ops.EALIGN
    assert call(y=A1) == ops.EALIGN


def test_argmax_host_validation_and_ws_size(ops):
    lib = ops.raw_library()
    need = ops.fp8blk_gemv_argmax_ws_bytes(1, 131072, 4096)
    assert need > 0 and need % 16 == 0
    # multi-panel shapes need an accumulation buffer in the workspace
    assert ops.fp8blk_gemv_argmax_ws_bytes(2, 1000, 8192) >= ops.fp8blk_gemv_argmax_ws_bytes(2, 1000, 4096) + 2 * 1000 * 4
    assert ops.fp8blk_gemv_argmax_ws_bytes(0, 10, 16) == 0
    assert ops.fp8blk_gemv_argmax_ws_bytes(1, 10, 17) == 0

    def call(ws=A16, ws_bytes=need, tokens=A16, logits=None):
        return lib.fp8blk_gemv_argmax(A16, A16, A16, logits, tokens, ws, ws_bytes, 1, 131072, 4096, None)

    assert call(tokens=None) == ops.EINVAL
    assert call(ws=None) == ops.EWS
    assert call(ws_bytes=need - 16) == ops.EWS
    assert call(ws=A4) == ops.EALIGN
    assert call(tokens=A1) == ops.EALIGN
    assert call(logits=A1) == ops.EALIGN


def test_nvfp4_host_validation(ops):
    lib = ops.raw_library()
    g = np.array([2.0 ** -4, 0.3, 2.0 ** -4, np.inf], dtype=np.float32)
    ids = np.array([0, 2], dtype=np.int32)

    def deq(eid=0, rows=16, cols=64, codes=A16, scales=A16, out=A16, n=4):
        return lib.nvfp4_expert_dequant(codes, scales, g.ctypes.data, n, eid, out, rows, cols, None)

    assert deq(eid=4) == ops.EINVAL
    assert deq(eid=-1) == ops.EINVAL
    assert deq(cols=48) == ops.EINVAL
    assert deq(codes=A4) == ops.EALIGN
    assert deq(scales=A1) == ops.EALIGN
    assert deq(out=A4) == ops.EALIGN
    assert deq(eid=1) == ops.ESCALE   # 0.3 is not a power of two
    assert deq(eid=3) == ops.ESCALE   # inf

    def full(ids_arr, x=A16, y=A16, scratch=A16):
        i = np.ascontiguousarray(ids_arr, dtype=np.int32)
        return lib.nvfp4_expert_dequant_gemv(A16, A16, g.ctypes.data, 4, i.ctypes.data, i.size,
                                             x, y, scratch, 16, 64, None)

    assert full([0, 0]) == ops.EINVAL
    assert full([0, 4]) == ops.EINVAL
    assert full([0, 1]) == ops.ESCALE
    assert full(ids, x=A4) == ops.EALIGN
    assert full(ids, scratch=A4) == ops.EALIGN


def test_nvfp4_fused_host_validation(ops):
    """The one-launch expert GEMV checks everything it can on the host (ids and
    global scales live on the device and are checked by the kernel)."""
    lib = ops.raw_library()

    def call(codes=A16, scales=A16, g=A4, n=4, ids=A4, k=2, x=A16, y=A4, rows=16, cols=512):
        return lib.nvfp4_expert_gemv(codes, scales, g, n, ids, k, x, y, rows, cols, None)

    assert call(cols=480) == ops.EINVAL      # not a multiple of 256
    assert call(cols=128) == ops.EINVAL
    assert call(k=0) == ops.EINVAL
    assert call(k=65537) == ops.EINVAL
    assert call(n=0) == ops.EINVAL
    assert call(rows=0) == ops.EINVAL
    assert call(ids=None) == ops.EINVAL
    assert call(g=None) == ops.EINVAL
    assert call(scales=A4) == ops.EALIGN     # scale rows are bulk-copied: 16-byte aligned
    assert call(codes=A4) == ops.EALIGN
    assert call(x=A4) == ops.EALIGN
    assert call(ids=A1) == ops.EALIGN
    assert call(rows=1 << 40) == ops.ERANGE


def test_mxfp4_host_validation(ops):
    lib = ops.raw_library()

    def call(codes=A16, scales=A16, n=4, ids=A4, k=2, x=A16, y=A4, rows=16, cols=1024):
        return lib.mxfp4_expert_gemv(codes, scales, n, ids, k, x, y, rows, cols, None)

    assert call(cols=768) == ops.EINVAL      # not a multiple of 512
    assert call(cols=256) == ops.EINVAL
    assert call(k=0) == ops.EINVAL
    assert call(n=0) == ops.EINVAL
    assert call(ids=None) == ops.EINVAL
    assert call(scales=A4) == ops.EALIGN
    assert call(x=A4) == ops.EALIGN
    assert call(ids=A1) == ops.EALIGN
    assert call(rows=1 << 40) == ops.ERANGE


def test_tuning_validation(ops):
    lib = ops.raw_library()
    assert lib.fp8blk_set_launch_tuning(0, 5, 1, 1, 0) == ops.EINVAL
    assert lib.fp8blk_set_launch_tuning(0, 0, 1, 1, 1) == ops.EINVAL
    assert lib.fp8blk_set_launch_tuning(0, 0, 1, 1, 0) == ops.OK
    lib.fp8blk_set_wait_limit.argtypes = [ctypes.c_int64]
    assert lib.fp8blk_set_wait_limit(-1) == ops.EINVAL
    assert lib.fp8blk_set_wait_limit(ops.WAIT_LIMIT_DEFAULT_NS + 1) == ops.EINVAL
    assert lib.fp8blk_set_wait_limit(0) == ops.OK
    assert lib.fp8blk_set_wait_limit(ops.WAIT_LIMIT_DEFAULT_NS) == ops.OK
