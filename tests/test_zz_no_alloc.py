"""fp8blk_gemv_argmax_noalloc: the fused GEMV + greedy argmax for callers that
cannot allocate device memory (code running during CUDA graph capture,
serving loops that must not call the device-synchronizing cudaMalloc, plain C
hosts without an allocator).  It keeps its workspace in a fixed array inside
the library, so these tests call it through the C ABI and check it against the
workspace-taking entry point on consecutive calls.

This file is collected last on purpose: it must pass both alone in a fresh
process and after every other test has used the library.
"""
import ctypes

import numpy as np
import pytest
import torch

from _helpers import scales_dev, to_dev
from fp8_block_scaled_fp8blk_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_fp8blk_gb300 import ops as o
    yield o
    assert o.fp8blk_device_status(clear=True) == 0


def _reference(ops, w, s, x, m, rows, cols):
    """Tokens and logits from the entry point that takes a caller workspace."""
    ws = ops.argmax_workspace(m, rows, cols, "cuda:0")
    logits = torch.empty((m, rows), dtype=torch.float32, device="cuda:0")
    tok = ops.fp8blk_gemv_argmax(w, s, x, ws, logits=logits)
    torch.cuda.synchronize()
    return tok.cpu().numpy().view(np.uint32), logits.cpu().numpy()


def _noalloc_c_abi(ops, w, s, x, m, rows, cols, with_logits):
    lib = ops.raw_library()
    tokens = torch.full((m,), -1, dtype=torch.int32, device="cuda:0")
    logits = torch.full((m, rows), np.nan, dtype=torch.float32, device="cuda:0") if with_logits else None
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.fp8blk_gemv_argmax_noalloc(
        ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(s.data_ptr()), ctypes.c_void_p(x.data_ptr()),
        ctypes.c_void_p(logits.data_ptr()) if with_logits else None,
        ctypes.c_void_p(tokens.data_ptr()), m, rows, cols, ctypes.c_void_p(stream))
    assert rc == ops.OK, ops._lib.fp8blk_strerror(rc)
    torch.cuda.synchronize()
    return tokens.cpu().numpy().view(np.uint32), (logits.cpu().numpy() if with_logits else None)


# Shapes that reach every kernel the fused argmax can run: the team kernel
# (small and ragged), the row-per-warp kernel (m = 1 from 96 MiB of weights
# when too wide for the tensor cores: 3072 x 36864), the tensor-core kernel
# (28672 and 131072 rows at m = 1, the 16384 x 4096 verify at m = 8) and the
# multi-panel accumulator (cols > 4096).
@pytest.mark.parametrize("m,rows,cols", [(1, 20000, 4096), (3, 1000, 1040), (8, 640, 4096),
                                         (1, 28672, 4096), (1, 131072, 4096), (8, 16384, 4096),
                                         (1, 64, 8192), (1, 3072, 36864)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(ops, m, rows, cols):
    cases = [synth.fp8blk_case(rows, cols, m, seed=900 + k) for k in range(2)]
    devs = [(to_dev(c.codes), scales_dev(c.scale_e8m0), to_dev(c.x)) for c in cases]
    refs = [_reference(ops, *d, m, rows, cols) for d in devs]
    # Two calls in a row, the second on different data: the shared array must
    # not carry anything over from the first.  Both entry points run the same
    # kernel on the same data in a fixed reduction order, so the logits must be
    # bit-identical (a stricter check than the oracle tolerance).
    for (w, s, x), (ref_tok, ref_logits) in zip(devs, refs):
        tok, logits = _noalloc_c_abi(ops, w, s, x, m, rows, cols, with_logits=True)
        assert np.array_equal(tok, ref_tok)
        assert np.array_equal(logits.view(np.uint32), ref_logits.view(np.uint32))
    for (w, s, x), (ref_tok, _) in zip(devs, refs):
        tok, _ = _noalloc_c_abi(ops, w, s, x, m, rows, cols, with_logits=False)
        assert np.array_equal(tok, ref_tok)


def test_noalloc_refuses_shapes_beyond_its_array(ops):
    lib = ops.raw_library()
    assert lib.fp8blk_noalloc_scratch_bytes() == 65792
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check comes first
    rc = lib.fp8blk_gemv_argmax_noalloc(fake, fake, fake, None, fake, 8, 100000, 8192, None)
    assert rc == ops.ERANGE


@pytest.mark.parametrize("m,rows,cols", [(1, 131072, 4096), (8, 16384, 4096), (3, 1000, 1040)])
def test_noalloc_inside_a_cuda_graph(ops, m, rows, cols):
    """The call this entry point exists for: recorded once into a CUDA graph
    (after one eager call on the device), then replayed with new activations
    copied into the captured input buffer; each replay's tokens and logits
    equal the workspace entry point's bit for bit."""
    lib = ops.raw_library()
    cases = [synth.fp8blk_case(rows, cols, m, seed=950 + k) for k in range(3)]
    w, s = to_dev(cases[0].codes), scales_dev(cases[0].scale_e8m0)
    xs = [to_dev(c.x) for c in cases]
    x_buf = xs[0].clone()
    tokens = torch.full((m,), -1, dtype=torch.int32, device="cuda:0")
    logits = torch.empty((m, rows), dtype=torch.float32, device="cuda:0")

    def call():
        rc = lib.fp8blk_gemv_argmax_noalloc(
            ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(s.data_ptr()), ctypes.c_void_p(x_buf.data_ptr()),
            ctypes.c_void_p(logits.data_ptr()), ctypes.c_void_p(tokens.data_ptr()), m, rows, cols,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == ops.OK

    call()  # the first call on the device precedes any capture (it looks up the array's address)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for x in xs:
        x_buf.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        ref_tok, ref_logits = _reference(ops, w, s, x, m, rows, cols)
        assert np.array_equal(tokens.cpu().numpy().view(np.uint32), ref_tok)
        assert np.array_equal(logits.cpu().numpy().view(np.uint32), ref_logits.view(np.uint32))
