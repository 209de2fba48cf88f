"""The kernels' give-up path, exercised without hanging anything.

Every wait of a CUDA-core GEMV kernel for a weight tile is bounded; when the
bound runs out the kernel lets the copies it has in flight land (with the
fixed one-second bound), sets FP8BLK_STATUS_WAIT_TIMEOUT in the device status
word and returns.  These tests shorten the consumer-side bound to zero
(fp8blk_set_wait_limit), so the first tile a warp finds not yet landed makes
it give up at once, and check that: the call returns; the status word says so
(or, if no wait found its tile missing, the outputs are exactly right); and --
with the limit restored -- the next call on the same buffers and workspace
gives the same bits as before and leaves the status clear.
"""
import numpy as np
import pytest
import torch

from _helpers import scales_dev, to_dev
from fp8_block_scaled_fp8blk_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_fp8blk_gb300 import ops as o
    o.fp8blk_device_status(clear=True)
    yield o
    o.set_wait_limit()
    o.set_m1_kernel(0, 0)
    o.set_tensor_core_min_m(0, 0)
    o.fp8blk_device_status(clear=True)


def _zero_limit_runs(ops, call, check_exact, attempts):
    """Run `call` under a zero wait limit `attempts` times.  Each run either
    reports a give-up in the status word, or (no wait found its tile missing)
    must have produced exactly the default-limit result.  Returns how many
    runs gave up."""
    gave_up = 0
    ops.set_wait_limit(0)
    try:
        for _ in range(attempts):
            call()
            status = ops.fp8blk_device_status(clear=True)
            assert status & ~ops.STATUS_WAIT_TIMEOUT == 0
            if status & ops.STATUS_WAIT_TIMEOUT:
                gave_up += 1
            else:
                check_exact()
    finally:
        ops.set_wait_limit()
    return gave_up


# The team kernel's consumers outpace its copies at these sizes, so a zero
# limit must make some wait give up; the row-per-warp kernel's consumers are
# slower than its copies, so there a give-up is possible but not certain.
@pytest.mark.parametrize("kernel,m,rows,cols,must_give_up", [("team", 2, 16384, 4096, True),
                                                             ("team", 1, 8192, 8192, True),
                                                             ("rowwarp", 1, 16384, 4096, False)])
def test_gemv_argmax_gives_up_then_recovers(ops, kernel, m, rows, cols, must_give_up):
    ops.set_m1_kernel(1 if kernel == "rowwarp" else 2, 0)
    ops.set_tensor_core_min_m(9, 0)  # the CUDA-core kernels take the configurable limit
    try:
        assert ops.plan_query(m, rows, cols)["kernel"] == (1 if kernel == "rowwarp" else 0)
        c = synth.fp8blk_case(rows, cols, m, seed=77)
        w, s, x = to_dev(c.codes), scales_dev(c.scale_e8m0), to_dev(c.x)
        ws = ops.argmax_workspace(m, rows, cols, "cuda:0")
        logits = torch.empty((m, rows), dtype=torch.float32, device="cuda:0")

        def call():
            return ops.fp8blk_gemv_argmax(w, s, x, ws, logits=logits)

        ref_tok = call().cpu().numpy().copy()
        ref_logits = logits.cpu().numpy().copy()
        assert ops.fp8blk_device_status(clear=True) == 0

        def exact():
            assert np.array_equal(logits.cpu().numpy().view(np.uint32), ref_logits.view(np.uint32))

        gave_up = _zero_limit_runs(ops, call, exact, attempts=20 if must_give_up else 5)
        if must_give_up:
            assert gave_up > 0, "no wait ran out with a zero limit"
        tok = call().cpu().numpy()
        assert ops.fp8blk_device_status() == 0
        assert np.array_equal(tok, ref_tok)
        assert np.array_equal(logits.cpu().numpy().view(np.uint32), ref_logits.view(np.uint32))
    finally:
        ops.set_m1_kernel(0, 0)
        ops.set_tensor_core_min_m(0, 0)


def test_fp4_expert_gemv_gives_up_then_recovers(ops):
    n_experts, rows, cols, n_active = 8, 2048, 4096, 6
    c = synth.nvfp4_case(n_experts, rows, cols, n_active, seed=78)
    codes, scales, x = to_dev(c.codes), to_dev(c.scales), to_dev(c.x)
    g = to_dev(c.gscale)
    ids = to_dev(np.asarray(c.ids, dtype=np.int32))
    y = torch.empty((n_active, rows), dtype=torch.float32, device="cuda:0")

    def call():
        return ops.nvfp4_expert_gemv(codes, scales, g, ids, x, y=y)

    call()
    ref = y.cpu().numpy().copy()
    assert ops.fp8blk_device_status(clear=True) == 0

    def exact():
        assert np.array_equal(y.cpu().numpy().view(np.uint32), ref.view(np.uint32))

    _zero_limit_runs(ops, call, exact, attempts=5)
    call()
    assert ops.fp8blk_device_status() == 0
    assert np.array_equal(y.cpu().numpy().view(np.uint32), ref.view(np.uint32))
