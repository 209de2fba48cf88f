"""GPU parity of the one-launch OCP MXFP4 routed-expert GEMV (the MTP block's
experts) against the CPU oracle, through the C ABI, on both kernels (CUDA
cores and tensor cores).

Bar: outputs within |gpu - oracle| <= 1e-5 * sum|w x| + 1e-6; one-hot x
reproduces every decoded weight exactly (e2m1 code x e8m0 scale); a 0xFF
scale poisons only its row; an out-of-range device id gives NaN and the
status bit.
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_close, to_dev
from fp8_block_scaled_fp8blk_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_fp8blk_gb300 import ops as o
    yield o
    assert o.fp8blk_device_status(clear=True) == 0


@pytest.fixture(params=[1, 2], ids=["cuda_cores", "tensor_cores"])
def fp4k(ops, request):
    ops.set_fp4_kernel(request.param)
    yield request.param
    ops.set_fp4_kernel(0)


def run(ops, case, ids=None, x=None):
    ids = case.ids if ids is None else ids
    x = case.x if x is None else x
    y = ops.mxfp4_expert_gemv(to_dev(case.codes), to_dev(case.scales), to_dev(np.asarray(ids, dtype=np.int32)),
                              to_dev(np.asarray(x, dtype=np.float32)))
    torch.cuda.synchronize()
    return y.cpu().numpy()


def test_mxfp4_full_config(ops, fp4k):
    w = synth.MXFP4_WORKLOAD
    case = synth.mxfp4_case(w["n_experts"], w["rows"], w["cols"], w["n_active"], w["seed"])
    y = run(ops, case)
    ref, a = oracle.mxfp4_expert_gemv(case.codes, case.scales, case.ids, case.x, nthreads=16)
    assert_close(y, ref, a, "mxfp4 6 of 64 2048x4096")


@pytest.mark.parametrize("n_experts,rows,cols,n_active", [(3, 1, 512, 1), (4, 7, 1024, 2), (8, 129, 4096, 3),
                                                          (5, 1000, 1536, 5), (6, 130, 4608, 4), (4, 65, 8192, 4)])
def test_mxfp4_ragged(ops, fp4k, n_experts, rows, cols, n_active):
    case = synth.mxfp4_case(n_experts, rows, cols, n_active, seed=rows * 17 + cols + n_active)
    y = run(ops, case)
    ref, a = oracle.mxfp4_expert_gemv(case.codes, case.scales, case.ids, case.x, nthreads=8)
    assert_close(y, ref, a, f"mxfp4 {n_experts}x{rows}x{cols} k={n_active}")


def test_mxfp4_one_hot_is_exact(ops, fp4k):
    """Every e2m1 code under e8m0 scales from 2^-127 to 2^127: x = e_c returns
    the decoded weight column exactly."""
    rows, cols = 8, 512
    case = synth.mxfp4_case(1, rows, cols, 1, seed=3)
    case.codes[0] = np.arange(rows * cols // 2, dtype=np.uint32).reshape(rows, cols // 2).astype(np.uint8)
    case.scales[0] = np.array([0, 1, 60, 119, 127, 128, 200, 254], dtype=np.uint8)[:, None]
    for c in (0, 1, 31, 32, 255, 300, 511):
        x = np.zeros(cols, dtype=np.float32)
        x[c] = 1.0
        y = run(ops, case, ids=[0], x=x)
        ref, _ = oracle.mxfp4_expert_gemv(case.codes, case.scales, np.array([0], dtype=np.int32), x)
        with np.errstate(over="ignore"):  # 6 * 2^127 is inf in f32 on both sides
            want = ref[0].astype(np.float32)
        assert np.array_equal(y[0], want), c


def test_mxfp4_scale_ff_poisons_only_its_row(ops, fp4k):
    case = synth.mxfp4_case(3, 40, 1024, 2, seed=9)
    case.scales[case.ids[1], 17, 5] = 0xFF
    y = run(ops, case)
    assert np.isnan(y[1, 17]) and not np.isnan(np.delete(y[1], 17)).any() and not np.isnan(y[0]).any()


def test_mxfp4_bad_and_repeated_ids(ops, fp4k):
    case = synth.mxfp4_case(4, 100, 512, 3, seed=10)
    assert ops.fp8blk_device_status(clear=True) == 0
    y = run(ops, case, ids=[2, 7, 2])
    assert np.isnan(y[1]).all() and np.array_equal(y[0], y[2])
    assert ops.fp8blk_device_status(clear=True) == ops.STATUS_BAD_EXPERT


def test_mxfp4_x_inf_and_nan(ops, fp4k):
    """An inf in x: the CUDA-core arm gives +-inf where its weight is nonzero
    and NaN where it is zero (0 * inf), as the oracle does; the tensor-core arm
    gives NaN everywhere (its x planes cannot hold an inf, so the non-finite
    32-column block poisons every sum).  A NaN in x makes every output NaN."""
    case = synth.mxfp4_case(2, 256, 1024, 2, seed=83)
    x = case.x.copy()
    x[100] = np.inf
    x[700] = 1e30
    y = run(ops, case, x=x)
    ref, _ = oracle.mxfp4_expert_gemv(case.codes, case.scales, case.ids, x, nthreads=8)
    assert np.isnan(ref).any() and np.isinf(ref).any() and not np.isfinite(ref).any()
    if fp4k == 1:
        assert np.array_equal(np.isnan(y), np.isnan(ref))
        assert np.array_equal(y[~np.isnan(ref)], ref[~np.isnan(ref)])
    else:
        assert np.isnan(y).all()
    x[5] = np.nan
    assert np.isnan(run(ops, case, x=x)).all()


def test_mxfp4_kernels_agree_many_active(ops):
    """32 of 64 experts active (the tensor cores' by-shape regime): the default
    gives the tensor-core kernel's bits, and both kernels meet the bound."""
    case = synth.mxfp4_case(64, 1024, 2048, 32, seed=11)
    runs = {}
    for k in (0, 1, 2):
        ops.set_fp4_kernel(k)
        runs[k] = run(ops, case)
    ops.set_fp4_kernel(0)
    assert np.array_equal(runs[0].view(np.uint32), runs[2].view(np.uint32))
    ref, a = oracle.mxfp4_expert_gemv(case.codes, case.scales, case.ids, case.x, nthreads=16)
    for k in (1, 2):
        assert_close(runs[k], ref, a, f"mxfp4 32 of 64, kernel {k}")


def test_mxfp4_x_wide_dynamic_range(ops, fp4k):
    """x spanning 2^-40 .. 2^20: the f32 block sums keep the small terms' share
    (on the tensor cores each 32-column block has its own plane exponent)."""
    case = synth.mxfp4_case(3, 256, 2048, 2, seed=89)
    rng = np.random.default_rng(90)
    x = (rng.standard_normal(2048) * np.exp2(rng.integers(-40, 21, 2048))).astype(np.float32)
    y = run(ops, case, x=x)
    ref, a = oracle.mxfp4_expert_gemv(case.codes, case.scales, case.ids, x, nthreads=8)
    assert_close(y, ref, a, "mxfp4 wide x")


def test_mxfp4_scales_across_the_e8m0_range(ops, fp4k):
    """Random codes and x under e8m0 scales drawn from 2^-127 .. 2^100 (every
    output stays finite in f32): the block factors are applied to the f32 block
    sums without overflow or loss beyond the bound."""
    case = synth.mxfp4_case(2, 384, 1536, 2, seed=91)
    rng = np.random.default_rng(92)
    case.scales[:] = rng.choice(np.array([0, 1, 2, 60, 100, 126, 127, 128, 160, 200, 227], dtype=np.uint8),
                                size=case.scales.shape)
    y = run(ops, case)
    ref, a = oracle.mxfp4_expert_gemv(case.codes, case.scales, case.ids, case.x, nthreads=8)
    assert np.isfinite(ref).all() and np.isfinite(y).all()
    assert_close(y, ref, a, "mxfp4 e8m0 range")


def test_mxfp4_bit_identical_rerun(ops, fp4k):
    """Two calls on the same inputs give the same bits (fixed reduction order)."""
    w = synth.MXFP4_WORKLOAD
    case = synth.mxfp4_case(w["n_experts"], w["rows"], w["cols"], w["n_active"], w["seed"])
    y1, y2 = run(ops, case), run(ops, case)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_mxfp4_tensor_cores_replayed_from_a_cuda_graph(ops):
    """The MXFP4 tensor-core GEMV recorded into a CUDA graph and replayed on new
    activations and new device ids gives the eager call's bits."""
    case = synth.mxfp4_case(16, 2048, 1024, 8, seed=93)
    codes, scales = to_dev(case.codes), to_dev(case.scales)
    rng = np.random.default_rng(94)
    ids_l = [np.asarray(case.ids, dtype=np.int32)] + [rng.choice(16, 8, replace=False).astype(np.int32)
                                                       for _ in range(2)]
    xs = [to_dev(case.x)] + [to_dev(rng.standard_normal(1024, dtype=np.float32)) for _ in range(2)]
    ids_buf, x_buf = to_dev(ids_l[0]).clone(), xs[0].clone()
    y = torch.empty((8, 2048), dtype=torch.float32, device="cuda:0")
    ops.set_fp4_kernel(2)
    try:
        ops.mxfp4_expert_gemv(codes, scales, ids_buf, x_buf, y=y)  # per-shape host state outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            ops.mxfp4_expert_gemv(codes, scales, ids_buf, x_buf, y=y)
        for ids, x in zip(ids_l, xs):
            ids_buf.copy_(to_dev(ids))
            x_buf.copy_(x)
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(y, ops.mxfp4_expert_gemv(codes, scales, to_dev(ids), x))
    finally:
        ops.set_fp4_kernel(0)
    assert ops.fp8blk_device_status(clear=True) == 0


def test_mxfp4_zero_block_under_large_scale_and_x(ops, fp4k):
    """A block of zero codes under the largest e8m0 scale (2^127), holding an x
    of 1e6: it adds exactly zero, so every output is finite and meets the bound
    (the scale must not meet x's magnitude before the zero block sum does)."""
    case = synth.mxfp4_case(2, 96, 512, 2, seed=95)
    case.codes[:, :, 0:16] = 0           # columns 0..31 (block 0) of every row: +0
    case.scales[:, :, 0] = 254           # 2^127
    x = case.x.copy()
    x[3] = 1e6
    y = run(ops, case, x=x)
    ref, a = oracle.mxfp4_expert_gemv(case.codes, case.scales, case.ids, x, nthreads=8)
    assert np.isfinite(ref).all() and np.isfinite(y).all()
    assert_close(y, ref, a, "mxfp4 zero block, scale 2^127, x 1e6")


def test_mxfp4_sign_and_power_of_two_invariants(ops, fp4k):
    """Bit-exact on both kernels: y(-x) = -y(x); x * 2^k gives y * 2^k; every
    e8m0 scale code + k gives y * 2^k."""
    case = synth.mxfp4_case(4, 300, 1024, 3, seed=98)
    y = run(ops, case)
    assert np.array_equal(run(ops, case, x=-case.x).view(np.uint32), (-y).view(np.uint32))
    for k in (-3, 5):
        xs = (case.x * np.float32(2.0 ** k)).astype(np.float32)
        assert np.array_equal(run(ops, case, x=xs), y * np.float32(2.0 ** k)), k
        shifted = synth.Mxfp4Case(case.codes, (case.scales.astype(np.int32) + k).astype(np.uint8), case.ids, case.x)
        assert np.array_equal(run(ops, shifted), y * np.float32(2.0 ** k)), k
