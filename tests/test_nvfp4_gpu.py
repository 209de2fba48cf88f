"""GPU parity of the NVFP4 routed-expert path (through the C ABI).

Bar: every dequantised bf16 scratch byte equals the oracle's, for every active
expert; the per-expert GEMV outputs are within the GEMV tolerance.
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


@pytest.fixture(scope="module")
def c5():
    w = synth.NVFP4_WORKLOAD
    return synth.nvfp4_case(w["n_experts"], w["rows"], w["cols"], w["n_active"], w["seed"])


def test_dequant_bit_exact_every_active_expert(ops, c5):
    codes, scales = to_dev(c5.codes), to_dev(c5.scales)
    for e in c5.ids:
        got = ops.nvfp4_expert_dequant(codes, scales, c5.gscale, int(e)).cpu().numpy().view(np.uint16)
        ref, nin = oracle.nvfp4_dequant_bf16(c5.codes[e], c5.scales[e], float(c5.gscale[e]))
        assert nin == 0
        assert np.array_equal(got, ref), f"expert {e}: {np.count_nonzero(got != ref)} bytes differ"


def test_dequant_every_code_and_scale_pair(ops):
    """All 16 e2m1 codes x all normal e4m3 scales in [2^-6, 2^2] x several g."""
    s_codes = np.array([((e + 7) << 3) | mt for e in range(-6, 3) for mt in range(8)], dtype=np.uint8)
    rows, cols = s_codes.size, 32
    codes = np.zeros((1, rows, cols // 2), dtype=np.uint8)
    for j in range(16):  # nibbles 0..15 in columns 0..15, again in 16..31
        codes[0, :, j] = (2 * (j % 8)) | ((2 * (j % 8) + 1) << 4)
    scales = np.repeat(s_codes[:, None], 2, axis=1)[None]
    for g in (2.0 ** -4, 1.0, 2.0 ** -100, -(2.0 ** 100)):
        gs = np.array([g], dtype=np.float32)
        got = ops.nvfp4_expert_dequant(to_dev(codes), to_dev(scales), gs, 0).cpu().numpy().view(np.uint16)
        ref, nin = oracle.nvfp4_dequant_bf16(codes[0], scales[0], g)
        assert nin == 0 and np.array_equal(got, ref), g


def test_expert_dequant_gemv_full_config(ops, c5):
    codes, scales, x = to_dev(c5.codes), to_dev(c5.scales), to_dev(c5.x)
    rows, cols = c5.codes.shape[1], 2 * c5.codes.shape[2]
    scratch = torch.empty((rows, cols), dtype=torch.int16, device="cuda:0")
    y = ops.nvfp4_expert_dequant_gemv(codes, scales, c5.gscale, c5.ids, x, scratch).cpu().numpy()
    ref, a, last = oracle.nvfp4_expert_dequant_gemv(c5.codes, c5.scales, c5.gscale, c5.ids, c5.x,
                                                    nthreads=16, want_scratch=True)
    assert_close(y, ref, a, "nvfp4 experts")
    assert np.array_equal(scratch.cpu().numpy().view(np.uint16), last)


def test_expert_dequant_gemv_ragged(ops):
    case = synth.nvfp4_case(n_experts=7, rows=131, cols=8224, n_active=3, seed=31)
    rows, cols = 131, 8224
    scratch = torch.empty((rows, cols), dtype=torch.int16, device="cuda:0")
    y = ops.nvfp4_expert_dequant_gemv(to_dev(case.codes), to_dev(case.scales), case.gscale,
                                      case.ids, to_dev(case.x), scratch).cpu().numpy()
    ref, a, _ = oracle.nvfp4_expert_dequant_gemv(case.codes, case.scales, case.gscale, case.ids,
                                                 case.x, nthreads=8)
    assert_close(y, ref, a, "nvfp4 ragged")


# ---- one-launch expert GEMV, ids on the device: NVFP4 decoded in registers
# (CUDA cores) or the e2m1 codes fed to kind::f8f6f4 MMAs as stored, x as e4m3
# planes per 16-column block (tensor cores)

@pytest.fixture(params=[1, 2], ids=["cuda_cores", "tensor_cores"])
def fp4k(ops, request):
    ops.set_fp4_kernel(request.param)
    yield request.param
    ops.set_fp4_kernel(0)


def fused(ops, case, ids=None, gscale=None, status=0):
    """One call into a NaN-filled output; the device status word must then
    read `status` (a kernel that gave up would leave NaNs and set bit 0)."""
    ids = case.ids if ids is None else ids
    g = case.gscale if gscale is None else gscale
    y = torch.full((len(ids), case.codes.shape[1]), float("nan"), dtype=torch.float32, device="cuda:0")
    ops.nvfp4_expert_gemv(to_dev(case.codes), to_dev(case.scales), to_dev(np.asarray(g, dtype=np.float32)),
                          to_dev(np.asarray(ids, dtype=np.int32)), to_dev(case.x), y=y)
    torch.cuda.synchronize()
    got = ops.fp8blk_device_status(clear=True)
    assert got == status, f"device status {got:#x}, expected {status:#x}"
    return y.cpu().numpy()


def test_fused_expert_gemv_full_config(ops, fp4k, c5):
    y = fused(ops, c5)
    ref, a, _ = oracle.nvfp4_expert_dequant_gemv(c5.codes, c5.scales, c5.gscale, c5.ids, c5.x, nthreads=16)
    assert_close(y, ref, a, "fused nvfp4 C5")


@pytest.mark.parametrize("n_experts,rows,cols,n_active", [(3, 1, 256, 1), (4, 7, 512, 2), (8, 129, 4096, 3),
                                                          (5, 1000, 1280, 5), (6, 130, 4352, 4),
                                                          (4, 65, 8192, 4), (70, 64, 256, 70),
                                                          (64, 300, 512, 64)])
def test_fused_expert_gemv_ragged(ops, fp4k, n_experts, rows, cols, n_active):
    """Ragged rows, one and several column panels (4352 = 4096 + 256), every
    expert active, more slots than one row group each, and more (slot, slab)
    units than SMs (64 x 300 rows)."""
    case = synth.nvfp4_case(n_experts, rows, cols, n_active, seed=rows * 31 + cols + n_active)
    y = fused(ops, case)
    ref, a, _ = oracle.nvfp4_expert_dequant_gemv(case.codes, case.scales, case.gscale, case.ids, case.x, nthreads=8)
    assert_close(y, ref, a, f"fused nvfp4 {n_experts}x{rows}x{cols} k={n_active}")


def test_fused_expert_gemv_repeated_ids_and_scales(ops, fp4k):
    """Repeated ids are allowed on the device path; per-expert global scales
    other than 2^-4 (any power of two) scale the result exactly."""
    case = synth.nvfp4_case(4, 300, 1024, 3, seed=55)
    ids = np.array([2, 0, 2], dtype=np.int32)
    g = np.array([2.0 ** -4, 2.0 ** 3, 2.0 ** -30, 1.0], dtype=np.float32)
    y = fused(ops, case, ids=ids, gscale=g)
    assert np.array_equal(y[0], y[2])
    ref, a, _ = oracle.nvfp4_expert_dequant_gemv(case.codes, case.scales, g, ids[:2], case.x, nthreads=8)
    assert_close(y[:2], ref, a, "fused nvfp4 scales")


def test_fused_expert_gemv_bad_expert_is_nan_and_flagged(ops, fp4k):
    case = synth.nvfp4_case(4, 200, 512, 3, seed=56)
    assert ops.fp8blk_device_status(clear=True) == 0
    g = np.array([2.0 ** -4, 0.75, 2.0 ** -4, 2.0 ** -4], dtype=np.float32)  # expert 1: not a power of two
    y = fused(ops, case, ids=np.array([3, 9, 1], dtype=np.int32), gscale=g,  # 9: out of range
              status=ops.STATUS_BAD_EXPERT)
    assert np.isnan(y[1]).all() and np.isnan(y[2]).all()
    ref, a, _ = oracle.nvfp4_expert_dequant_gemv(case.codes, case.scales, g, np.array([3], dtype=np.int32), case.x)
    assert_close(y[:1], ref, a, "good slot next to bad ones")
    assert ops.fp8blk_device_status() == 0


def test_fused_matches_two_step_path(ops, fp4k, c5):
    """Both arms use the same bf16 weight values; their sums agree within the
    GEMV tolerance of each other."""
    codes, scales, x = to_dev(c5.codes), to_dev(c5.scales), to_dev(c5.x)
    rows, cols = c5.codes.shape[1], 2 * c5.codes.shape[2]
    scratch = torch.empty((rows, cols), dtype=torch.int16, device="cuda:0")
    y2 = ops.nvfp4_expert_dequant_gemv(codes, scales, c5.gscale, c5.ids, x, scratch).cpu().numpy()
    y1 = fused(ops, c5)
    _, a, _ = oracle.nvfp4_expert_dequant_gemv(c5.codes, c5.scales, c5.gscale, c5.ids, c5.x, nthreads=16)
    assert np.all(np.abs(y1.astype(np.float64) - y2) <= 2 * (1e-5 * a + 1e-6))


def test_fused_x_wide_dynamic_range(ops, fp4k):
    """x spanning 2^-40 .. 2^20: the f32 sums keep the small terms' share (on
    the tensor cores each 16-column block has its own plane exponent, so a
    small entry is only cut relative to its block's maximum)."""
    case = synth.nvfp4_case(3, 256, 2048, 2, seed=77)
    rng = np.random.default_rng(78)
    x = (rng.standard_normal(2048) * np.exp2(rng.integers(-40, 21, 2048))).astype(np.float32)
    case = synth.Nvfp4Case(case.codes, case.scales, case.gscale, case.ids, x)
    y = fused(ops, case)
    ref, a, _ = oracle.nvfp4_expert_dequant_gemv(case.codes, case.scales, case.gscale, case.ids, case.x, nthreads=8)
    assert_close(y, ref, a, "fused nvfp4 wide x")


def test_fused_nan_scale_poisons_only_its_row(ops, fp4k):
    """An e4m3 NaN scale (0x7F) makes its 16 weights NaN: that row's output is
    NaN, every other row is untouched."""
    case = synth.nvfp4_case(2, 300, 1024, 2, seed=79)
    scales = case.scales.copy()
    e = int(case.ids[1])
    scales[e, 133, 5] = 0x7F
    case = synth.Nvfp4Case(case.codes, scales, case.gscale, case.ids, case.x)
    y = fused(ops, case)
    assert np.isnan(y[1, 133]) and np.isnan(y).sum() == 1
    ok = np.ones_like(y, dtype=bool)
    ok[1, 133] = False
    ref, a, _ = oracle.nvfp4_expert_dequant_gemv(case.codes, case.scales, case.gscale, case.ids, case.x, nthreads=8)
    assert_close(y[ok], ref[ok], a[ok], "rows next to the NaN scale")


def test_fused_zero_block_under_large_scale_and_x(ops, fp4k):
    """A block of zero codes under the largest e4m3 scale (448), holding an x
    of 3e38: it adds exactly zero, so every output is finite and meets the
    bound (the scale must not meet x's magnitude before the zero block sum
    does)."""
    case = synth.nvfp4_case(2, 96, 512, 2, seed=96)
    codes, scales = case.codes.copy(), case.scales.copy()
    codes[:, :, 0:8] = 0                 # columns 0..15 (block 0) of every row: +0
    scales[:, :, 0] = 0x7E               # 448
    x = case.x.copy()
    x[3] = 3e38
    cx = synth.Nvfp4Case(codes, scales, case.gscale, case.ids, x)
    y = fused(ops, cx)
    ref, a, _ = oracle.nvfp4_expert_dequant_gemv(cx.codes, cx.scales, cx.gscale, cx.ids, cx.x, nthreads=8)
    assert np.isfinite(ref).all() and np.isfinite(y).all()
    assert_close(y, ref, a, "nvfp4 zero block, scale 448, x 3e38")


def test_fused_bit_identical_rerun(ops, fp4k, c5):
    """Two calls on the same inputs give the same bits (fixed reduction order)."""
    y1, y2 = fused(ops, c5), fused(ops, c5)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_fused_x_inf_and_nan(ops, fp4k):
    """An inf in x (next to a large finite element): the CUDA-core arm gives
    +-inf where its weight is nonzero and NaN where it is zero (0 * inf), as
    the oracle does; the tensor-core arm gives NaN everywhere (every exact sum
    is non-finite).  A NaN in x makes every output NaN on both."""
    case = synth.nvfp4_case(2, 256, 1024, 2, seed=81)
    x = case.x.copy()
    x[100] = np.inf
    x[700] = 1e30
    cx = synth.Nvfp4Case(case.codes, case.scales, case.gscale, case.ids, x)
    y = fused(ops, cx)
    ref, _, _ = oracle.nvfp4_expert_dequant_gemv(cx.codes, cx.scales, cx.gscale, cx.ids, cx.x, nthreads=8)
    assert np.isnan(ref).any() and np.isinf(ref).any() and not np.isfinite(ref).any()
    if fp4k == 1:
        assert np.array_equal(np.isnan(y), np.isnan(ref))
        assert np.array_equal(y[~np.isnan(ref)], ref[~np.isnan(ref)])
    else:  # e4m3 planes hold no inf: the non-finite block poisons every sum
        assert np.isnan(y).all()
    x[5] = np.nan
    y = fused(ops, synth.Nvfp4Case(case.codes, case.scales, case.gscale, case.ids, x))
    assert np.isnan(y).all()


def test_fused_kernels_agree(ops, c5):
    """Both arms within the GEMV tolerance of each other on the full workload."""
    runs = {}
    for k in (1, 2):
        ops.set_fp4_kernel(k)
        runs[k] = fused(ops, c5)
    ops.set_fp4_kernel(0)
    _, a, _ = oracle.nvfp4_expert_dequant_gemv(c5.codes, c5.scales, c5.gscale, c5.ids, c5.x, nthreads=16)
    assert np.all(np.abs(runs[1].astype(np.float64) - runs[2]) <= 2 * (1e-5 * a + 1e-6))


def test_fused_default_routes_by_shape(ops):
    """The by-shape default gives the CUDA-core kernel's bits below 12288
    active rows and the tensor-core kernel's bits from there on."""
    small = synth.nvfp4_case(8, 256, 1024, 2, seed=83)          # 512 active rows
    large = synth.nvfp4_case(16, 2048, 512, 16, seed=84)        # 32768 active rows
    for case, arm in ((small, 1), (large, 2)):
        ops.set_fp4_kernel(0)
        y0 = fused(ops, case)
        ops.set_fp4_kernel(arm)
        y1 = fused(ops, case)
        ops.set_fp4_kernel(0)
        assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32)), f"default is not arm {arm}"
    ref, a, _ = oracle.nvfp4_expert_dequant_gemv(large.codes, large.scales, large.gscale, large.ids, large.x,
                                                 nthreads=16)
    assert_close(y0, ref, a, "fused nvfp4 16 x 2048 x 512, tensor cores")


def test_fused_tensor_cores_replayed_from_a_cuda_graph(ops):
    """The tensor-core expert GEMV recorded into a CUDA graph and replayed on
    new activations and new device ids gives the eager call's bits."""
    case = synth.nvfp4_case(16, 2048, 1024, 8, seed=85)
    codes, scales, g = to_dev(case.codes), to_dev(case.scales), to_dev(np.asarray(case.gscale, dtype=np.float32))
    rng = np.random.default_rng(86)
    ids_l = [np.asarray(case.ids, dtype=np.int32)] + [rng.choice(16, 8, replace=False).astype(np.int32)
                                                       for _ in range(2)]
    xs = [to_dev(case.x)] + [to_dev(rng.standard_normal(1024, dtype=np.float32)) for _ in range(2)]
    ids_buf, x_buf = to_dev(ids_l[0]).clone(), xs[0].clone()
    y = torch.empty((8, 2048), dtype=torch.float32, device="cuda:0")
    ops.set_fp4_kernel(2)
    try:
        ops.nvfp4_expert_gemv(codes, scales, g, ids_buf, x_buf, y=y)  # per-shape host state outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            ops.nvfp4_expert_gemv(codes, scales, g, ids_buf, x_buf, y=y)
        for ids, x in zip(ids_l, xs):
            ids_buf.copy_(to_dev(ids))
            x_buf.copy_(x)
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(y, ops.nvfp4_expert_gemv(codes, scales, g, to_dev(ids), x))
    finally:
        ops.set_fp4_kernel(0)
    assert ops.fp8blk_device_status(clear=True) == 0


def test_tensor_core_kernels_back_to_back(ops):
    """The NVFP4 and e4m3 tensor-core kernels (each holding all of an SM's
    tensor memory) queued back to back on one stream, with programmatic
    dependent launch, give the bits of the same calls made one at a time."""
    c4 = synth.nvfp4_case(8, 1024, 2048, 8, seed=87)
    f = synth.fp8blk_case(16384, 4096, 8, seed=88)
    codes, scales, g, ids, x4 = (to_dev(c4.codes), to_dev(c4.scales),
                                 to_dev(np.asarray(c4.gscale, dtype=np.float32)),
                                 to_dev(np.asarray(c4.ids, dtype=np.int32)), to_dev(c4.x))
    w, s, x8 = to_dev(f.codes), to_dev(ops.fp8blk_scales_from_e8m0(f.scale_e8m0)), to_dev(f.x)
    ops.set_fp4_kernel(2)
    try:
        ref4 = ops.nvfp4_expert_gemv(codes, scales, g, ids, x4)
        torch.cuda.synchronize()
        ref8 = ops.fp8blk_gemv(w, s, x8)
        torch.cuda.synchronize()
        outs = []
        for _ in range(3):
            outs.append(ops.nvfp4_expert_gemv(codes, scales, g, ids, x4))
            outs.append(ops.fp8blk_gemv(w, s, x8))
        torch.cuda.synchronize()
        for k, o in enumerate(outs):
            assert torch.equal(o, ref4 if k % 2 == 0 else ref8), k
    finally:
        ops.set_fp4_kernel(0)
    assert ops.fp8blk_device_status(clear=True) == 0


def test_fused_sign_and_power_of_two_invariants(ops, fp4k):
    """Bit-exact on both kernels: y(-x) = -y(x); x * 2^k gives y * 2^k; a
    global scale times 2^k gives y * 2^k (every product and sum scales
    exactly, so the rounding is the same)."""
    case = synth.nvfp4_case(4, 300, 1024, 3, seed=97)
    y = fused(ops, case)
    neg = fused(ops, synth.Nvfp4Case(case.codes, case.scales, case.gscale, case.ids, -case.x))
    assert np.array_equal(neg.view(np.uint32), (-y).view(np.uint32))
    for k in (-3, 5):
        xs = (case.x * np.float32(2.0 ** k)).astype(np.float32)
        yx = fused(ops, synth.Nvfp4Case(case.codes, case.scales, case.gscale, case.ids, xs))
        assert np.array_equal(yx, y * np.float32(2.0 ** k)), k
        gs = (np.asarray(case.gscale, dtype=np.float32) * np.float32(2.0 ** k)).astype(np.float32)
        yg = fused(ops, case, gscale=gs)
        assert np.array_equal(yg, y * np.float32(2.0 ** k)), k
