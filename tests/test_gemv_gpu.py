"""GPU parity of fp8blk_gemv (through the C ABI) against the CPU oracle.

Bar: |gpu - oracle| <= 1e-5 * sum_c |w x| + 1e-6 per output element, plus
bit-exact invariants (one-hot reproduces decoded weights, negation, power-of-
two grid scaling, duplicated rows, determinism across runs and launch shapes).
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_close, scales_dev, to_dev
from fp8_block_scaled_fp8blk_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_fp8blk_gb300 import ops as o
    yield o
    o.set_launch_tuning()
    assert o.fp8blk_device_status(clear=True) == 0


def run_gemv(ops, case):
    w = to_dev(case.codes)
    s = scales_dev(case.scale_e8m0)
    x = to_dev(case.x)
    y = ops.fp8blk_gemv(w, s, x)
    torch.cuda.synchronize()
    return y.cpu().numpy()


# Shapes spanning several tiles and ragged tails: rows not a multiple of the
# stage or of 128, columns not a multiple of 128, one-warp teams, multi-panel
# rows (cols > 4096), every m.
RAGGED = [(1, 1, 16), (1, 130, 272), (2, 257, 400), (3, 1000, 1040), (4, 129, 4096),
          (5, 77, 4112), (6, 300, 16), (7, 515, 2064), (8, 257, 8208), (8, 640, 4096),
          (1, 4097, 8192), (2, 96, 12304), (3, 2, 48), (8, 1, 16)]


@pytest.mark.parametrize("m,rows,cols", RAGGED)
def test_gemv_matches_oracle_ragged(ops, m, rows, cols):
    case = synth.fp8blk_case(rows, cols, m, seed=1000 + rows + cols + m)
    y = run_gemv(ops, case)
    ref, a = oracle.fp8blk_gemv(case.codes, case.scale_e8m0, case.x, nthreads=8)
    assert_close(y, ref, a, f"m={m} {rows}x{cols}")


@pytest.mark.parametrize("name", ["gemv_512x1024_m1", "gemv_4096x4096_m1"])
def test_gemv_named_workloads_full(ops, name):
    case = synth.workload_case(name)
    y = run_gemv(ops, case)
    ref, a = oracle.fp8blk_gemv(case.codes, case.scale_e8m0, case.x, nthreads=16)
    assert_close(y, ref, a, name)


def test_gemv_verify_m8_full_size(ops):
    case = synth.workload_case("verify_16384x4096_m8")
    y = run_gemv(ops, case)
    ref, a = oracle.fp8blk_gemv(case.codes, case.scale_e8m0, case.x, nthreads=16)
    assert_close(y, ref, a, "verify_16384x4096_m8")


def test_gemv_one_hot_is_exact(ops):
    rows, cols = 260, 1040
    rng = np.random.default_rng(5)
    codes = synth.finite_e4m3_codes(rng, (rows, cols))
    scale = synth.e8m0_codes(rng, ((rows + 127) // 128, (cols + 127) // 128), -20, 20)
    w, s = to_dev(codes), scales_dev(scale)
    for c0 in (0, 7, 128, 255, 1032):
        cs = list(range(c0, c0 + 8))
        x = np.zeros((8, cols), dtype=np.float32)
        for i, c in enumerate(cs):
            x[i, c] = 1.0
        y = ops.fp8blk_gemv(w, s, to_dev(x)).cpu().numpy()
        e = np.eye(cols, dtype=np.float32)[cs]
        ref, _ = oracle.fp8blk_gemv(codes, scale, e)
        assert np.array_equal(y.astype(np.float64), ref), c0


def test_gemv_invariants_bit_exact(ops):
    rows, cols, m = 384, 2064, 3
    case = synth.fp8blk_case(rows, cols, m, seed=77)
    w, s, x = to_dev(case.codes), scales_dev(case.scale_e8m0), to_dev(case.x)
    y = ops.fp8blk_gemv(w, s, x)
    y_neg = ops.fp8blk_gemv(w, s, -x)
    assert torch.equal(y_neg, -y)
    s8 = scales_dev(case.scale_e8m0 + np.uint8(3))
    assert torch.equal(ops.fp8blk_gemv(w, s8, x), y * 8.0)
    # determinism: same call twice, and under other launch shapes
    assert torch.equal(ops.fp8blk_gemv(w, s, x), y)
    for tune in (dict(target_stage_bytes=8192), dict(ctas_per_sm=1, use_pdl=0),
                 dict(max_stages=2, l2_prefetch=0), dict(target_stage_bytes=131072, ctas_per_sm=1)):
        ops.set_launch_tuning(**tune)
        assert torch.equal(ops.fp8blk_gemv(w, s, x), y), tune
    ops.set_launch_tuning()


def test_gemv_duplicated_rows_identical(ops):
    rows, cols = 512, 4096
    case = synth.fp8blk_case(rows, cols, 2, seed=3)
    case.scale_e8m0[...] = 124  # one scale everywhere: rows r and r' are identical weights
    for r in (1, 9, 130, 300, 511):
        case.codes[r] = case.codes[0]
    y = run_gemv(ops, case)
    for r in (1, 9, 130, 300, 511):
        assert np.array_equal(y[:, r], y[:, 0])


def test_gemv_nan_code_only_poisons_its_row(ops):
    case = synth.fp8blk_case(64, 256, 1, seed=4)
    case.codes[5, 17] = 0x7F
    y = run_gemv(ops, case)
    assert np.isnan(y[0, 5]) and not np.isnan(np.delete(y[0], 5)).any()


def test_gemv_extreme_scales(ops):
    """e8m0 codes 0 (subnormal 2^-127) and 254 with tiny/huge x stay within tolerance."""
    rows, cols = 256, 256
    case = synth.fp8blk_case(rows, cols, 2, seed=6)
    case.scale_e8m0[...] = np.array([[0, 254], [127, 1]], dtype=np.uint8)
    case.x[0] *= 1e-30
    case.x[1] *= 1e-20
    y = run_gemv(ops, case)
    ref, a = oracle.fp8blk_gemv(case.codes, case.scale_e8m0, case.x)
    assert_close(y, ref, a, "extreme scales")


def test_gemv_writes_only_its_outputs(ops):
    """Canary: bytes around y stay untouched."""
    case = synth.fp8blk_case(300, 1040, 3, seed=8)
    w, s, x = to_dev(case.codes), scales_dev(case.scale_e8m0), to_dev(case.x)
    buf = torch.full((3 * 300 + 64,), 12345.0, device="cuda:0")
    y = buf[32:32 + 900].view(3, 300)
    ops.fp8blk_gemv(w, s, x, y=y)
    torch.cuda.synchronize()
    assert torch.all(buf[:32] == 12345.0) and torch.all(buf[932:] == 12345.0)


def test_bf16_gemv_matches_oracle(ops):
    rng = np.random.default_rng(12)
    for m, rows, cols in [(1, 2048, 4096), (3, 131, 272), (8, 70, 8208), (2, 9, 16)]:
        # bf16 patterns with exponents in [2^-17, 2^13]: products stay in f32 range
        sign = rng.integers(0, 2, size=(rows, cols), dtype=np.uint16) << 15
        expo = rng.integers(110, 141, size=(rows, cols), dtype=np.uint16) << 7
        b = sign | expo | rng.integers(0, 128, size=(rows, cols), dtype=np.uint16)
        x = rng.standard_normal((m, cols)).astype(np.float32)
        y = ops.fp8blk_bf16_gemv(to_dev(b.view(np.int16)), to_dev(x)).cpu().numpy()
        ref, a = oracle.bf16_gemv(b, x, nthreads=8)
        assert_close(y, ref, a, f"bf16 m={m} {rows}x{cols}")


def test_device_status_clean(ops):
    assert ops.fp8blk_device_status() == 0


@pytest.mark.parametrize("choice", [1, 2])
def test_m1_both_kernels_match_oracle(ops, choice):
    """m = 1 is served by the row-per-warp kernel (large) or the team kernel
    (small); force each on ragged and multi-panel shapes, plain and argmax."""
    ops.set_m1_kernel(choice)
    try:
        for rows, cols in [(1, 16), (130, 272), (1000, 1040), (4097, 4096), (77, 8208), (300, 12304)]:
            case = synth.fp8blk_case(rows, cols, 1, seed=rows * 7 + cols + choice)
            y = run_gemv(ops, case)
            ref, a = oracle.fp8blk_gemv(case.codes, case.scale_e8m0, case.x, nthreads=8)
            assert_close(y, ref, a, f"m1 kernel {choice} {rows}x{cols}")
            w, s, x = to_dev(case.codes), scales_dev(case.scale_e8m0), to_dev(case.x)
            ws = ops.argmax_workspace(1, rows, cols, "cuda:0")
            logits = torch.empty((1, rows), dtype=torch.float32, device="cuda:0")
            tok = ops.fp8blk_gemv_argmax(w, s, x, ws, logits=logits).cpu().numpy().view(np.uint32)
            lg = logits.cpu().numpy()
            assert_close(lg, ref, a, f"m1 argmax logits {choice} {rows}x{cols}")
            assert tok[0] == oracle.argmax(lg[0].astype(np.float64))
        rng = np.random.default_rng(40 + choice)
        for rows, cols in [(2048, 4096), (131, 272), (70, 8208)]:
            sign = rng.integers(0, 2, size=(rows, cols), dtype=np.uint16) << 15
            expo = rng.integers(110, 141, size=(rows, cols), dtype=np.uint16) << 7
            b = sign | expo | rng.integers(0, 128, size=(rows, cols), dtype=np.uint16)
            x = rng.standard_normal((1, cols)).astype(np.float32)
            yb = ops.fp8blk_bf16_gemv(to_dev(b.view(np.int16)), to_dev(x)).cpu().numpy()
            ref, a = oracle.bf16_gemv(b, x, nthreads=8)
            assert_close(yb, ref, a, f"m1 bf16 kernel {choice} {rows}x{cols}")
    finally:
        ops.set_m1_kernel(0)
