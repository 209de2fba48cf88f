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
