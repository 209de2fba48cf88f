"""GPU parity of the fused GEMV + greedy argmax (through the C ABI).

Bar: (i) every token equals the lowest-index argmax of the same call's f32
logits, bit for bit; (ii) it equals the oracle's token whenever the oracle's
top-2 gap exceeds twice the tolerance band; (iii) logits match the oracle
within tolerance; tie cases resolve to the lowest index.
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import REL, ABS, assert_close, scales_dev, to_dev
from fp8_block_scaled_fp8blk_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_fp8blk_gb300 import ops as o
    yield o
    assert o.fp8blk_device_status(clear=True) == 0


def call(ops, case, with_logits=True, ws=None):
    rows, cols = case.codes.shape
    m = case.x.shape[0]
    w, s, x = to_dev(case.codes), scales_dev(case.scale_e8m0), to_dev(case.x)
    if ws is None:
        ws = ops.argmax_workspace(m, rows, cols, "cuda:0")
    logits = torch.empty((m, rows), dtype=torch.float32, device="cuda:0") if with_logits else None
    tok = ops.fp8blk_gemv_argmax(w, s, x, ws, logits=logits)
    torch.cuda.synchronize()
    return tok.cpu().numpy().view(np.uint32), (logits.cpu().numpy() if with_logits else None)


def check_tokens(tok, logits, ref, a):
    m = ref.shape[0]
    for i in range(m):
        own = oracle.argmax(logits[i].astype(np.float64))
        assert tok[i] == own, f"row {i}: token {tok[i]} vs argmax of own logits {own}"
        ot = oracle.argmax(ref[i])
        srt = np.sort(ref[i])[::-1]
        band = REL * a[i].max() + ABS
        if srt.size > 1 and srt[0] - srt[1] > 2 * band:
            assert tok[i] == ot, f"row {i}: token {tok[i]} vs oracle {ot}"


@pytest.mark.parametrize("m,rows,cols", [(1, 4097, 1040), (3, 1000, 272), (8, 640, 4096),
                                         (2, 300, 8208), (1, 1, 16), (5, 129, 4112)])
def test_argmax_matches_oracle(ops, m, rows, cols):
    case = synth.fp8blk_case(rows, cols, m, seed=rows + cols + 7 * m)
    tok, logits = call(ops, case)
    ref, a = oracle.fp8blk_gemv(case.codes, case.scale_e8m0, case.x, nthreads=8)
    assert_close(logits, ref, a, "logits")
    check_tokens(tok, logits, ref, a)
    tok2, _ = call(ops, case, with_logits=False)
    assert np.array_equal(tok, tok2)


def test_argmax_ties_resolve_to_lowest_index(ops):
    rows, cols = 2048, 1024
    case = synth.fp8blk_case(rows, cols, 1, seed=21)
    case.scale_e8m0[...] = 127
    case.x[...] = np.abs(case.x) + 0.01
    # every other weight is a positive e4m3 value below 1.0 (code & 0x37), so
    # an all-1.0 row (code 0x38) has the strictly largest logit
    case.codes &= np.uint8(0x37)
    for r in (5, 6, 700, 2047):  # same block, another CTA, last row
        case.codes[r] = 0x38
    tok, logits = call(ops, case)
    assert logits[0, 5] == logits[0, 6] == logits[0, 700] == logits[0, 2047]
    assert logits[0, 5] == logits[0].max()
    assert tok[0] == 5
    case.codes[5] = 0
    case.codes[6] = 0
    tok, _ = call(ops, case)
    assert tok[0] == 700


def test_argmax_ties_at_row_zero_and_across_ctas(ops):
    rows, cols = 65536, 512
    case = synth.fp8blk_case(rows, cols, 2, seed=22)
    case.scale_e8m0[...] = 127
    case.codes[:] = 0  # every logit is 0: all tie -> token 0
    tok, logits = call(ops, case)
    assert np.all(logits == 0) and list(tok) == [0, 0]
    case.codes[rows - 1, :] = 0x38
    case.codes[40000, :] = 0x38
    case.x[...] = 1.0
    tok, _ = call(ops, case)
    assert list(tok) == [40000, 40000]


def test_argmax_workspace_reuse_across_calls(ops):
    case = synth.fp8blk_case(9000, 1024, 2, seed=23)
    ws = ops.argmax_workspace(2, 9000, 1024, "cuda:0")
    first, _ = call(ops, case, ws=ws)
    for _ in range(3):
        again, _ = call(ops, case, ws=ws)
        assert np.array_equal(first, again)
    assert int(ws[:4].view(torch.int32).item()) == 0  # arrival counter back at zero


def test_argmax_nan_rows_never_win(ops):
    case = synth.fp8blk_case(512, 256, 1, seed=24)
    case.codes[:, 0] = 0x7F  # every logit NaN ...
    tok, logits = call(ops, case)
    assert np.isnan(logits).all() and tok[0] == 0
    case.codes[300, 0] = 0x38  # ... except row 300
    tok, logits = call(ops, case)
    assert tok[0] == 300


def test_head_argmax_full_size(ops):
    """131072 x 4096 vocab head, m = 1, in the launch configuration the bench times."""
    case = synth.workload_case("head_argmax_131072x4096_m1")
    tok, logits = call(ops, case)
    tok_nl, _ = call(ops, case, with_logits=False)
    assert tok_nl[0] == tok[0]
    ref, a = oracle.fp8blk_gemv(case.codes, case.scale_e8m0, case.x, nthreads=16)
    assert_close(logits, ref, a, "head logits")
    check_tokens(tok, logits, ref, a)
    srt = np.sort(ref[0])[::-1]
    assert srt[0] - srt[1] > 2 * (REL * a[0].max() + ABS), "seeded head has a clear winner"
    assert tok[0] == oracle.argmax(ref[0])
