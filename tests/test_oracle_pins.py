"""Pins for the CPU oracle: each check compares the oracle with something that
does not come from the oracle itself (torch's own float8/bf16 decoders and
conversions, the OCP format tables, math.ldexp, numpy float64 matmul, brute
force), chosen so that a plausible slip (a dropped term, a wrong bias, a
transposed operand, a swapped nibble, a wrong tie rule) fails at least one.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_fp8blk_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FINITE_E4M3 = [c for c in range(256) if c not in (0x7F, 0xFF)]


def _parse_value(tok: str) -> float:
    return float(tok)  # handles 'nan', 'inf', '-0'


def _golden_format_values():
    out = {"e4m3": {}, "e2m1": {}}
    with open(os.path.join(GOLDEN, "ocp_fp8_fp4_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt, code, val = line.split()
            out[fmt][int(code, 16)] = _parse_value(val)
    return out


def _same(a: float, b: float) -> bool:
    """Equal including the sign of zero; NaN equals NaN."""
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


def torch_e4m3_table() -> np.ndarray:
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def torch_e8m0_table() -> np.ndarray:
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()


# ------------------------------------------------------------------ checks
def e4m3_table_ok(t: np.ndarray) -> bool:
    ref = torch_e4m3_table()
    gold = _golden_format_values()["e4m3"]
    if not all(_same(float(t[c]), float(ref[c])) for c in range(256)):
        return False
    return all(_same(float(t[c]), v) for c, v in gold.items())


def e2m1_table_ok(t: np.ndarray) -> bool:
    gold = _golden_format_values()["e2m1"]
    return len(gold) == 16 and all(_same(float(t[c]), gold[c]) for c in range(16))


def e8m0_decoder_ok(dec) -> bool:
    ref = torch_e8m0_table()
    for c in range(255):
        v = dec(c)
        if v != math.ldexp(1.0, c - 127) or v != ref[c]:
            return False
    return True


# ------------------------------------------------------------------ e4m3
def test_e4m3_every_code_matches_torch_and_ocp_table():
    assert e4m3_table_ok(oracle.e4m3_table())


def test_e4m3_scalar_and_table_agree():
    t = oracle.e4m3_table()
    assert all(_same(oracle.e4m3_value(c), float(t[c])) for c in range(256))


def test_e4m3_structure():
    t = oracle.e4m3_table()
    pos = t[0x00:0x7F]
    assert np.all(np.diff(pos) > 0), "finite positive codes must be strictly increasing"
    for c in FINITE_E4M3:
        if c < 0x80:
            assert _same(float(t[c | 0x80]), -float(t[c]))
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.isfinite(t[FINITE_E4M3]).all()


def test_e4m3_teeth_wrong_bias_and_missing_subnormals_fail():
    good = oracle.e4m3_table()
    wrong_bias = good * 2.0  # bias 6 instead of 7
    assert not e4m3_table_ok(wrong_bias)
    no_sub = good.copy()
    no_sub[[0x01, 0x07, 0x81]] = 0.0  # flush subnormals
    assert not e4m3_table_ok(no_sub)


# ------------------------------------------------------------------ e2m1
def test_e2m1_every_code_matches_ocp_table():
    t = oracle.e2m1_table()
    assert e2m1_table_ok(t)
    assert all(_same(oracle.e2m1_value(c), float(t[c])) for c in range(16))


def test_e2m1_teeth_swapped_mantissa_fails():
    t = oracle.e2m1_table()
    bad = t.copy()
    bad[[0x2, 0x3]] = bad[[0x3, 0x2]]
    assert not e2m1_table_ok(bad)


# ------------------------------------------------------------------ e8m0
def test_e8m0_every_code_matches_ldexp_and_torch():
    assert e8m0_decoder_ok(oracle.e8m0_value)


def test_e8m0_ff_is_refused():
    with pytest.raises(oracle.OracleError):
        oracle.e8m0_value(0xFF)


def test_e8m0_teeth_bias_128_fails():
    assert not e8m0_decoder_ok(lambda c: math.ldexp(1.0, c - 128))


# ------------------------------------------------------------------ bf16
def test_bf16_value_is_top_half_of_f32():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    for b, r in zip(bits, ref):
        assert _same(oracle.bf16_value(int(b)), float(r))


def test_bf16_rne_matches_torch_float_to_bfloat16():
    rng = np.random.default_rng(11)
    with np.errstate(over="ignore"):
        big = (rng.standard_normal(1000) * 3e38).astype(np.float32)  # near and past overflow
    vals = [
        rng.standard_normal(3000).astype(np.float32),
        (rng.standard_normal(1000) * 1e-39).astype(np.float32),     # f32/bf16 subnormals
        big,
        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 2 ** -133, 2 ** -134,
                  3 * 2 ** -134, 3.3895313892515355e38, 3.3961776e38, 0.0, -0.0],
                 dtype=np.float32),                                   # ties, tiny, overflow
    ]
    v = np.concatenate(vals)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for x, r in zip(v, ref):
        bits, inexact = oracle.bf16_rne(float(x))
        assert bits == int(r), (float(x), hex(bits), hex(int(r)))
        back = oracle.bf16_value(bits)
        assert inexact == (not _same(back, float(x)))


# ------------------------------------------------------------------ GEMV
def _decode_with_torch(codes: np.ndarray, scale_e8m0: np.ndarray) -> np.ndarray:
    """Dense float64 weights via torch's float8 view and math.ldexp scales."""
    rows, cols = codes.shape
    w = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    s = np.vectorize(lambda c: math.ldexp(1.0, int(c) - 127))(scale_e8m0).astype(np.float64)
    s_full = np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)[:rows, :cols]
    return w * s_full


GEMV_SHAPES = [(1, 16, 1), (130, 272, 3), (257, 400, 8), (128, 128, 2), (300, 1040, 5),
               (64, 2048, 1)]


@pytest.mark.parametrize("rows,cols,m", GEMV_SHAPES)
def test_gemv_matches_numpy_float64_matmul(rows, cols, m):
    case = synth.fp8blk_case(rows, cols, m, seed=rows * 31 + cols)
    # widen the scale range so every grid cell differs and misindexing shows
    rng = np.random.default_rng(rows + cols)
    case.scale_e8m0[...] = synth.e8m0_codes(rng, case.scale_e8m0.shape, -20, 20)
    y, a = oracle.fp8blk_gemv(case.codes, case.scale_e8m0, case.x)
    w = _decode_with_torch(case.codes, case.scale_e8m0)
    x = case.x.astype(np.float64)
    ref = x @ w.T
    ref_abs = np.abs(x) @ np.abs(w).T
    assert y.shape == (m, rows)
    np.testing.assert_allclose(a, ref_abs, rtol=1e-12, atol=0)
    assert np.all(np.abs(y - ref) <= 1e-12 * ref_abs + 1e-300)


def test_gemv_thread_count_does_not_change_results():
    case = synth.fp8blk_case(300, 1040, 3, seed=5)
    y1, a1 = oracle.fp8blk_gemv(case.codes, case.scale_e8m0, case.x, nthreads=1)
    y4, a4 = oracle.fp8blk_gemv(case.codes, case.scale_e8m0, case.x, nthreads=4)
    assert np.array_equal(y1, y4) and np.array_equal(a1, a4)


@pytest.mark.parametrize("rows,cols", [(1, 16), (16, 128), (130, 272), (129, 256)])
def test_gemv_one_hot_reproduces_each_decoded_weight(rows, cols):
    rng = np.random.default_rng(rows ^ cols)
    codes = synth.finite_e4m3_codes(rng, (rows, cols))
    scale = synth.e8m0_codes(rng, ((rows + 127) // 128, (cols + 127) // 128), -10, 10)
    w = _decode_with_torch(codes, scale)
    for c0 in range(0, cols, 8):
        cs = list(range(c0, min(c0 + 8, cols)))
        x = np.zeros((len(cs), cols), dtype=np.float32)
        for i, c in enumerate(cs):
            x[i, c] = 1.0
        y, _ = oracle.fp8blk_gemv(codes, scale, x)
        for i, c in enumerate(cs):
            assert np.array_equal(y[i], w[:, c])  # == treats -0 and +0 as equal


def test_gemv_refuses_e8m0_ff():
    case = synth.fp8blk_case(130, 272, 1, seed=3)
    case.scale_e8m0[1, 2] = 0xFF
    with pytest.raises(oracle.OracleError):
        oracle.fp8blk_gemv(case.codes, case.scale_e8m0, case.x)


def test_gemv_negating_x_negates_y_and_pow2_grid_scales_y():
    case = synth.fp8blk_case(257, 400, 2, seed=9)
    y, _ = oracle.fp8blk_gemv(case.codes, case.scale_e8m0, case.x)
    yn, _ = oracle.fp8blk_gemv(case.codes, case.scale_e8m0, -case.x)
    assert np.array_equal(yn, -y)
    y2, _ = oracle.fp8blk_gemv(case.codes, case.scale_e8m0 + np.uint8(3), case.x)
    assert np.array_equal(y2, y * 8.0)


# ------------------------------------------------------------------ argmax
def _golden_ties():
    cases = []
    with open(os.path.join(GOLDEN, "argmax_ties.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            vals, exp = line.split(";")
            cases.append((np.array([_parse_value(t) for t in vals.split()]), int(exp)))
    return cases


def _brute_lowest_argmax(v: np.ndarray) -> int:
    finite_or_inf = [k for k in range(len(v)) if not math.isnan(v[k])]
    if not finite_or_inf:
        return 0
    top = max(v[k] for k in finite_or_inf)
    if top == -math.inf:
        return 0
    return min(k for k in finite_or_inf if v[k] == top)


def test_argmax_golden_tie_cases():
    for v, exp in _golden_ties():
        assert oracle.argmax(v) == exp, v
        assert _brute_lowest_argmax(v) == exp, v


def test_argmax_teeth_highest_index_rule_fails_fixtures():
    def highest(v):
        k = _brute_lowest_argmax(v)
        top = v[k]
        return max(i for i in range(len(v)) if v[i] == top) if not math.isnan(top) else 0

    assert any(highest(v) != exp for v, exp in _golden_ties())


def test_argmax_random_heavy_ties_match_brute_force():
    rng = np.random.default_rng(123)
    for _ in range(300):
        n = int(rng.integers(1, 200))
        v = rng.integers(-3, 4, size=n).astype(np.float64)
        v[rng.random(n) < 0.05] = np.nan
        assert oracle.argmax(v) == _brute_lowest_argmax(v)


# ------------------------------------------------------------------ NVFP4
def test_nvfp4_products_match_torch_bfloat16_and_are_exact():
    e2m1 = _golden_format_values()["e2m1"]
    s_codes = [((e + 7) << 3) | m for e in range(-6, 3) for m in range(8)]
    s_vals = torch.tensor(s_codes, dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    g = 2.0 ** -4
    rows = len(s_codes)
    cols = 16
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    for j in range(8):
        codes[:, j] = (2 * j) | ((2 * j + 1) << 4)  # nibbles 0..15 in column order
    scales = np.array(s_codes, dtype=np.uint8).reshape(rows, 1)
    out, n_inexact = oracle.nvfp4_dequant_bf16(codes, scales, g)
    assert n_inexact == 0
    vals = torch.tensor([e2m1[n] for n in range(16)], dtype=torch.float32)
    ref = (vals[None, :] * s_vals[:, None] * g).to(torch.bfloat16).view(torch.int16)
    assert np.array_equal(out, ref.numpy().view(np.uint16))


def test_nvfp4_low_nibble_is_the_even_column():
    codes = np.array([[0x21, 0x00, 0x00, 0x00, 0x00, 0x00, 0x00, 0x00]], dtype=np.uint8)
    scales = np.array([[0x38]], dtype=np.uint8)  # e4m3 1.0
    out, _ = oracle.nvfp4_dequant_bf16(codes, scales, 1.0)
    assert oracle.bf16_value(int(out[0, 0])) == 0.5  # nibble 0x1
    assert oracle.bf16_value(int(out[0, 1])) == 1.0  # nibble 0x2


def test_bf16_exactness_domain_of_e4m3_times_e8m0():
    """e4m3(code) * 2^(c-127) survives bf16 for every finite code iff c in [3, 246]."""
    e4 = torch_e4m3_table()
    exact_cs = []
    for c in range(255):
        s = math.ldexp(1.0, c - 127)
        all_exact = True
        for code in FINITE_E4M3:
            v = float(e4[code]) * s
            bits, inexact = oracle.bf16_rne(v)
            ref = torch.tensor([v], dtype=torch.float64).float()
            f32_exact = float(ref[0]) == v
            rt = float(ref.to(torch.bfloat16).double()[0]) if f32_exact else math.nan
            assert inexact == (not (f32_exact and rt == v)), (code, c)
            all_exact &= not inexact
        if all_exact:
            exact_cs.append(c)
    assert exact_cs == list(range(3, 247))


def test_bf16_gemv_matches_numpy():
    rng = np.random.default_rng(2)
    b = rng.integers(0, 1 << 16, size=(70, 96), dtype=np.uint16)
    b[(b & 0x7F80) == 0x7F80] = 0x3F80  # no inf/NaN patterns
    x = rng.standard_normal((2, 96)).astype(np.float32)
    y, a = oracle.bf16_gemv(b, x)
    w = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    ref = x.astype(np.float64) @ w.T
    ref_abs = np.abs(x.astype(np.float64)) @ np.abs(w).T
    np.testing.assert_allclose(a, ref_abs, rtol=1e-12)
    assert np.all(np.abs(y - ref) <= 1e-12 * ref_abs + 1e-300)


def test_nvfp4_expert_composite_matches_manual_composition():
    case = synth.nvfp4_case(n_experts=5, rows=40, cols=64, n_active=3, seed=8)
    y, a, scratch = oracle.nvfp4_expert_dequant_gemv(case.codes, case.scales, case.gscale,
                                                     case.ids, case.x, want_scratch=True)
    for k, e in enumerate(case.ids):
        b, nin = oracle.nvfp4_dequant_bf16(case.codes[e], case.scales[e], float(case.gscale[e]))
        assert nin == 0
        yk, _ = oracle.bf16_gemv(b, case.x)
        assert np.array_equal(y[k], yk[0])
        if k == len(case.ids) - 1:
            assert np.array_equal(scratch, b)


def _nvfp4_decode_numpy(codes, scales, g, block=16, low_first=True):
    """Independent NVFP4 decode to bf16 bits: golden OCP e2m1 values, torch's
    float8_e4m3fn decoder for the scales, torch's float -> bfloat16 rounding,
    and the layout read for the routed experts ("Module dsv4_gpu" page, enum
    ExpertKind: trunk = modelopt NVFP4): column 2j in the low nibble, one e4m3
    scale per 16 consecutive columns of a row, one f32 global scale.  `block`
    and `low_first` exist only so the teeth below can break the layout."""
    e2m1 = _golden_format_values()["e2m1"]
    t = np.array([e2m1[n] for n in range(16)], dtype=np.float64)
    e4 = torch_e4m3_table()
    lo, hi = codes & 15, codes >> 4
    nib = np.stack([lo, hi] if low_first else [hi, lo], axis=-1).reshape(codes.shape[:-1] + (2 * codes.shape[-1],))
    s = np.repeat(e4[scales], block, axis=-1)[..., : nib.shape[-1]]
    v = torch.from_numpy(t[nib] * s * float(g))
    return v.float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16), v.numpy()


@pytest.mark.parametrize("rows,cols,seed", [(37, 256, 21), (5, 4096, 22), (64, 96, 23)])
def test_nvfp4_matches_independent_decode_and_layout_teeth(rows, cols, seed):
    """The oracle's bf16 bytes equal an independent decode at widths with many
    16-column scale blocks per row; a 32-column scale index or a high-nibble-
    first reading gives different bytes, so either slip fails here."""
    case = synth.nvfp4_case(n_experts=2, rows=rows, cols=cols, n_active=1, seed=seed)
    for e in range(2):
        g = float(case.gscale[e])
        out, n_inexact = oracle.nvfp4_dequant_bf16(case.codes[e], case.scales[e], g)
        assert n_inexact == 0
        want, exact = _nvfp4_decode_numpy(case.codes[e], case.scales[e], g)
        assert np.array_equal(out, want)
        # the bf16 bytes carry the exact products (no rounding anywhere)
        back = torch.from_numpy(want.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
        assert np.array_equal(back, exact)
        sc = case.scales[e]
        by32 = sc[:, np.minimum(np.arange(cols) // 32, sc.shape[1] - 1)]
        wrong_scale, _ = _nvfp4_decode_numpy(case.codes[e], by32, g, block=1)
        wrong_nibble, _ = _nvfp4_decode_numpy(case.codes[e], sc, g, low_first=False)
        assert not np.array_equal(out, wrong_scale)
        assert not np.array_equal(out, wrong_nibble)


def test_nvfp4_expert_gemv_matches_independent_decode_and_matmul():
    case = synth.nvfp4_case(n_experts=6, rows=33, cols=512, n_active=4, seed=24)
    y, a, _ = oracle.nvfp4_expert_dequant_gemv(case.codes, case.scales, case.gscale, case.ids, case.x)
    x = case.x.astype(np.float64)
    for k, e in enumerate(case.ids):
        _, w = _nvfp4_decode_numpy(case.codes[e], case.scales[e], float(case.gscale[e]))
        np.testing.assert_allclose(a[k], np.abs(w) @ np.abs(x), rtol=1e-12)
        assert np.all(np.abs(y[k] - w @ x) <= 1e-12 * a[k])


def test_nvfp4_expert_rejects_bad_ids():
    case = synth.nvfp4_case(n_experts=4, rows=8, cols=32, n_active=2, seed=1)
    for ids in ([0, 0], [0, 4], [-1, 1]):
        with pytest.raises(oracle.OracleError):
            oracle.nvfp4_expert_dequant_gemv(case.codes, case.scales, case.gscale,
                                             np.array(ids, dtype=np.int32), case.x)


# ------------------------------------------------------------------ MXFP4 experts
def _mxfp4_decode_numpy(codes, scales, block=32, low_first=True):
    """Independent decode: golden OCP e2m1 values, torch's e8m0 decoder, the
    documented layout (column 2j in the low nibble, one scale per 32 columns).
    `block` / `low_first` exist only so the teeth below can break the layout."""
    e2m1 = _golden_format_values()["e2m1"]
    t = np.array([e2m1[n] for n in range(16)], dtype=np.float64)
    e8 = torch_e8m0_table()
    lo, hi = codes & 15, codes >> 4
    nib = np.stack([lo, hi] if low_first else [hi, lo], axis=-1).reshape(codes.shape[:-1] + (2 * codes.shape[-1],))
    s = np.repeat(e8[scales].astype(np.float64), block, axis=-1)[..., : nib.shape[-1]]
    return t[nib] * s


def test_mxfp4_one_hot_reproduces_each_weight():
    e2m1 = _golden_format_values()["e2m1"]
    e8 = torch_e8m0_table()
    s_codes = [0, 1, 100, 119, 127, 128, 200, 254]
    rows, cols = len(s_codes), 64
    codes = np.zeros((1, rows, cols // 2), dtype=np.uint8)
    for j in range(cols // 2):  # nibbles 0..15 in column order, twice per row
        codes[0, :, j] = ((2 * j) % 16) | (((2 * j + 1) % 16) << 4)
    scales = np.array([[s, (s + 7) % 255] for s in s_codes], dtype=np.uint8)[None]
    for c in range(cols):
        x = np.zeros(cols, dtype=np.float32)
        x[c] = 1.0
        y, _ = oracle.mxfp4_expert_gemv(codes, scales, np.array([0], dtype=np.int32), x)
        for r in range(rows):
            want = e2m1[c % 16] * float(e8[scales[0, r, c // 32]])
            assert float(y[0, r]) == want, (r, c)  # sums start at +0: the sign of a zero is not graded


def test_mxfp4_matches_independent_numpy_decode_and_layout_teeth():
    case = synth.mxfp4_case(n_experts=5, rows=37, cols=256, n_active=3, seed=11)
    y, a = oracle.mxfp4_expert_gemv(case.codes, case.scales, case.ids, case.x)
    x = case.x.astype(np.float64)
    for k, e in enumerate(case.ids):
        w = _mxfp4_decode_numpy(case.codes[e], case.scales[e])
        np.testing.assert_allclose(a[k], np.abs(w) @ np.abs(x), rtol=1e-12)
        assert np.all(np.abs(y[k] - w @ x) <= 1e-12 * a[k])
        # teeth: indexing the 32-column scales by c / 16, or taking the high nibble
        # first, gives other numbers
        sc = case.scales[e]
        by16 = sc[:, np.minimum(np.arange(256) // 16, sc.shape[1] - 1)]
        wrong_scale = _mxfp4_decode_numpy(case.codes[e], by16, block=1)
        wrong_nibble = _mxfp4_decode_numpy(case.codes[e], sc, low_first=False)
        for wrong in (wrong_scale, wrong_nibble):
            assert np.max(np.abs(y[k] - wrong @ x)) > 1e-6 * np.max(a[k])


def test_mxfp4_scale_ff_is_nan_for_its_row_only():
    case = synth.mxfp4_case(n_experts=2, rows=6, cols=64, n_active=2, seed=12)
    case.scales[case.ids[0], 3, 1] = 0xFF
    y, _ = oracle.mxfp4_expert_gemv(case.codes, case.scales, case.ids, case.x)
    assert np.isnan(y[0, 3]) and not np.isnan(np.delete(y[0], 3)).any() and not np.isnan(y[1]).any()


def test_mxfp4_ids_repeat_allowed_and_range_checked():
    case = synth.mxfp4_case(n_experts=3, rows=4, cols=32, n_active=2, seed=13)
    y, _ = oracle.mxfp4_expert_gemv(case.codes, case.scales, np.array([1, 1], dtype=np.int32), case.x)
    assert np.array_equal(y[0], y[1])
    for ids in ([3], [-1]):
        with pytest.raises(oracle.OracleError):
            oracle.mxfp4_expert_gemv(case.codes, case.scales, np.array(ids, dtype=np.int32), case.x)
