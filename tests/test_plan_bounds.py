"""CPU checks of the streaming-GEMV launch geometry: for many shapes, every
shared-memory read, bulk copy, global read and output write the kernel's index
arithmetic can form stays inside its buffer, every output has a thread that
writes it, and the resources fit the device.  These are the bounds the kernel
relies on; they are checked here, without a GPU, before any launch."""
import itertools

import pytest

GB300 = dict(sms=152, smem_per_sm=233472, smem_per_block=232448)
STATIC_SMEM = 4736 + 128  # team kernel: red/argmax buffers, barriers, counters (ptxas report)
ROWWARP_STATIC_SMEM = 1024  # row-per-warp kernel: barriers + argmax scratch
MAX_GRID = 1024


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_fp8blk_gb300 import build
    build.build()
    from fp8_block_scaled_fp8blk_gb300 import ops as o
    return o


SHAPES = sorted(set(
    [(1, 512, 1024), (1, 4096, 4096), (1, 131072, 4096), (8, 16384, 4096), (1, 2048, 4096)]
    + [(m, r, c) for m, r, c in itertools.product(
        range(1, 9), (1, 7, 8, 127, 128, 129, 130, 1000, 4097),
        (16, 32, 48, 272, 512, 1008, 1024, 1040, 2048, 4080, 4096, 4112, 8192, 8208, 12304,
         16384, 20000 - 20000 % 16))]))


def _check_common(p, rows, cols, bpw):
    pc, panels = p["panel_cols"], p["panels"]
    # column panels tile [0, cols) exactly, in 16-column chunks
    assert pc % 16 == 0 and 16 <= pc <= 4096
    assert (panels - 1) * pc < cols <= panels * pc
    R, sb, ns = p["stage_rows"], p["stage_bytes"], p["stages"]
    # stage rows: a power of two dividing 128 (a group never straddles a scale row block)
    assert R & (R - 1) == 0 and 128 % R == 0
    # smem row reads: row < R, chunk*16 < pwb <= pc*bpw  =>  offset + 16 <= R * pc * bpw
    assert sb == R * pc * bpw and sb % 16 == 0 and sb < (1 << 20)
    assert 2 <= ns <= 8
    # groups cover the rows; copies of the last group stop at `rows`
    assert p["n_groups"] * R >= rows > (p["n_groups"] - 1) * R


def _check_partition(n_groups, workers):
    ends = [(b * n_groups // workers, (b + 1) * n_groups // workers) for b in range(workers)]
    assert ends[0][0] == 0 and ends[-1][1] == n_groups
    assert all(ends[i][1] == ends[i + 1][0] for i in range(workers - 1))


T8_SMEM = 1024 + 4 * 32768 + 8 * 6144 + 8 * 256 * 4  # A ring, B operands, block-max table
T8_STATIC_SMEM = 2048
T8_MAX_KB = 256


def check_tc_plan(p, m, rows, cols, bpw):
    """Tensor-core kernel: one CTA per SM over whole 128-row tiles (one scale
    row block each), every 128-column K-block of a tile in one pass.  Every
    tile's box starts inside the matrix (TMA y in [0, rows)) on a 128-column
    boundary (x a multiple of 16, as TMA requires); the ring, operands and the
    block-max table (m x K-blocks) fit the shared memory."""
    assert bpw == 1 and 128 <= cols <= 128 * T8_MAX_KB and 1 <= m <= 8
    assert p["panels"] == 1 and p["panel_cols"] == cols
    n_tiles = -(-rows // 128)
    assert p["n_groups"] == n_tiles and p["ctas_per_sm"] == 1 and p["stages"] == 4
    assert p["dynamic_smem_bytes"] == T8_SMEM
    assert p["dynamic_smem_bytes"] + T8_STATIC_SMEM <= GB300["smem_per_block"]
    nkb = -(-cols // 128)
    assert m * nkb <= 8 * T8_MAX_KB
    assert all((kb * 128) % 16 == 0 for kb in range(nkb))
    grid = min(GB300["sms"], n_tiles, MAX_GRID)
    _check_partition(n_tiles, grid)
    for b in range(grid):
        t0, t1 = b * n_tiles // grid, (b + 1) * n_tiles // grid
        assert t1 > t0 and all(0 <= 128 * t < rows for t in range(t0, t1))
    return p


def check_plan(ops, m, rows, cols, bpw):
    p = ops.plan_query(m, rows, cols, bpw, **GB300)
    if p["kernel"] == 2:
        return check_tc_plan(p, m, rows, cols, bpw)
    _check_common(p, rows, cols, bpw)
    pc, tw, teams = p["panel_cols"], p["team_warps"], p["teams"]
    R, sb, ns, dyn = p["stage_rows"], p["stage_bytes"], p["stages"], p["dynamic_smem_bytes"]
    if p["kernel"] == 1:
        # row-per-warp kernel: 4 warps per CTA, each with a private ring
        assert m == 1 and teams == 4 and 1 <= R <= 8
        # a lane's chunks k*32 + lane, k < 8*bpw, cover the whole panel row
        assert 32 * 8 * bpw * 16 >= pc * bpw
        assert dyn == teams * ns * sb
        assert dyn + ROWWARP_STATIC_SMEM <= GB300["smem_per_block"]
        assert p["ctas_per_sm"] * (dyn + ROWWARP_STATIC_SMEM + 1024) <= GB300["smem_per_sm"]
        grid = min(-(-p["n_groups"] // 4), GB300["sms"] * p["ctas_per_sm"], MAX_GRID)
        _check_partition(p["n_groups"], grid * 4)
        return p
    assert p["kernel"] == 0
    rb, rt = p["row_batches"], p["rows_per_batch"]
    mp = 1
    while mp < m:
        mp *= 2
    assert rt == 8 // mp
    # every chunk of a panel row has a thread: team_threads * 16 columns >= panel
    team_threads = tw * 32
    assert teams * tw == 8 and team_threads * 16 >= pc
    assert R == teams * rb * rt and 1 <= rb <= 8
    # finalize: outputs per team per stage = rb * 8 slots, covered by the stride loop
    assert team_threads % 8 == 0
    assert dyn == ns * sb
    assert dyn + STATIC_SMEM <= GB300["smem_per_block"]
    assert p["ctas_per_sm"] * (dyn + STATIC_SMEM + 1024) <= GB300["smem_per_sm"]
    grid = min(p["n_groups"], GB300["sms"] * p["ctas_per_sm"], MAX_GRID)
    assert 1 <= grid <= MAX_GRID
    _check_partition(p["n_groups"], grid)
    return p


@pytest.mark.parametrize("bpw", [1, 2])
@pytest.mark.parametrize("m1_kernel", [1, 2])
def test_plans_stay_in_bounds(ops, bpw, m1_kernel):
    ops.set_m1_kernel(m1_kernel)
    try:
        for m, rows, cols in SHAPES:
            check_plan(ops, m, rows, cols, bpw)
    finally:
        ops.set_m1_kernel(0)


def test_tensor_core_plans_stay_in_bounds(ops):
    ops.set_tensor_core_min_m(2, 1)  # every m >= 2 shape that qualifies
    try:
        seen = 0
        for m, rows, cols in SHAPES + [(8, 1_000_000, 4096), (5, 300_000, 16384), (2, 8, 128)]:
            p = check_plan(ops, m, rows, cols, 1)
            seen += p["kernel"] == 2
        assert seen > 100
        ops.set_tensor_core_min_m(1, 1)  # m = 1 too
        for m, rows, cols in SHAPES:
            check_plan(ops, m, rows, cols, 1)
    finally:
        ops.set_tensor_core_min_m(0, 0)


def test_headline_plans(ops):
    p = check_plan(ops, 1, 4096, 4096, 1)
    assert p["panels"] == 1 and p["kernel"] == 0  # small: team kernel
    p = check_plan(ops, 1, 131072, 4096, 1)
    assert p["kernel"] == 2  # the vocab head: tensor cores
    assert check_plan(ops, 1, 28672, 4096, 1)["kernel"] == 2  # 112 MiB: tensor cores
    assert check_plan(ops, 1, 8192, 4096, 1)["kernel"] == 0  # 32 MiB: team kernel
    assert check_plan(ops, 1, 3072, 36864, 1)["kernel"] == 1  # 108 MiB, too wide for the tensor cores
    ops.set_m1_kernel(1)
    try:
        assert check_plan(ops, 1, 131072, 4096, 1)["kernel"] == 1  # forced: row-per-warp
    finally:
        ops.set_m1_kernel(0)
    p = check_plan(ops, 8, 16384, 4096, 1)
    assert p["kernel"] == 2 and p["ctas_per_sm"] == 1  # batched verify: tensor cores
    assert check_plan(ops, 4, 16384, 4096, 1)["kernel"] == 2  # m = 4 at 64 MiB: tensor cores
    assert check_plan(ops, 4, 8192, 4096, 1)["kernel"] == 2  # m = 4 at 32 MiB: tensor cores
    assert check_plan(ops, 4, 4096, 4096, 1)["kernel"] == 0  # m = 4 at 16 MiB: CUDA cores
    assert check_plan(ops, 2, 8192, 4096, 1)["kernel"] == 0  # m = 2 at 32 MiB: CUDA cores
    assert check_plan(ops, 8, 2048, 4096, 1)["kernel"] == 0  # small: CUDA cores
    assert check_plan(ops, 1, 4096, 4096, 1)["kernel"] == 0  # 16 MiB m = 1: team kernel


# Launch-tuning settings (fp8blk_set_launch_tuning is public): stage sizes,
# CTAs per SM and ring depths across their documented ranges.
TUNINGS = [(0, 0, 1, 1, 0), (16384, 1, 1, 1, 6), (16384, 2, 1, 1, 3), (16384, 2, 1, 1, 4),
           (32768, 1, 1, 1, 3), (32768, 1, 1, 1, 4), (65536, 1, 1, 1, 2), (16384, 3, 1, 1, 4),
           (8192, 4, 1, 0, 2), (131072, 1, 0, 0, 8), (4096, 2, 1, 1, 8), (0, 1, 1, 1, 0),
           (0, 2, 1, 1, 3), (16384, 2, 1, 1, 0), (65536, 1, 1, 1, 0)]


@pytest.mark.parametrize("tuning", TUNINGS)
def test_plans_stay_in_bounds_under_launch_tuning(ops, tuning):
    ops.set_launch_tuning(*tuning)
    try:
        for m1_kernel in (1, 2):
            ops.set_m1_kernel(m1_kernel)
            for bpw in (1, 2):
                for m, rows, cols in SHAPES:
                    check_plan(ops, m, rows, cols, bpw)
    finally:
        ops.set_m1_kernel(0)
        ops.set_launch_tuning()
