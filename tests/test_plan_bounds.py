"""CPU checks of the streaming-GEMV launch geometry: for many shapes, every
shared-memory read, bulk copy, global read and output write the kernel's index
arithmetic can form stays inside its buffer, every output has a thread that
writes it, and the resources fit the device.  These are the bounds the kernel
relies on; they are checked here, without a GPU, before any launch."""
import itertools

import pytest

GB300 = dict(sms=152, smem_per_sm=233472, smem_per_block=232448)
STATIC_SMEM = 4736 + 64  # red/argmax buffers of the kernel (ptxas report) + s_is_last slack
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


def check_plan(ops, m, rows, cols, bpw):
    p = ops.plan_query(m, rows, cols, bpw, **GB300)
    pc, panels, tw, teams = p["panel_cols"], p["panels"], p["team_warps"], p["teams"]
    rb, rt, R, sb, ns = p["row_batches"], p["rows_per_batch"], p["stage_rows"], p["stage_bytes"], p["stages"]
    mp = 1
    while mp < m:
        mp *= 2
    assert rt == 8 // mp
    # column panels tile [0, cols) exactly, in 16-column chunks
    assert pc % 16 == 0 and 16 <= pc <= 4096
    assert (panels - 1) * pc < cols <= panels * pc
    # every chunk of a panel row has a thread: team_threads * 16 columns >= panel
    team_threads = tw * 32
    assert teams * tw == 8 and team_threads * 16 >= pc
    # stage rows: a power of two dividing 128 (a group never straddles a scale row block)
    assert R == teams * rb * rt and R & (R - 1) == 0 and 128 % R == 0
    assert 1 <= rb <= 8
    # smem row reads: lrow < R, chunk*16 < pwb <= pc*bpw  =>  offset + 16 <= R * pc * bpw
    assert sb == R * pc * bpw and sb % 16 == 0 and sb < (1 << 20)
    max_read_end = (R - 1) * pc * bpw + pc * bpw
    assert max_read_end <= sb
    # finalize: outputs per team per stage = rb * 8 slots, covered by the stride loop
    assert team_threads % 8 == 0
    # ring depth and shared memory
    assert 2 <= ns <= 8
    dyn = p["dynamic_smem_bytes"]
    assert dyn == ns * sb + 64
    assert dyn + STATIC_SMEM <= GB300["smem_per_block"]
    assert p["ctas_per_sm"] * (dyn + STATIC_SMEM + 1024) <= GB300["smem_per_sm"]
    # groups cover the rows; copies of the last group stop at `rows`
    assert p["n_groups"] * R >= rows > (p["n_groups"] - 1) * R
    grid = min(p["n_groups"], GB300["sms"] * p["ctas_per_sm"], MAX_GRID)
    assert 1 <= grid <= MAX_GRID
    # CTA group ranges partition [0, n_groups) with no gaps
    ng = p["n_groups"]
    ends = [(b * ng // grid, (b + 1) * ng // grid) for b in range(grid)]
    assert ends[0][0] == 0 and ends[-1][1] == ng
    assert all(ends[i][1] == ends[i + 1][0] for i in range(grid - 1))
    return p


@pytest.mark.parametrize("bpw", [1, 2])
def test_plans_stay_in_bounds(ops, bpw):
    for m, rows, cols in SHAPES:
        check_plan(ops, m, rows, cols, bpw)


def test_headline_plans(ops):
    p = check_plan(ops, 1, 4096, 4096, 1)
    assert p["panels"] == 1 and p["stage_rows"] == 8
    p = check_plan(ops, 8, 16384, 4096, 1)
    assert p["ctas_per_sm"] == 1
