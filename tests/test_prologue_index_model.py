"""CPU model of the backward prologue's -D table indexing (csrc/attn_prep.cu,
bwd_prologue_bf16_kernel): the kernel reaches a written entry's batch row b,
position t and chunk c by carrying from one division (per four-row group for
rows at least a block wide; per thread and pass for narrower rows).  Every
thread of the launch is replayed here and each (b, t, c) it writes is
compared with the plain divisions of the entry's flat index, over shapes with
one and several batch rows, short and long sequences and row widths from 2
to 224 chunks."""
import itertools

import pytest

BLOCK, U, R = 256, 4, 4


def narrow_rows(B, T, dot_units, grid):
    """The flattened pass (dot_units < BLOCK): yields (u, b, t, c) per write."""
    rows = B * T
    n_units = rows * dot_units
    for blk in range(grid):
        for tid in range(BLOCK):
            lane = tid & 31
            base = (blk * BLOCK + (tid & ~31)) * U
            while base < n_units:
                u0 = base + lane
                row0 = u0 // dot_units
                c = u0 - row0 * dot_units
                b, t = divmod(row0, T)
                for i in range(U):
                    u = base + 32 * i + lane
                    if u < n_units:
                        yield u, b, t, c
                    c += 32
                    while c >= dot_units:
                        c -= dot_units
                        t += 1
                        if t == T:
                            t, b = 0, b + 1
                base += grid * BLOCK * U


def wide_rows(B, T, grid):
    """The group loop (rows at least a block wide): yields (row, b, t) per row."""
    rows = B * T
    n_groups = (rows + R - 1) // R
    for blk in range(grid):
        for grp in range(blk, n_groups, grid):
            row0 = grp * R
            nr = min(R, rows - row0)
            b0, t0 = divmod(row0, T)
            for r in range(nr):
                t, b = t0 + r, b0
                while t >= T:
                    t, b = t - T, b + 1
                yield row0 + r, b, t


@pytest.mark.parametrize("B,T", list(itertools.product([1, 2, 3], [1, 3, 5, 17, 64, 130])))
def test_narrow_row_indexing(B, T):
    for du in (2, 4, 8, 12, 16, 24, 32, 48, 96, 128, 160, 224):
        for grid in (1, 3):
            seen = set()
            for u, b, t, c in narrow_rows(B, T, du, grid):
                row = u // du
                assert (b, t, c) == (row // T, row % T, u % du), (B, T, du, grid, u)
                seen.add(u)
            assert len(seen) == B * T * du            # every chunk written exactly once


@pytest.mark.parametrize("B,T", list(itertools.product([1, 2, 3, 5], [1, 2, 3, 5, 70, 101])))
def test_wide_row_indexing(B, T):
    for grid in (1, 7):
        rows = [row for row, b, t in wide_rows(B, T, grid) if (b, t) == divmod(row, T)]
        assert sorted(rows) == list(range(B * T))


def test_gpt2_shaped_launch():
    """The GPT-2-shaped workload's own geometry and grid (B=8, T=1024,
    96 chunks per row, min(rows/4, 4 x 152) blocks)."""
    B, T, du = 8, 1024, 96
    grid = min((B * T + 3) // 4, 152 * 4)
    n = 0
    for u, b, t, c in narrow_rows(B, T, du, grid):
        row = u // du
        assert (b, t, c) == (row // T, row % T, u % du)
        n += 1
    assert n == B * T * du
