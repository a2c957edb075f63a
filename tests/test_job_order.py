"""Host-side check of the job sequence of the single cooperative kernel
(input mode kInStageKV in attn_kernel.cuh), restated here from the
kernel's description: per round r of work tiles (tiles r*grid ..
(r+1)*grid - 1, tile = head * n_qblocks + query block), the heads whose
first work tile falls in round r, key tile 0 of all of them, then key tile
1, and so on.  Block b stages jobs b, b + grid, ...

Every key tile of every head must be staged exactly once (a missing one
would leave its readers waiting for a flag until their time limit), and a
job must never come after the jobs of a later round.  No GPU needed.
"""
import itertools

import pytest


def job_of(s, grid, n_bh, nqb, T):
    """(head, key tile) of job s: the arithmetic the kernel uses."""
    base = 0
    for r in itertools.count():
        h0 = (r * grid + nqb - 1) // nqb
        h1 = min(((r + 1) * grid + nqb - 1) // nqb, n_bh)
        cnt = (h1 - h0) * T
        if s < base + cnt:
            o = s - base
            j = o // (h1 - h0)
            return h0 + (o - j * (h1 - h0)), j, r
        base += cnt


def first_round(h, grid, nqb):
    return (h * nqb) // grid


@pytest.mark.parametrize("n_bh,nqb,T,grid", [
    (128, 9, 18, 152),    # the 8 x 16 x 2304 x 64 workload
    (32, 36, 72, 152),    # 2 x 16 heads, 9216 patches
    (2, 9, 17, 18),       # fewer work tiles than multiprocessors
    (80, 9, 17, 152),     # several rounds per block
    (3, 10, 20, 30),
    (1, 1, 1, 1),
    (7, 3, 5, 4),         # a round that starts no new head
    (5, 40, 3, 152),
    (2, 40, 3, 10),       # rounds inside one head: most start no new head
])
def test_every_key_tile_once_in_order_of_need(n_bh, nqb, T, grid):
    grid = min(grid, n_bh * nqb)  # the kernel's grid: min(work tiles, SMs)
    n_jobs = n_bh * T
    seen = {}
    last_round = -1
    for s in range(n_jobs):
        h, j, r = job_of(s, grid, n_bh, nqb, T)
        assert 0 <= h < n_bh and 0 <= j < T
        assert (h, j) not in seen, f"job {s} repeats {(h, j)}"
        seen[(h, j)] = s
        assert r == first_round(h, grid, nqb)  # staged with the round that first needs it
        assert r >= last_round                  # rounds in order
        last_round = r
    assert len(seen) == n_jobs
    # within a round, key tile j of every head before key tile j + 1
    for h in range(n_bh):
        for j in range(1, T):
            hh = [g for g in range(n_bh) if first_round(g, grid, nqb) == first_round(h, grid, nqb)]
            assert all(seen[(g, j - 1)] < seen[(h, j)] for g in hh)
