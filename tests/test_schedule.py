"""The forward kernel's job schedule, checked on the CPU.

A mirror of the issue order in `exact_attention_61_gb300/csrc/attn_fwd_kernel.cuh` (`JobOrder`
and the MMA warp's loop) is checked for the two properties its bounded waits rely on, for every
pair of per-tile key-tile counts the kernel can see and every ring depth it is built with:

1. No deadlock in the K/V ring: when the MMA warp waits for key tile j' to land, it has already
   committed the "stage empty" signal the loader needs to load j' into that stage.
2. Unambiguous parity waits on `o_done`: a softmax warpgroup at its job j may wait for phase j-1
   of its tile's `o_done` barrier (the previous O += P V). A parity wait is only exact if at
   most one phase can be pending, i.e. when S of job j completes, every O += P V of that tile up
   to j-2 has completed. The tensor core executes MMAs in issue order, so that holds if those
   P V groups were issued before S(job j). Where it does not hold the kernel waits at every job
   (lockstep), which keeps the count exact by induction.
"""
import itertools

import pytest


class JobOrder:
    """Mirror of JobOrder: for each key tile j, tile 0 then tile 1 while both need keys, then
    tile 1's remaining tiles."""

    def __init__(self, n0, n1):
        self.n0, self.n1 = n0, n1

    def total(self):
        return self.n0 + self.n1

    def job(self, t, j):
        if self.n1 == 0:
            return j
        return 2 * j + t if j < self.n0 else 2 * self.n0 + (j - self.n0)

    def tile_of(self, g):
        if self.n1 == 0:
            return 0, g
        if g < 2 * self.n0:
            return g & 1, g >> 1
        return 1, self.n0 + (g - 2 * self.n0)

    def last_job(self, j):
        return j if self.n1 == 0 else self.job(1, j)


def issue_order(jobs, sbufs):
    """The MMA warp's program: S of the first `sbufs` jobs, then for each job g: P V(g), the
    commits of that job (kv_empty after the tile's last job), then S(g + sbufs)."""
    prog = [("S", g) for g in range(min(sbufs, jobs.total()))]
    for g in range(jobs.total()):
        t, j = jobs.tile_of(g)
        prog.append(("PV", g))
        if g == jobs.last_job(j):
            prog.append(("kv_empty", j))
        if g + sbufs < jobs.total():
            prog.append(("S", g + sbufs))
    return prog


def check_schedule(n0, n1, stages, sbufs, lockstep_tail=False):
    jobs = JobOrder(n0, n1)
    prog = issue_order(jobs, sbufs)
    pos = {op: i for i, op in enumerate(prog)}
    problems = []
    # 1. ring: S of the first job of key tile j' waits for j' to land, which needs
    #    kv_empty(j' - stages) committed earlier in the same program.
    for op, g in (o for o in prog if o[0] == "S"):
        t, j = jobs.tile_of(g)
        if j >= stages and pos[("kv_empty", j - stages)] > pos[("S", g)]:
            problems.append(f"deadlock: S({g}) needs tile {j}, freed only after it")
    # 2. o_done parity
    single_tile = n0 == 0 or n1 == 0
    for t, n in ((0, n0), (1, n1)):
        for j in range(1, n):
            lockstep = single_tile or (lockstep_tail and t == 1 and j >= n0)
            if lockstep:
                continue  # waits every job: exact by induction
            g = jobs.job(t, j)
            for jj in range(j - 1):  # P V(t, jj) for jj <= j - 2
                if pos[("PV", jobs.job(t, jj))] > pos[("S", g)]:
                    problems.append(f"ambiguous o_done wait: tile {t} job {j} (P V of job {jj} may be pending)")
    return problems


# The one-CTA kernel: 256 rows per CTA (two 128-row tiles), so tile 1 needs 0, n0 or n0 + 1
# key tiles under any mask; 4 stages / 3 S buffers at d=64, 2 / 2 at d=128.
@pytest.mark.parametrize("stages,sbufs", [(4, 3), (2, 2)])
def test_one_cta_schedule_is_deadlock_free_and_exact(stages, sbufs):
    for n0 in range(0, 40):
        for n1 in {0, n0, n0 + 1}:
            if n0 == 0 and n1 == 0:
                continue
            assert check_schedule(n0, n1, stages, sbufs) == [], (n0, n1)


def test_mirror_matches_the_documented_order():
    jobs = JobOrder(3, 4)
    assert [jobs.tile_of(g) for g in range(7)] == [(0, 0), (1, 0), (0, 1), (1, 1), (0, 2), (1, 2), (1, 3)]
    assert [jobs.job(1, j) for j in range(4)] == [1, 3, 5, 6]
    assert issue_order(jobs, 3)[:6] == [("S", 0), ("S", 1), ("S", 2), ("PV", 0), ("S", 3), ("PV", 1)]


def test_a_two_tile_tail_needs_lockstep():
    """With tile 1 two key tiles ahead of tile 0 (n1 = n0 + 2, as when 256-row tiles are
    paired), the tail's second job could see two pending phases: the check finds it, and
    waiting at every tail job removes it."""
    problems = check_schedule(5, 7, 4, 3)
    assert any("ambiguous" in p for p in problems)
    for n0, n1 in itertools.product(range(1, 30), repeat=2):
        if n1 >= n0:
            assert check_schedule(n0, n1, 6, 3, lockstep_tail=True) == [], (n0, n1)


def test_a_shallow_ring_with_deep_lookahead_deadlocks():
    """The check is not vacuous: S issued three jobs ahead through a one-stage ring would wait
    for a stage its own program frees only later."""
    assert any("deadlock" in p for p in check_schedule(6, 6, 1, 3))
