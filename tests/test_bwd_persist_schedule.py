"""The persistent d = 64 backward kernel's barrier protocol, checked on the CPU.

A model of `exact_attention_61_gb300/csrc/attn_bwd_persist.cuh`. One CTA's roles run as
coroutines over mbarriers with the hardware's parity-wait rule:
- the loader: K/V per item, the Q/dO ring per Q tile, an end-of-list hand-off;
- the dQ warps: an acknowledgement per item, the dQ read-out and reduce per Q tile;
- the MMA warp: per item the K/V copy into TMEM (tcgen05.cp), then the MMAs;
- the two compute warpgroups, one per 64-query half.

The tensor core executes the MMA warp's copies and MMAs in issue order. Copies land after
random delays, and the roles advance at random. Over many random schedules and item lists the model
checks three things:

1. every parity wait is exact: when it polls, the barrier has completed either the phase
   it waits for or the one before it;
2. no data hazard. S^T/dP^T never overwrite P^T/dS^T that dV/dK still have to read. K/V in
   TMEM are copied over only once the previous item's S^T/dP^T executed (checked when the
   copy is issued, not only when it runs). K and V in shared
   memory are reloaded only after every reader is done; V shares the second dS buffer. A dS
   buffer is rewritten only after the dQ that read it. The dQ columns are overwritten only
   after they were read out. The accumulators are overwritten only after the previous
   item's epilogue read them. A ring stage is reloaded only after its MMAs, its vector
   reads and its dQ reduce are done;
3. no deadlock: every schedule finishes.
"""
import random

import pytest

ST = 4  # Q/dO ring stages at d = 64


class HazardError(AssertionError):
    pass


class Bar:
    def __init__(self, name, count=1):
        self.name, self.count, self.arrived, self.tx, self.done = name, count, 0, 0, 0

    def _maybe_complete(self):
        if self.arrived == self.count and self.tx == 0:
            self.done += 1
            self.arrived = 0

    def arrive(self, tx=0):
        self.arrived += 1
        self.tx += tx
        if self.arrived > self.count:
            raise HazardError(f"{self.name}: more arrivals than its count in one phase")
        self._maybe_complete()

    def complete_tx(self, n):
        self.tx -= n
        self._maybe_complete()


class Model:
    def __init__(self, items, rng, plant=None, tc_weight=2, slow=None):
        """items: Q tiles per work item of this CTA (the list ends with the -1 hand-off).
        slow: index of a role (loader, dQ warps, MMA, warpgroup 0, warpgroup 1) that runs
        twenty times less often than the others."""
        self.items, self.rng, self.plant, self.tc_weight, self.slow = items, rng, plant, tc_weight, slow
        B = Bar
        self.kv = B("kv")
        self.qd_full = [B(f"qd_full{s}") for s in range(ST)]
        self.qd_empty = [B(f"qd_empty{s}", 4) for s in range(ST)]  # MMA, two warpgroups, dQ store
        self.sdp = [B(f"sdp{h}") for h in range(2)]
        self.pds = [B(f"pds{h}") for h in range(2)]
        self.dq_full = B("dq_full")
        self.dq_read = B("dq_read")
        self.acc = B("acc")
        self.dq_item = B("dq_item")  # the dQ warps read item k (passed their K/V wait)
        self.acc_free = B("acc_free", 2)
        self.queue = []  # tensor core FIFO: ("mma", fn) / ("commit", bar)
        self.tma = []    # copies in flight
        # data state
        self.smem_kv = None            # item whose K/V landed in shared memory
        self.tmem_kv = None            # item whose K/V are in TMEM
        self.sdp_reads_kv = {}         # item -> S^T/dP^T MMAs issued, not executed
        self.k_smem_readers = {}       # item -> dQ MMAs issued, not executed (they read K)
        self.half = {}                 # (h) -> ("S", gi) executed S/dP, or ("P", gi) written P/dS
        self.dv_pending = {}           # (gi, h) -> dV/dK MMAs issued, not executed
        self.ds_buf = [None, None]     # Q tile whose dS is in each buffer
        self.ds_readers = [0, 0]       # dQ MMAs issued, not executed, per buffer
        self.dq_tmem = None            # ("dq", gi) executed / ("read", gi) read out
        self.stage = [None] * ST       # Q tile landed in each ring stage
        self.stage_mma = {}            # gi -> MMAs issued on its stage, not executed
        self.stage_vec_busy = set()    # gi whose vectors a compute warpgroup is reading
        self.stage_reduce = set()      # gi whose dQ tile the reduce is reading
        self.acc_item = None           # item accumulated into dV/dK
        self.acc_pending = 0           # dV/dK MMAs issued, not executed
        self.acc_read = [True, True]   # the accumulators were read out, per warpgroup
        self.v_copied = set()          # items whose V was copied into TMEM

    # ---- tensor core and copies ----------------------------------------------------------
    def issue(self, fn):
        self.queue.append(("mma", fn))

    def commit(self, bar):
        self.queue.append(("commit", bar))

    def tc_step(self):
        if not self.queue:
            return False
        kind, x = self.queue.pop(0)
        if kind == "mma":
            x()
        else:
            x.arrive()
        return True

    def tma_step(self):
        if not self.tma:
            return False
        self.tma.pop(self.rng.randrange(len(self.tma)))()
        return True

    def wait(self, bar, k):
        """Wait for phase k of `bar` (its k-th completion, 0-based), checking exactness."""
        while True:
            if bar.done not in (k, k + 1):
                raise HazardError(f"{bar.name}: wait for phase {k} while {bar.done} completed")
            if bar.done == k + 1:
                return
            yield

    # ---- roles ---------------------------------------------------------------------------
    def loader(self):
        gi = 0
        for k, n_it in enumerate(self.items):
            if k > 0 and self.plant != "loader_no_dq_item_wait":
                yield from self.wait(self.dq_item, k - 1)
            if n_it < 0:  # end of the list: complete the K/V barrier's next phase with no bytes
                if k > 0:
                    if self.plant == "end_waits_kv_only":
                        yield from self.wait(self.kv, k - 1)
                    else:
                        yield from self.wait(self.acc, k - 1)
                self.kv.arrive()
                return
            if k > 0 and self.plant != "loader_no_acc_wait":
                yield from self.wait(self.acc, k - 1)
            if self.k_smem_readers.get(k - 1, 0):
                raise HazardError(f"K of item {k} reloaded while a dQ product of item {k - 1} reads K")
            if self.ds_readers[1]:
                raise HazardError(f"V of item {k} loaded over dS buffer 1 while a dQ product reads it")
            if k > 0 and (k - 1) not in self.v_copied:
                raise HazardError(f"K/V of item {k} reloaded before item {k - 1}'s copy into TMEM")
            self.kv.arrive(tx=1)

            def land_kv(k=k):
                self.smem_kv = k
                self.ds_buf[1] = None  # V lands over the second dS buffer
                self.kv.complete_tx(1)
            self.tma.append(land_kv)
            for _ in range(n_it):
                s = gi % ST
                if gi >= ST:
                    yield from self.wait(self.qd_empty[s], gi // ST - 1)
                    old = gi - ST
                    if self.stage_mma.get(old, 0) or old in self.stage_vec_busy or old in self.stage_reduce:
                        raise HazardError(f"stage {s} reloaded while Q tile {old} still uses it")
                self.stage_mma[gi] = 0
                self.qd_full[s].arrive(tx=1)

                def land_q(s=s, gi=gi):
                    self.stage[s] = gi
                    self.qd_full[s].complete_tx(1)
                self.tma.append(land_q)
                gi += 1
                yield

    def dq_warps(self):
        gi = 0
        for k, n_it in enumerate(self.items):
            yield from self.wait(self.kv, k)
            if n_it < 0:
                return
            self.dq_item.arrive()
            for _ in range(n_it):
                yield from self.wait(self.dq_full, gi)
                if self.dq_tmem != ("dq", gi):
                    raise HazardError(f"dQ read-out of Q tile {gi} finds {self.dq_tmem}")
                self.dq_tmem = ("read", gi)
                self.dq_read.arrive()
                self.stage_reduce.add(gi)
                yield  # the reduce reads the staged tile
                self.stage_reduce.discard(gi)
                self.qd_empty[gi % ST].arrive()
                gi += 1

    def mma(self):
        gi = 0

        def issue_sdp(g, h, k):
            self.sdp_reads_kv[k] = self.sdp_reads_kv.get(k, 0) + 1
            self.stage_mma[g] += 1

            def run(g=g, h=h, k=k):
                if self.tmem_kv != k:
                    raise HazardError(f"S^T/dP^T({g}) read K/V of item {self.tmem_kv} in TMEM, not {k}")
                if self.stage[g % ST] != g:
                    raise HazardError(f"S^T/dP^T({g}) read stage {g % ST} before Q tile {g} landed")
                prev = self.half.get(h)
                if prev is not None and prev[0] == "P" and self.dv_pending.get((prev[1], h), 0):
                    raise HazardError(f"S^T/dP^T({g}) overwrote P^T/dS^T({prev[1]}) before dV/dK read them")
                self.half[h] = ("S", g)
                self.sdp_reads_kv[k] -= 1
                self.stage_mma[g] -= 1
            self.issue(run)
            self.commit(self.sdp[h])

        for k, n_it in enumerate(self.items):
            if self.plant != "mma_cp_before_kv_wait":
                yield from self.wait(self.kv, k)
            if n_it < 0:
                if self.plant == "mma_cp_before_kv_wait":
                    yield from self.wait(self.kv, k)
                return
            # the K/V copy into TMEM, queued ahead of the item's MMAs
            if self.sdp_reads_kv.get(k - 1, 0):
                raise HazardError(f"K/V of item {k} copied into TMEM while S^T/dP^T of item {k - 1} read it")

            def cp(k=k):
                if self.smem_kv != k:
                    raise HazardError(f"K/V copy of item {k} read shared memory holding item {self.smem_kv}")
                self.tmem_kv = k
                self.v_copied.add(k)
            self.issue(cp)
            if self.plant == "mma_cp_before_kv_wait":
                yield from self.wait(self.kv, k)
            for h in range(2):
                if h == 0:
                    yield from self.wait(self.qd_full[gi % ST], gi // ST)
                issue_sdp(gi, h, k)
            for it in range(n_it):
                for h in range(2):
                    yield from self.wait(self.pds[h], gi)
                    if it == 0 and h == 0 and k > 0 and self.plant != "mma_no_acc_free_wait":
                        yield from self.wait(self.acc_free, k - 1)
                    first = it == 0 and h == 0
                    self.dv_pending[(gi, h)] = 2
                    self.acc_pending += 2
                    self.stage_mma[gi] += 2

                    def dv(g=gi, h=h, k=k, first=first):
                        if self.half.get(h) != ("P", g):
                            raise HazardError(f"dV/dK({g}, {h}) read {self.half.get(h)}")
                        if self.stage[g % ST] != g:
                            raise HazardError(f"dV/dK({g}) read stage {g % ST} holding Q tile {self.stage[g % ST]}")
                        if first:
                            if not all(self.acc_read):
                                raise HazardError(f"item {k} overwrote dV/dK before the epilogue read them")
                            self.acc_item = k
                            self.acc_read = [False, False]
                        self.dv_pending[(g, h)] -= 1
                        self.acc_pending -= 1
                        self.stage_mma[g] -= 1
                    self.issue(dv)
                    self.issue(lambda g=gi, h=h: self._dv_tail(g, h))
                    if it + 1 < n_it:
                        if h == 0:
                            yield from self.wait(self.qd_full[(gi + 1) % ST], (gi + 1) // ST)
                        issue_sdp(gi + 1, h, k)
                if gi > 0:
                    yield from self.wait(self.dq_read, gi - 1)
                self.ds_readers[gi & 1] += 1
                self.k_smem_readers[k] = self.k_smem_readers.get(k, 0) + 1

                def dq(g=gi, k=k):
                    if self.ds_buf[g & 1] != g:
                        raise HazardError(f"dQ({g}) read dS buffer {g & 1} holding {self.ds_buf[g & 1]}")
                    if self.smem_kv != k:
                        raise HazardError(f"dQ({g}) read K of item {self.smem_kv}, not {k}")
                    if self.dq_tmem is not None and self.dq_tmem[0] == "dq":
                        raise HazardError(f"dQ({g}) overwrote dQ({self.dq_tmem[1]}) before its read-out")
                    self.dq_tmem = ("dq", g)
                    self.ds_readers[g & 1] -= 1
                    self.k_smem_readers[k] -= 1
                self.issue(dq)
                self.commit(self.dq_full)
                self.commit(self.qd_empty[gi % ST])
                gi += 1
                yield
            self.commit(self.acc)

    def _dv_tail(self, g, h):
        # the second of the two products (dK) of half h: same bookkeeping as the first
        self.dv_pending[(g, h)] -= 1
        self.acc_pending -= 1
        self.stage_mma[g] -= 1

    def compute(self, h):
        gi = 0
        for k, n_it in enumerate(self.items):
            yield from self.wait(self.kv, k)
            if n_it < 0:
                return
            for _ in range(n_it):
                s = gi % ST
                yield from self.wait(self.qd_full[s], gi // ST)
                yield from self.wait(self.sdp[h], gi)
                if self.half.get(h) != ("S", gi):
                    raise HazardError(f"warpgroup {h} read S^T/dP^T({gi}) but TMEM holds {self.half.get(h)}")
                self.stage_vec_busy.add(gi)
                yield  # reads the tile's LSE/D vectors
                self.stage_vec_busy.discard(gi)
                b = gi & 1
                if self.ds_readers[b]:
                    raise HazardError(f"dS({gi}) written over buffer {b} while dQ({self.ds_buf[b]}) reads it")
                if b == 1 and k not in self.v_copied:
                    raise HazardError(f"dS({gi}) written over V of item {k} before its copy into TMEM")
                self.ds_buf[b] = gi
                self.half[h] = ("P", gi)
                self.pds[h].arrive()
                self.qd_empty[s].arrive()
                gi += 1
                yield
            yield from self.wait(self.acc, k)
            if self.acc_pending or self.acc_item != k:
                raise HazardError(f"epilogue of item {k} read dV/dK before every product executed")
            yield  # reads its half of dV and dK out of TMEM
            if self.acc_item != k:
                raise HazardError(f"dV/dK of item {self.acc_item} overwrote item {k}'s during its epilogue")
            self.acc_read[h] = True
            self.acc_free.arrive()
            yield

    def run(self, max_steps=400000):
        roles = [self.loader(), self.dq_warps(), self.mma(), self.compute(0), self.compute(1)]
        weight = {id(r): (1 if i == self.slow else 20) for i, r in enumerate(roles)}
        live = list(roles)
        for _ in range(max_steps):
            choices = ["role"] * (len(live) * 4) + ["tc"] * self.tc_weight + ["tma"] * 2
            progressed = False
            for pick in self.rng.sample(choices, len(choices)):
                if pick == "tc" and self.tc_step():
                    progressed = True
                    break
                if pick == "tma" and self.tma_step():
                    progressed = True
                    break
                if pick == "role" and live:
                    r = self.rng.choices(live, weights=[weight[id(x)] for x in live])[0]
                    try:
                        next(r)
                    except StopIteration:
                        live.remove(r)
                    progressed = True
                    break
            if not live and not self.queue and not self.tma:
                return
            if not progressed:
                break
        raise HazardError("no progress: deadlock or runaway schedule")


def item_lists(rng, n, short_only=False):
    out = []
    for _ in range(n):
        hi = 4 if short_only else 9
        out.append([rng.randint(1, hi) for _ in range(rng.randint(0, 4))] + [-1])
    return out


def test_persistent_backward_random_schedules():
    rng = random.Random(6102)
    for items in item_lists(rng, 120) + item_lists(rng, 60, short_only=True):
        for tc_weight in (1, 3, 12):  # a slow, medium and fast tensor core
            for slow in (None, rng.randrange(5)):  # every role at one speed, or one role lagging
                Model(items, random.Random(rng.random()), tc_weight=tc_weight, slow=slow).run()


def test_persistent_backward_headline_items():
    """The item lists one CTA gets at the headline size: 13-14 non-causal key tiles of 32 Q
    tiles each, and a causal mix (a key tile kt sees 32 - kt Q tiles)."""
    rng = random.Random(9)
    Model([32] * 13 + [-1], rng).run(max_steps=4 * 10 ** 6)
    Model([32, 24, 17, 11, 6, 2, 1, -1], rng).run(max_steps=4 * 10 ** 6)


@pytest.mark.parametrize("plant", ["end_waits_kv_only", "loader_no_acc_wait", "mma_no_acc_free_wait",
                                   "mma_cp_before_kv_wait", "loader_no_dq_item_wait"])
def test_model_catches_planted_protocol_errors(plant):
    """Each planted mistake is caught as a hazard or an inexact parity wait on some
    schedule. The first is the end-of-list hand-off that waits only for the previous
    item's K/V copy: with items of at most four Q tiles the loader never blocks on the ring,
    and the K/V barrier can run two phases ahead of a role. The fourth queues the K/V copy
    into TMEM before the K/V in shared memory landed. The last starts an item without the dQ
    warps' acknowledgement of the previous one: after a one-tile item every MMA can finish
    while the dQ warps are still on the item before, and the K/V barrier runs two phases
    ahead of them."""
    rng = random.Random(11)
    caught = 0
    for items in item_lists(rng, 100, short_only=True):
        for tc_weight in (1, 3):
            for slow in (None, 1, 4):  # every role at one speed, or the dQ warps or warpgroup 1 lagging
                try:
                    Model(items, random.Random(rng.random()), plant=plant, tc_weight=tc_weight, slow=slow).run()
                except HazardError:
                    caught += 1
    assert caught > 0
