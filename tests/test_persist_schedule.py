"""The persistent forward kernel's barrier protocol, checked on the CPU.

A model of `exact_attention_61_gb300/csrc/attn_fwd_persist.cuh`: the loader, the S issuer,
the two softmax warpgroups (which issue their own O += P V, or hand P to a dedicated
P V warp), and the store warp run as coroutines over mbarriers with the hardware's
parity-wait rule. The tensor core executes each issuing thread's MMAs in that thread's
order but interleaves threads at random; a commit arrives once its thread's earlier MMAs
have executed; TMA copies land after random delays. Over many random schedules and work
lists (causal and ragged items included) the model checks:

1. every parity wait is exact: when it polls, the barrier has completed either the phase
   it waits for or the one before it (so the hardware's parity test cannot pass early or
   block on a later phase);
2. no data hazard: S is read only after its MMA executed, an S/P buffer is overwritten
   only after the O += P V that read it executed, a ring stage or Q buffer is reloaded
   only after every MMA (and the output store) that reads it is done, O is read out or
   rescaled only after its O += P V executed, and the next item's first O += P V runs only
   after the previous output was read;
3. no deadlock: every schedule finishes.
"""
import random

import pytest

ST, SB = 4, 3  # ring stages and S/P buffers of the head-dimension-64 kernel


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


def tile_of(n0, n1, jj):
    if n1 == 0:
        return 0, jj
    if jj < 2 * n0:
        return jj & 1, jj >> 1
    return 1, n0 + (jj - 2 * n0)


def job(n0, n1, t, j):
    if n1 == 0:
        return j
    return 2 * j + t if j < n0 else 2 * n0 + (j - n0)


def last_job(n0, n1, j):
    return j if n1 == 0 else job(n0, n1, 1, j)


class Model:
    def __init__(self, items, pv_by_wg, rng, plant=None, tc_weight=2):
        self.items, self.pv_by_wg, self.rng, self.plant = items, pv_by_wg, rng, plant
        self.tc_weight = tc_weight  # relative chance that the tensor core moves at a step
        B = Bar
        self.q_full = [[B(f"q_full{b}{t}") for t in range(2)] for b in range(2)]
        self.q_empty = [[B(f"q_empty{b}{t}") for t in range(2)] for b in range(2)]
        self.k_full = [B(f"k_full{s}") for s in range(ST)]
        self.v_full = [B(f"v_full{s}") for s in range(ST)]
        self.kv_empty = [B(f"kv_empty{s}") for s in range(ST)]
        self.s_full = [[B(f"s_full{t}{b}") for b in range(SB)] for t in range(2)]
        self.pv_done = [B(f"pv_done{b}") for b in range(SB)]
        self.p_full = [B(f"p_full{b}") for b in range(SB)]
        self.o_done = [[B(f"o_done{t}{i}") for i in range(2)] for t in range(2)]
        self.o_free = [B(f"o_free{t}") for t in range(2)]
        self.o_staged = [[B(f"o_staged{b}{t}") for t in range(2)] for b in range(2)]
        # tensor core: per issuing thread, a FIFO of ops ("mma", fn) / ("commit", bar)
        self.queues = {}
        self.tma = []  # in flight: [delay, fn]
        # data state
        self.sbuf = [None] * SB          # ("S", g, executed) or ("P", g)
        self.pv_read = set()             # jobs whose O += P V executed
        self.s_exec = set()              # jobs whose S executed
        self.stage_tile = [None] * ST    # ring tile in each stage (landed)
        self.stage_readers = {}          # ring tile -> number of MMAs still to execute
        self.q_tile = {}                 # (qb, t) -> item whose Q landed there
        self.q_readers = {}              # (item, t) -> S MMAs still to execute
        self.q_store_busy = set()        # (qb, t) buffers an output store is reading
        self.o_pv_pending = [0, 0]       # O += P V issued, not executed, per tile
        self.o_item = [None, None]       # item whose O accumulation is in TMEM per tile
        self.o_read = [True, True]       # the item's O was read out (epilogue)
        self.expected_readers = {}

    # ---- tensor core -----------------------------------------------------------------
    def issue(self, who, fn):
        self.queues.setdefault(who, []).append(("mma", fn))

    def commit(self, who, bar):
        self.queues.setdefault(who, []).append(("commit", bar))

    def tc_step(self):
        ready = [w for w, q in self.queues.items() if q]
        if not ready:
            return False
        q = self.queues[self.rng.choice(ready)]
        kind, x = q.pop(0)
        if kind == "mma":
            x()
        else:
            x.arrive()
        return True

    def tma_step(self):
        if not self.tma:
            return False
        i = self.rng.randrange(len(self.tma))
        self.tma.pop(i)()
        return True

    # ---- roles ---------------------------------------------------------------------------
    def wait(self, bar, k):
        """Wait for phase k of `bar` (k-th completion, 0-based), checking exactness."""
        while True:
            if bar.done not in (k, k + 1):
                raise HazardError(f"{bar.name}: wait for phase {k} while {bar.done} completed")
            if bar.done == k + 1:
                return
            yield

    def loader(self):
        G = 0
        for a, (n0, n1) in enumerate(self.items):
            qb = a & 1
            if a >= 2:
                for t in range(2):
                    yield from self.wait(self.q_empty[qb][t], (a >> 1) - 1)
            for t in range(2):
                nt = n1 if t else n0
                if nt > 0:
                    prev = self.q_tile.get((qb, t))
                    if prev is not None and self.q_readers.get((prev, t), 0):
                        raise HazardError(f"Q buffer {qb},{t} reloaded while S of item {prev} pending")
                    if (qb, t) in self.q_store_busy:
                        raise HazardError(f"Q buffer {qb},{t} reloaded while its output store reads it")
                    self.q_full[qb][t].arrive(tx=1)

                    def land(qb=qb, t=t, a=a):
                        self.q_tile[(qb, t)] = a
                        self.q_full[qb][t].complete_tx(1)
                    self.tma.append(land)
                    self.q_readers[(a, t)] = nt
                else:
                    self.q_full[qb][t].arrive(tx=0)
            for j in range(max(n0, n1)):
                s = G % ST
                if G >= ST:
                    yield from self.wait(self.kv_empty[s], G // ST - 1)
                    old = G - ST
                    if self.stage_readers.get(old, 0):
                        raise HazardError(f"ring stage {s} reloaded while tile {old} has readers")
                # readers of this tile: an S per Q tile that uses it, a P V per Q tile that uses it
                self.stage_readers[G] = 2 * ((j < n0) + (j < n1))
                self.k_full[s].arrive(tx=1)
                self.v_full[s].arrive(tx=1)

                def land_k(s=s, G=G):
                    self.stage_tile[s] = G
                    self.k_full[s].complete_tx(1)

                def land_v(s=s):
                    self.v_full[s].complete_tx(1)
                self.tma += [land_k, land_v]
                G += 1
                yield

    def s_issuer(self):
        g = Gb = 0
        pend = [None] * SB
        for a, (n0, n1) in enumerate(self.items):
            qb = a & 1
            for t in range(2):
                yield from self.wait(self.q_full[qb][t], a >> 1)
            for jj in range(n0 + n1):
                t, j = tile_of(n0, n1, jj)
                Gt = Gb + j
                s, b = Gt % ST, g % SB
                yield from self.wait(self.k_full[s], Gt // ST)
                if g >= SB:
                    if self.plant != "s_issuer_no_pv_wait":
                        yield from self.wait(self.pv_done[b], g // SB - 1)
                    st, last = pend[b]
                    if last:
                        self.kv_empty[st].arrive()

                def s_mma(g=g, b=b, s=s, Gt=Gt, a=a, t=t, qb=qb):
                    if self.stage_tile[s] != Gt:
                        raise HazardError(f"S({g}) reads stage {s} before tile {Gt} landed")
                    if self.q_tile.get((qb, t)) != a:
                        raise HazardError(f"S({g}) reads Q buffer {qb},{t} before item {a} landed")
                    old = self.sbuf[b]
                    if old is not None and old[0] == "P" and old[1] not in self.pv_read:
                        raise HazardError(f"S({g}) overwrites P({old[1]}) before its P V executed")
                    self.sbuf[b] = ("S", g)
                    self.s_exec.add(g)
                    self.stage_readers[Gt] -= 1
                    self.q_readers[(a, t)] -= 1
                self.issue("S", s_mma)
                self.commit("S", self.s_full[t][b])
                pend[b] = (s, jj == last_job(n0, n1, j))
                g += 1
                yield
            Gb += max(n0, n1)

    def issue_pv(self, who, t, g, b, s, Gt, first, kk, a):
        self.o_pv_pending[t] += 1

        def pv(t=t, g=g, b=b, s=s, Gt=Gt, first=first, a=a):
            if self.sbuf[b] != ("P", g):
                raise HazardError(f"P V({g}) reads buffer {b} holding {self.sbuf[b]}")
            if self.stage_tile[s] != Gt:
                raise HazardError(f"P V({g}) reads stage {s} before tile {Gt} landed")
            if first:
                if not self.o_read[t]:
                    raise HazardError(f"first P V of item {a} overwrites O_{t} before it was read")
                self.o_item[t] = a
                self.o_read[t] = False
            self.pv_read.add(g)
            self.stage_readers[Gt] -= 1
            self.o_pv_pending[t] -= 1
        self.issue(who, pv)
        self.commit(who, self.o_done[t][kk & 1])
        if self.plant == "pv_done_first":
            self.queues[who].insert(len(self.queues[who]) - 1, ("commit", self.pv_done[b]))
        else:
            self.commit(who, self.pv_done[b])

    def softmax(self, t):
        kk = 0
        uses = [0] * SB
        g0 = Gb = 0
        for a, (n0, n1) in enumerate(self.items):
            nt = n1 if t else n0
            qb = a & 1
            for j in range(nt):
                g = g0 + job(n0, n1, t, j)
                b = g % SB
                yield from self.wait(self.s_full[t][b], uses[b])
                uses[b] += 1
                if self.sbuf[b] != ("S", g) or g not in self.s_exec:
                    raise HazardError(f"softmax {t} reads S({g}) but buffer {b} holds {self.sbuf[b]}")
                self.sbuf[b] = ("P", g)
                if j > 0 and self.rng.random() < 0.3:  # rescale O_t
                    if self.plant != "no_rescale_wait":
                        yield from self.wait(self.o_done[t][(kk - 1) & 1], (kk - 1) >> 1)
                    if self.o_pv_pending[t]:
                        raise HazardError(f"softmax {t} rescales O while a P V into it is pending")
                Gt = Gb + j
                s = Gt % ST
                if self.pv_by_wg:
                    yield from self.wait(self.v_full[s], Gt // ST)
                    self.issue_pv(f"WG{t}", t, g, b, s, Gt, j == 0, kk, a)
                else:
                    self.p_full[b].arrive()
                kk += 1
                yield
            if nt > 0:
                if kk >= 2 and self.plant != "single_epilogue_wait":
                    yield from self.wait(self.o_done[t][(kk - 2) & 1], (kk - 2) >> 1)
                yield from self.wait(self.o_done[t][(kk - 1) & 1], (kk - 1) >> 1)
                if self.o_pv_pending[t] or self.o_item[t] != a:
                    raise HazardError(f"epilogue of item {a} tile {t} reads O before its P V executed")
                if self.q_readers.get((a, t), 0):
                    raise HazardError(f"item {a} tile {t} stages O over Q while S still reads it")
                self.o_read[t] = True
                if not self.pv_by_wg:
                    self.o_free[t].arrive()
                self.o_staged[qb][t].arrive()
                yield
            g0 += n0 + n1
            Gb += max(n0, n1)

    def pv_warp(self):
        g = Gb = 0
        kk = [0, 0]
        items_t = [0, 0]
        for a, (n0, n1) in enumerate(self.items):
            for jj in range(n0 + n1):
                t, j = tile_of(n0, n1, jj)
                b = g % SB
                if j == 0 and items_t[t] > 0:
                    yield from self.wait(self.o_free[t], items_t[t] - 1)
                Gt = Gb + j
                s = Gt % ST
                yield from self.wait(self.p_full[b], g // SB)
                yield from self.wait(self.v_full[s], Gt // ST)
                self.issue_pv("PV", t, g, b, s, Gt, j == 0, kk[t], a)
                kk[t] += 1
                g += 1
                yield
            items_t[0] += n0 > 0
            items_t[1] += n1 > 0
            Gb += max(n0, n1)

    def store(self):
        staged = [[0, 0], [0, 0]]
        for a, (n0, n1) in enumerate(self.items):
            qb = a & 1
            for t in range(2):
                nt = n1 if t else n0
                if nt > 0:
                    if self.plant != "store_no_wait":
                        yield from self.wait(self.o_staged[qb][t], staged[qb][t])
                    staged[qb][t] += 1
                    self.q_store_busy.add((qb, t))
                    yield  # the store reads the staging tile
                    self.q_store_busy.discard((qb, t))
                self.q_empty[qb][t].arrive()

    def run(self, max_steps=200000):
        roles = [self.loader(), self.s_issuer(), self.softmax(0), self.softmax(1), self.store()]
        if not self.pv_by_wg:
            roles.append(self.pv_warp())
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
                    r = self.rng.choice(live)
                    try:
                        next(r)
                    except StopIteration:
                        live.remove(r)
                    progressed = True
                    break
            if not live and not any(self.queues.values()) and not self.tma:
                return
            if not progressed:
                break
        raise HazardError("no progress: deadlock or runaway schedule")


def item_lists(rng, n):
    out = []
    for _ in range(n):
        items = []
        for _ in range(rng.randint(1, 5)):
            kind = rng.choice(["full", "causal", "tail"])
            n0 = rng.randint(1, 6)
            items.append((n0, n0) if kind == "full" else (n0, n0 + 1) if kind == "causal" else (n0, 0))
        out.append(items)
    return out


@pytest.mark.parametrize("pv_by_wg", [True, False])
def test_persistent_protocol_random_schedules(pv_by_wg):
    rng = random.Random(61 + pv_by_wg)
    for items in item_lists(rng, 120):
        for tc_weight in (1, 3, 12):  # a slow, medium and fast tensor core
            Model(items, pv_by_wg, random.Random(rng.random()), tc_weight=tc_weight).run()


@pytest.mark.parametrize("pv_by_wg", [True, False])
def test_persistent_protocol_headline_items(pv_by_wg):
    """The item lists one CTA gets at the headline size: seven non-causal items of 32 key
    tiles, and a causal mix of long and short items (n0 = 2 ct + 1, n1 = 2 ct + 2)."""
    rng = random.Random(7)
    Model([(32, 32)] * 7, pv_by_wg, rng).run(max_steps=10 ** 6)
    Model([(2 * c + 1, 2 * c + 2) for c in (15, 11, 11, 6, 6, 1, 1)], pv_by_wg, rng).run(max_steps=10 ** 6)


@pytest.mark.parametrize("plant", ["no_rescale_wait", "single_epilogue_wait", "store_no_wait",
                                   "s_issuer_no_pv_wait", "pv_done_first"])
def test_model_catches_planted_protocol_errors(plant):
    """Each planted mistake (a wait left out of one role) is caught as a hazard or an
    inexact parity wait on some schedule."""
    rng = random.Random(5)
    caught = 0
    for items in item_lists(rng, 100):
        for tc_weight in (1, 3):
            try:
                Model(items, True, random.Random(rng.random()), plant=plant, tc_weight=tc_weight).run()
            except HazardError:
                caught += 1
    assert caught > 0
