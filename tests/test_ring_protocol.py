"""Host-side checks of the fused GEMM kernel's pipeline protocol (no GPU).

The kernel's roles hand work to each other through mbarriers that are waited
for by phase parity: `mbarrier.try_wait.parity P` returns once the barrier's
current phase has the other parity, i.e. once the phase before it completed.
Such a wait is unambiguous only if the waiter has seen the barrier's previous
phase complete: a waiter that is one phase ahead passes at once (it takes the
phase before for its own), one that is two phases behind waits a whole phase
too long.  Two rules of the launch geometry keep every wait unambiguous:

* with two MMA warps taking alternate pipeline stages the ring depth is even, so
  that a slot's previous stage was the same warp's (it waited for that fill);
* there are at least as many accumulator buffers as epilogue groups, so that an
  epilogue group's own previous item, completed, implies that its buffer's
  previous use completed (each MMA warp's operations complete in issue order).

`test_geometry_keeps_the_rules` checks the library's geometry for a grid of
shapes and every forced tile width and copy scheme.  The model below plays the
protocol of the kernel's roles -- producer, scale-layout warp, one or two MMA
warps, epilogue groups -- under random interleavings, with TMA fills landing,
scale copies and MMAs completing and epilogue drains finishing in any order the
barriers allow (MMAs of one warp in issue order).  It checks that every wait
returns on the phase it meant, that no slot, scale-factor region or accumulator
buffer is overwritten while it is read, and that nothing deadlocks: clean with
the geometry's rules, and caught when a rule is broken.
"""
import itertools
import random

import pytest


class _Bar:
    """mbarrier: expected arrivals per phase and the number of completed phases."""

    def __init__(self, count):
        self.count, self.pend, self.c = count, count, 0

    def arrive(self):
        self.pend -= 1
        assert self.pend >= 0
        if self.pend == 0:
            self.c += 1
            self.pend = self.count

    def passes(self, k):
        """try_wait.parity for the completion of phase k (k = -1: the phase before
        the first, which a fresh barrier reports as complete)."""
        return (self.c & 1) != (k & 1)


class _Violation(AssertionError):
    pass


def _check(cond, what):
    if not cond:
        raise _Violation(what)


def _play(seed, ns, mma_warps, acc_bufs, epi_groups, items, stages_per_item, lookahead=False):
    """One random interleaving of the kernel's roles over one CTA's items.

    items[phase] work items of stages_per_item[phase] pipeline stages each; stage
    g of the CTA's sequence uses ring slot g % ns (fill g // ns of that slot); MMA
    warp w issues the stages with g % mma_warps == w into its own accumulator of
    the item's buffer (item index % acc_bufs); every MMA warp waits for the buffer
    and commits once per item; epilogue group e drains the items with index %
    epi_groups == e.  With lookahead, an MMA warp about to issue a stage tests
    (without waiting) whether its next stage's fill and scale factors are there,
    and if so skips those waits at that stage (the kernel's copy look-ahead with
    MMA-warp copies).  Raises _Violation on a wrong-phase wait or test, a data
    hazard or a deadlock."""
    rnd = random.Random(seed)
    seq = []  # (item, first stage of the item, last stage of the item)
    per_item = []
    for phase in range(2):
        for _ in range(items[phase]):
            it = len(per_item)
            per_item.append(stages_per_item[phase])
            for ks in range(stages_per_item[phase]):
                seq.append((it, ks == 0, ks + 1 == stages_per_item[phase]))
    G, n_items = len(seq), len(per_item)
    full = [_Bar(1) for _ in range(ns)]
    sfull = [_Bar(1) for _ in range(ns)]
    sfready = [_Bar(1) for _ in range(ns)]
    empty = [_Bar(1) for _ in range(ns)]
    tfull = [_Bar(mma_warps) for _ in range(acc_bufs)]
    tempty = [_Bar(1) for _ in range(acc_bufs)]  # the epilogue group's threads, as one
    slot_data, slot_sf = [None] * ns, [None] * ns
    readers = [set() for _ in range(ns)]
    buf_item = [None] * acc_bufs       # item whose accumulators the buffer holds
    buf_done = [0] * acc_bufs          # its stages completed so far (all warps)
    buf_drain = [False] * acc_bufs
    events = []
    prod = {"g": 0}
    lay = {"g": 0}
    mma = [{"g": 0, "item": 0, "state": "tempty", "queue": [], "pre": -1} for _ in range(mma_warps)]
    epi = [{"next": e, "busy": False} for e in range(epi_groups)]

    def wait(bar, k, name):
        if not bar.passes(k):
            return False
        _check(bar.c == k + 1, f"{name}: wait for phase {k} returned at {bar.c} completed phases")
        return True

    def producer():
        g = prod["g"]
        if g >= G:
            return False
        s, k = g % ns, g // ns
        if not wait(empty[s], k - 1, "empty"):
            return False
        _check(not readers[s], "slot refilled while its MMAs run")
        events.append(("fill", s, g))
        events.append(("sfill", s, g))
        prod["g"] += 1
        return True

    def layout():
        g = lay["g"]
        if g >= G:
            return False
        s, k = g % ns, g // ns
        if not wait(sfull[s], k, "sfull"):
            return False
        _check(not readers[s], "scale factors overwritten while MMAs read them")
        events.append(("sfcopy", s, g))
        lay["g"] += 1
        return True

    def mma_warp(w):
        st = mma[w]
        it = st["item"]
        if it >= n_items:
            return False
        a, use = it % acc_bufs, it // acc_bufs
        if st["state"] == "tempty":
            if not wait(tempty[a], use - 1, "tempty"):
                return False
            st["state"] = "stages"
            return True
        # this warp's next stage of the item, if any
        while st["g"] < G and seq[st["g"]][0] == it and st["g"] % mma_warps != w:
            st["g"] += 1
        if st["g"] < G and seq[st["g"]][0] == it:
            g = st["g"]
            s, k = g % ns, g // ns
            if st["state"] == "stages" and st["pre"] != g:
                if not wait(full[s], k, "full"):
                    return False
                st["state"] = "sf"
                return True
            if st["pre"] != g and not wait(sfready[s], k, "sfready"):
                return False
            gn = g + mma_warps  # this warp's next stage
            if lookahead and gn < G:
                sn, kn = gn % ns, gn // ns
                if full[sn].passes(kn) and sfready[sn].passes(kn):
                    _check(full[sn].c == kn + 1 and sfready[sn].c == kn + 1,
                           f"look-ahead test passed on phase {full[sn].c - 1} for phase {kn}")
                    st["pre"] = gn
            _check(slot_data[s] == g and slot_sf[s] == g, "MMAs issued on another stage's data")
            _check(not buf_drain[a] and buf_item[a] in (None, "free", it),
                   "accumulator written while the epilogue reads it")
            buf_item[a] = it
            readers[s].add(g)
            st["queue"].append(("mma", s, g, a))
            events.append(("mma", w))
            st["g"] += 1
            st["state"] = "stages"
            return True
        # end of the item: one commit for the buffer (after this warp's MMAs)
        st["queue"].append(("tfull", a))
        events.append(("mma", w))
        st["item"] += 1
        st["state"] = "tempty"
        return True

    def epilogue(e):
        st = epi[e]
        it = st["next"]
        if it >= n_items or st["busy"]:
            return False
        a, use = it % acc_bufs, it // acc_bufs
        if not wait(tfull[a], use, "tfull"):
            return False
        _check(buf_item[a] == it and buf_done[a] == per_item[it], "epilogue read an unfinished item")
        buf_drain[a] = True
        st["busy"] = True
        events.append(("drain", e))
        return True

    def complete(i):
        ev = events.pop(i)
        if ev[0] == "fill":
            slot_data[ev[1]] = ev[2]
            full[ev[1]].arrive()
        elif ev[0] == "sfill":
            sfull[ev[1]].arrive()
        elif ev[0] == "sfcopy":
            slot_sf[ev[1]] = ev[2]
            sfready[ev[1]].arrive()
        elif ev[0] == "mma":  # the warp's oldest outstanding operation
            op = mma[ev[1]]["queue"].pop(0)
            if op[0] == "mma":
                _, s, g, a = op
                readers[s].discard(g)
                buf_done[a] += 1
                empty[s].arrive()
            else:
                tfull[op[1]].arrive()
        else:  # drain
            st = epi[ev[1]]
            a = st["next"] % acc_bufs
            buf_drain[a] = False
            buf_item[a] = "free"
            buf_done[a] = 0
            st["next"] += epi_groups
            st["busy"] = False
            tempty[a].arrive()

    roles = [producer, layout] + [lambda w=w: mma_warp(w) for w in range(mma_warps)] + \
        [lambda e=e: epilogue(e) for e in range(epi_groups)]
    for _ in range(200000):
        acts = [("role", i) for i in range(len(roles))] + [("event", i) for i in range(len(events))]
        rnd.shuffle(acts)
        for kind, i in acts:
            if kind == "event":
                complete(i)
                break
            if roles[i]():
                break
        else:
            finished = (prod["g"] >= G and lay["g"] >= G and all(m["item"] >= n_items for m in mma)
                        and all(e["next"] >= n_items for e in epi) and not events)
            _check(finished, "deadlock")
            return
    raise _Violation("no progress")


def _cases(n, seed0):
    rnd = random.Random(seed0)
    for i in range(n):
        items = [rnd.randint(0, 5), rnd.randint(0, 6)]
        if sum(items) == 0:
            items[1] = 1
        yield seed0 + i, items, [rnd.choice([1, 2, 3, 14]), rnd.choice([1, 2, 4])]


def _violations(n, seed0, **kw):
    bad = 0
    for seed, items, per in _cases(n, seed0):
        try:
            _play(seed, items=items, stages_per_item=per, **kw)
        except _Violation:
            bad += 1
    return bad


@pytest.mark.parametrize("ns,mma_warps,acc_bufs,epi_groups", [
    (5, 1, 4, 2), (3, 1, 3, 3), (3, 1, 3, 2),   # one MMA warp (decode, prefill, dense)
    (4, 2, 4, 2), (2, 2, 2, 2), (6, 2, 3, 2),   # two MMA warps, even ring depth
])
def test_protocol_clean_under_the_geometry_rules(ns, mma_warps, acc_bufs, epi_groups):
    assert _violations(300, 1000, ns=ns, mma_warps=mma_warps, acc_bufs=acc_bufs,
                       epi_groups=epi_groups) == 0


@pytest.mark.parametrize("ns", [4, 6])
def test_lookahead_clean_with_an_even_ring(ns):
    """The MMA warps' look-ahead (scheme 1: each warp copies its next stage's scale
    factors early when that stage has landed) with the geometry's even ring."""
    assert _violations(300, 3000, ns=ns, mma_warps=2, acc_bufs=4, epi_groups=2, lookahead=True) == 0


def test_lookahead_with_an_odd_ring_is_caught():
    """The same test with 3 slots: the slot of a warp's next stage last held the
    other warp's stage, and the non-blocking test can pass on that fill."""
    assert _violations(600, 7000, ns=3, mma_warps=2, acc_bufs=4, epi_groups=2, lookahead=True) > 0


def test_odd_ring_depth_with_two_mma_warps_is_caught():
    """Two MMA warps on alternate stages with 3 slots (the rule broken): an
    interleaving in which a slot's fill lands after later fills makes the other
    warp pass its wait for the slot's next fill on that one.  (Deeper odd rings
    need more fills to land out of order and show it less often: 5 slots about
    one schedule in a thousand of this model's.)"""
    assert _violations(600, 5000, ns=3, mma_warps=2, acc_bufs=4, epi_groups=2) > 0


def test_fewer_buffers_than_groups_is_caught():
    """Two accumulator buffers drained by three epilogue groups (the rule broken)."""
    assert _violations(400, 9000, ns=3, mma_warps=1, acc_bufs=2, epi_groups=3) > 0


def _random_shapes(n, seed):
    """Valid shapes drawn at random: d_model a multiple of 128, d_inter of 64 (the
    widths run as they are and the ones run wider), T, E and topk over their ranges."""
    rnd = random.Random(seed)
    out = []
    for _ in range(n):
        D = 128 * rnd.choice([1, 2, 3, 4, 7, 8, 12, 23, 56, 64])
        I = 64 * rnd.choice([1, 2, 3, 4, 5, 6, 8, 12, 16, 32])
        E = rnd.choice([1, 3, 8, 33, 64, 257, 384, 1024])
        K = rnd.randint(1, min(16, E))
        T = rnd.choice([1, 5, 16, 64, 128, 512, 1024, 4096])
        out.append((T, D, I, E, K))
    return out


SHAPES = [(16, 7168, 256, 257, 9), (128, 7168, 256, 257, 9), (512, 7168, 2048, 33, 9),
          (4096, 7168, 256, 257, 9), (256, 512, 256, 5, 3), (96, 1024, 512, 3, 2),
          (16, 256, 128, 9, 3), (200, 2048, 1024, 4, 3), (8, 128, 128, 1, 1), (64, 1536, 1024, 64, 6),
          (64, 2944, 384, 16, 4), (16, 384, 192, 9, 3)]


def test_geometry_keeps_the_rules():
    """The library's GEMM geometry (moe_mxfp4_get_gemm_config) for every shape
    above, forced tile width and copy scheme keeps the rules the kernel's
    barriers and tensor-memory layout depend on."""
    import mixture_experts_mxfp4_gb300 as moe
    from mixture_experts_mxfp4_gb300 import build

    build.build()
    moe.load_library()
    try:
        for shape, rows, copies in itertools.product(SHAPES + _random_shapes(60, 7), (0, 16, 32, 64, 128),
                                                     range(5)):
            moe.set_tuning(rows, copies)
            c = moe.gemm_config(*shape)
            where = (shape, rows, copies, c.as_dict())
            if rows:
                assert c.tile_rows == rows, where
            assert 1 <= c.num_stages <= 8, where
            assert c.mma_warps in (1, 2) and 2 <= c.epi_groups <= 3 and c.acc_bufs <= 4, where
            assert c.acc_bufs >= c.epi_groups, where
            if c.mma_warps == 2:
                assert c.num_stages % 2 == 0, where
            if c.lookahead:
                assert c.num_stages % c.mma_warps == 0 and c.num_stages > c.mma_warps, where
            if not c.sf_by_layout_warp:
                assert c.mma_warps == 2, where
            if c.wide_sf:
                assert c.sf_by_layout_warp and c.mma_warps == 1, where
            assert c.acc_bufs * c.acc_cols <= c.sf_col0, where
            assert c.sf_col0 + c.num_stages * c.sf_cols <= c.tmem_cols <= 512, where
            assert c.tmem_cols >= 32 and c.tmem_cols & (c.tmem_cols - 1) == 0, where
            assert c.num_stages * c.slot_bytes <= c.smem_bytes <= c.smem_limit, where
            pl = moe.get_plan(*shape)  # widths the kernels run at
            assert pl.d_model_run % c.stage1_k == 0 and pl.d_inter_run % c.stage2_k == 0, where
    finally:
        moe.set_tuning(0, 0)
