"""A discrete-event model of the tensor-core kernel's barrier protocol (CPU only).

One block of the persistent tensor-core kernel (weight_quantized_gemm_gb300/csrc/prefill_kernel.cuh)
is modelled as its roles -- the activation producer, the weight producer, the MMA issuer, the
dequant / epilogue warps (two agents, one per column half of the tile; thread 64 in the first)
and the store warp, which stores each 32-row slab as soon as its half has staged it -- exchanging
arrivals on mbarriers with the hardware's phase-parity semantics: a wait for parity P passes as
soon as the barrier's current phase has the other parity, which is only correct when the waiter
is neither two phases behind nor waiting two phases ahead. Copies (TMA), MMA completion and store
reads land after random delays. Each tile's ring positions are its stages, then (persistent form)
its staging positions: kSlots contiguous ring slots where the output tile is staged, after skipped
slots when the run would wrap, released by the store warp once the tile's store has read them.

The model checks, for every configuration the sweep visits, that the block finishes (no
deadlock) and that no slot is refilled, re-dequantized or staged into before its previous use has
ended. It is the protocol the kernel implements, restated; it does not run the kernel.
"""
import random

import pytest


SLABS_PER_HALF = 4   # 32-row slabs per column half of a 256-row tile


class Bar:
    """An mbarrier: `count` arrivals and the announced transaction bytes complete a phase."""

    def __init__(self, count):
        self.count, self.pending, self.tx, self.phase = count, count, 0, 0

    def arrive(self, n=1, tx=0):
        self.pending -= n
        self.tx += tx
        self._check()

    def complete_tx(self, b):
        self.tx -= b
        self._check()

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):   # mbarrier.try_wait.parity
        return (self.phase & 1) != parity


def run_block(S, k_slots, nks, tiles, residual, pre_stages=0, seed=0, delay=4):
    """One block over `tiles` tiles of `nks` stages on a ring of S slots whose output tile takes
    k_slots slots. pre_stages: how many of the next tile's stages the dequant warps may handle
    before a tile's epilogue (bounded by the slots the staging leaves free). Returns
    (finished, why)."""
    rnd = random.Random(seed)
    full_x = [Bar(1) for _ in range(S)]
    full_a = [Bar(2) for _ in range(S)]   # one arrival per epilogue agent (the kernel: per dequant warp)
    empty = [Bar(1) for _ in range(S)]
    acc_full, staged, taken, res_full, wt_staged = (Bar(1) for _ in range(5))
    acc_empty = Bar(2)
    slabs = [Bar(1) for _ in range(2 * SLABS_PER_HALF)]   # one arrival: the half's agent
    half_done = Bar(2)   # both halves finished the tile's epilogue (the block's named barrier)
    events = []
    clock = [0]
    ended, landed, dequantized = set(), {}, set()

    def later(fn):
        events.append((clock[0] + rnd.randint(1, delay), fn))

    def staging_of(g_end):   # (first staging slot, positions taken after the tile's stages)
        a = g_end % S
        return (0, S - a + k_slots) if a + k_slots > S else (a, k_slots)

    def wait(bar, parity):
        while not bar.done(parity):
            yield "blocked"

    def land(bar, g):
        def fn():
            landed[g] = landed.get(g, 0) + 1
            bar.complete_tx(1)
        return fn

    def producer(act):
        g = s = ph = 0
        for tj in range(tiles):
            _, staging = staging_of(g + nks)
            n = nks + staging
            for i in range(n):
                if not act and i == nks and tj > 0:
                    yield from wait(taken, (tj - 1) & 1)
                if g == 0 and act:   # the first stage leaves before the block barrier
                    full_x[0].arrive(1, 2)
                    later(land(full_x[0], 0))
                    later(land(full_x[0], 0))
                elif g > 0:
                    yield from wait(empty[s], ph ^ 1)
                    if g >= S:
                        assert g - S in ended, f"slot {s} refilled before position {g - S} ended"
                    if i < nks:
                        if act:
                            full_x[s].arrive(1, 2)   # expect_tx for both producers' copies
                        later(land(full_x[s], g))
                    elif act:
                        full_x[s].arrive()
                g += 1
                s += 1
                if s == S:
                    s, ph = 0, ph ^ 1
                if act and residual and i == n - 1:
                    if tj > 0:
                        yield from wait(taken, (tj - 1) & 1)
                    res_full.arrive(1, 1)
                    later(lambda: res_full.complete_tx(1))
                yield "step"
            if not act:
                wt_staged.arrive()

    def mma():
        g = s = ph = 0
        for tj in range(tiles):
            _, skip = staging_of(g + nks)
            if tj > 0:
                yield from wait(acc_empty, (tj - 1) & 1)
            ready = False
            for i in range(nks):
                if not ready:
                    yield from wait(full_a[s], ph)
                s2, ph2 = (0, ph ^ 1) if s + 1 == S else (s + 1, ph)
                ready = i + 1 < nks and full_a[s2].done(ph2)
                assert landed.get(g) == 2 and g in dequantized, f"MMA of position {g} before its data"
                later(lambda e=empty[s], gg=g: (ended.add(gg), e.arrive()))
                g += 1
                s += 1
                if s == S:
                    s, ph = 0, ph ^ 1
                yield "step"
            later(lambda: acc_full.arrive())
            for _ in range(skip):
                g += 1
                s += 1
                if s == S:
                    s, ph = 0, ph ^ 1

    def epilogue_warps(half):
        g = s = ph = 0
        pre = 0
        g_tile = 0

        def stage(gpos, sl, p):
            yield from wait(full_x[sl], p)
            assert landed.get(gpos) == 2, f"dequantization of position {gpos} before its data"
            yield from wait(empty[sl], p ^ 1)
            assert gpos < S or gpos - S in ended, f"TMEM stage of position {gpos} reused early"
            dequantized.add(gpos)
            full_a[sl].arrive()

        for tj in range(tiles):
            _, nstg = staging_of(g_tile + nks)
            for _ in range(pre, nks):
                yield from stage(g, s, ph)
                g += 1
                s += 1
                if s == S:
                    s, ph = 0, ph ^ 1
                yield "step"
            for _ in range(nstg):
                yield from wait(full_x[s], ph)
                yield from wait(empty[s], ph ^ 1)
                assert g < S or g - S in ended, f"staging slot of position {g} still in use"
                full_a[s].arrive()
                g += 1
                s += 1
                if s == S:
                    s, ph = 0, ph ^ 1
            g_tile = g
            pre = 0
            if tj + 1 < tiles:
                for _ in range(min(nks, S - nstg, pre_stages)):
                    yield from stage(g, s, ph)
                    g += 1
                    s += 1
                    if s == S:
                        s, ph = 0, ph ^ 1
                    pre += 1
            yield from wait(acc_full, tj & 1)
            if residual:
                yield from wait(res_full, tj & 1)
            if tj > 0:
                yield from wait(taken, (tj - 1) & 1)   # before this tile's first slab
            for k in range(SLABS_PER_HALF):
                slabs[half * SLABS_PER_HALF + k].arrive()
                yield "step"
            acc_empty.arrive()
            half_done.arrive()
            yield from wait(half_done, tj & 1)   # the epilogue warps' barrier
            if half == 0:
                staged.arrive()   # thread 64 (the taken wait above already covered it)
            yield "step"

    def store_warp():
        g = 0
        for tj in range(tiles):
            g_end = g + nks
            _, staging = staging_of(g_end)
            g = g_end + staging
            for kk in range(SLABS_PER_HALF):
                for hh in range(2):
                    yield from wait(slabs[hh * SLABS_PER_HALF + kk], tj & 1)
            yield from wait(staged, tj & 1)
            yield from wait(wt_staged, tj & 1)
            taken.arrive()
            for k in range(g_end, g):   # after the store has read the staged tile
                later(lambda e=empty[k % S], kk=k: (ended.add(kk), e.arrive()))
            yield "step"

    roles = {"act": producer(True), "wt": producer(False), "mma": mma(),
             "epilogue0": epilogue_warps(0), "epilogue1": epilogue_warps(1), "store": store_warp()}
    alive, idle = set(roles), 0
    while alive:
        clock[0] += 1
        due = [e for e in events if e[0] <= clock[0]]
        for e in due:
            events.remove(e)
            e[1]()
        progressed = bool(due)
        for name in list(alive):
            for _ in range(rnd.randint(1, 3)):
                try:
                    state = next(roles[name])
                except AssertionError as err:
                    return False, f"{name}: {err}"
                except StopIteration:
                    alive.discard(name)
                    progressed = True
                    break
                if state == "blocked":
                    break
                progressed = True
        idle = 0 if (progressed or events) else idle + 1
        if idle > 50:
            return False, f"deadlock, blocked: {sorted(alive)}"
    return True, ""


CASES = [(S, k, nks, tiles)
         for S in (2, 3, 4, 6, 8)
         for k in range(1, S + 1) if 2 * k - 1 <= S
         for nks in (1, 2, 3, 5, 32)
         for tiles in (1, 3, 6)]


@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("pre_stages", [0, 2])
def test_protocol_finishes_and_never_reuses_a_slot_early(residual, pre_stages):
    bad = []
    for S, k, nks, tiles in CASES:
        for seed in range(6):
            ok, why = run_block(S, k, nks, tiles, residual, pre_stages, seed)
            if not ok:
                bad.append(((S, k, nks, tiles, seed), why))
    assert not bad, bad[:5]


def test_model_catches_a_producer_that_skips_staging_positions():
    """The first persistent form: the weight producer passed the staging positions without
    waiting and the store warp did not wait for it; the model must find that fault."""
    import inspect
    src = inspect.getsource(run_block)
    src = src.replace("                if not act and i == nks and tj > 0:\n"
                      "                    yield from wait(taken, (tj - 1) & 1)\n", "")
    src = src.replace("                elif g > 0:\n", "                elif g > 0 and (i < nks or act):\n")
    src = src.replace("            yield from wait(wt_staged, tj & 1)\n", "")
    ns = dict(globals())
    exec(src, ns)
    failures = sum(not ns["run_block"](3, 2, 56, 3, False, 0, seed)[0] for seed in range(8))
    assert failures > 0


def test_model_catches_too_many_early_stages():
    """Dequantizing one more of the next tile's stages before the epilogue than the ring holds
    besides the staging slots waits on a slot that only this epilogue frees."""
    import inspect
    src = inspect.getsource(run_block).replace("min(nks, S - nstg, pre_stages)", "min(nks, S - nstg + 1, pre_stages)")
    ns = dict(globals())
    exec(src, ns)
    assert not ns["run_block"](3, 1, 32, 3, False, 3, 0)[0]
