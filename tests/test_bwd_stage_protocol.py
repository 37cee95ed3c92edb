"""The mbarrier protocol of the backward kernels' streamed side, modelled on the CPU.

Four agents run their programs against phase-counting barriers, one step at a time in
random order: the TMA warp fills stage g % 4 with stream half g (g = 2 t + u: tile t,
half u) after the MMAs of half g - 4 released it; the MMA warp issues the scores of a half
once it has landed, then, per tile and half, waits for the elementwise warpgroup's P and
dS, issues the half's products and releases its stage; the two elementwise warpgroups of
half u (one per 32 columns of it) each wait for the half's statistics and scores and hand
back their part of P and dS: the half's barrier completes when both have. Every schedule must finish, and
every wait must see the phase it means (try_wait.parity succeeds as soon as the phase of
that parity is the latest completed one, so a wait one fill behind would pass silently).
"""
import random

import pytest

STAGES = 4


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.completed = count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def ready(self, parity):
        return (self.completed & 1) != parity


def run(n_tiles, seed):
    rnd = random.Random(seed)
    st_full = [Bar(1) for _ in range(STAGES)]
    st_empty = [Bar(1) for _ in range(STAGES)]
    s_full, p_full = [Bar(1), Bar(1)], [Bar(256), Bar(256)]
    holds = [None] * STAGES

    def tma():
        for g in range(2 * n_tiles):
            h = g % STAGES
            if g >= STAGES:
                while not st_empty[h].ready(((g - STAGES) // STAGES) & 1):
                    yield
                assert st_empty[h].completed == (g - STAGES) // STAGES + 1
            holds[h] = g
            st_full[h].arrive()
            yield

    def mma():
        def scores(g, u):
            h = g % STAGES
            while not st_full[h].ready((g // STAGES) & 1):
                yield
            assert holds[h] == g
            s_full[u].arrive()
        if n_tiles > 0:
            yield from scores(0, 0)
            yield from scores(1, 1)
        for t in range(n_tiles):
            for u in range(2):
                g = 2 * t + u
                while not p_full[u].ready(t & 1):
                    yield
                assert holds[g % STAGES] == g
                st_empty[g % STAGES].arrive()
                if t + 1 < n_tiles:
                    yield from scores(g + 2, u)
                yield

    def warpgroup(u, sub):
        for t in range(n_tiles):
            g = 2 * t + u
            while not st_full[g % STAGES].ready((g // STAGES) & 1):
                yield
            assert holds[g % STAGES] == g
            while not s_full[u].ready(t & 1):
                yield
            assert s_full[u].completed == t + 1
            for _ in range(128):
                p_full[u].arrive()
            yield

    agents = {"tma": tma(), "mma": mma(), "wg00": warpgroup(0, 0), "wg01": warpgroup(0, 1),
              "wg10": warpgroup(1, 0), "wg11": warpgroup(1, 1)}
    for _ in range(200000):
        if not agents:
            return
        name = rnd.choice(sorted(agents))
        try:
            next(agents[name])
        except StopIteration:
            del agents[name]
    raise AssertionError(f"no progress with {n_tiles} tiles: {sorted(agents)} still waiting")


@pytest.mark.parametrize("n_tiles", list(range(0, 10)) + [31, 32])
def test_every_schedule_finishes_on_its_own_phases(n_tiles):
    for seed in range(25):
        run(n_tiles, seed)
