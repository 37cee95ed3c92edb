"""The mbarrier protocol of the backward's dK/dV kernel, modelled on the CPU.

Agents run their programs against phase-counting barriers, one step at a time in random
order:
  * the TMA warp fills stage g % 4 with stream half g (g = 2 t + u: tile t, half u) after
    the MMAs of half g - 4 released it;
  * the MMA warp issues S^T and dP^T of a half once it has landed; then, per tile and half,
    waits for the elementwise warps' P^T (TMEM) and dS^T (shared memory), issues dV, dK,
    releases the stage, issues dQ^T over the half's dP^T columns, then S^T of the half's
    next tile and, once the elementwise warps have read dQ^T, its dP^T;
  * the two elementwise warpgroups of half u (one per 32 columns of it) each wait for the
    half's statistics and scores, write their part of P^T and dS^T and arrive, then wait
    for dQ^T, read it and arrive again.
Issued MMAs and commits go to a tensor pipe that executes them in issue order at random
later times (a commit arrives once everything issued before it has executed). Every
schedule must finish; every wait must see the phase it means; and every operand must hold
what it means when it is read or overwritten: the right stream half in a stage, S^T and
dP^T of the right tile, P^T and dS^T that the products have not yet read are never
overwritten, and dQ^T is read whole before the next dP^T lands on its columns.
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


def run(n_tiles, seed, skip_dq_read_wait=False, early_release=False):
    """Two mistakes can be planted: skip_dq_read_wait issues the next dP^T without waiting
    for the dQ^T readers; early_release commits the stage's release before dK, which still
    reads its Q half. (Writing the next dS^T before the next scores' commit would not be
    one: the dQ^T commit that the elementwise warps wait for already follows dK and dQ^T.)"""
    rnd = random.Random(seed)
    st_full = [Bar(1) for _ in range(STAGES)]
    st_empty = [Bar(1) for _ in range(STAGES)]
    s_full, p_full = [Bar(1), Bar(1)], [Bar(256), Bar(256)]
    dq_full, dq_read = [Bar(1), Bar(1)], [Bar(256), Bar(256)]
    holds = [None] * STAGES
    # TMEM columns of each half, per 32-column part (sub): ("S"|"P"|"dP"|"dQ", tile)
    tm_s = [[None, None], [None, None]]
    tm_dp = [[None, None], [None, None]]
    ds = [[None, None], [None, None]]      # shared-memory dS^T of each half, per part
    dv_done = [-1, -1]                     # last tile whose dV read P^T of half u
    ds_done = [[-1, -1], [-1, -1]]         # last tile whose dK / dQ read dS^T of half u
    dp_read = [[-1, -1], [-1, -1]]         # last tile whose dP^T the part has loaded
    dq_taken = [[-1, -1], [-1, -1]]        # last tile whose dQ^T the part has loaded
    pipe = []

    def execute_one():
        op = pipe.pop(0)
        kind = op[0]
        if kind == "commit":
            op[1].arrive()
            return
        _, u, t, g = op
        if kind in ("S", "dP", "dV", "dK"):
            assert holds[g % STAGES] == g, f"{kind} of half {g} read stage holding {holds[g % STAGES]}"
        if kind == "S":
            for sub in range(2):
                if tm_s[u][sub] is not None and tm_s[u][sub][0] == "P":
                    assert dv_done[u] == tm_s[u][sub][1], "S^T overwrote a P^T that dV had not read"
                tm_s[u][sub] = ("S", t)
        elif kind == "dP":
            for sub in range(2):
                if tm_dp[u][sub] is not None:
                    assert tm_dp[u][sub][0] == "dQ" and dq_taken[u][sub] == tm_dp[u][sub][1], \
                        "dP^T overwrote a dQ^T that was not read"
                tm_dp[u][sub] = ("dP", t)
        elif kind == "dV":
            assert all(tm_s[u][sub] == ("P", t) for sub in range(2)), "dV read the wrong P^T"
            dv_done[u] = t
        elif kind == "dK":
            assert all(ds[u][sub] == ("dS", t) for sub in range(2)), "dK read the wrong dS^T"
            ds_done[u][0] = t
        elif kind == "dQ":
            assert all(ds[u][sub] == ("dS", t) for sub in range(2)), "dQ^T read the wrong dS^T"
            for sub in range(2):
                assert tm_dp[u][sub] == ("dP", t) and dp_read[u][sub] == t, \
                    "dQ^T overwrote a dP^T that was not read"
                tm_dp[u][sub] = ("dQ", t)
            ds_done[u][1] = t

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
        def s_half(g, u):
            h = g % STAGES
            while not st_full[h].ready((g // STAGES) & 1):
                yield
            pipe.append(("S", u, g // 2, g))

        def dp_half(g, u):
            pipe.append(("dP", u, g // 2, g))
            pipe.append(("commit", s_full[u]))

        if n_tiles > 0:
            yield from s_half(0, 0)
            dp_half(0, 0)
            yield from s_half(1, 1)
            dp_half(1, 1)
        for t in range(n_tiles):
            for u in range(2):
                g = 2 * t + u
                while not p_full[u].ready(t & 1):
                    yield
                pipe.append(("dV", u, t, g))
                if early_release:
                    pipe.append(("commit", st_empty[g % STAGES]))
                pipe.append(("dK", u, t, g))
                if not early_release:
                    pipe.append(("commit", st_empty[g % STAGES]))
                pipe.append(("dQ", u, t, g))
                pipe.append(("commit", dq_full[u]))
                if t + 1 < n_tiles:
                    yield from s_half(g + 2, u)
                    if not skip_dq_read_wait:
                        while not dq_read[u].ready(t & 1):
                            yield
                    dp_half(g + 2, u)
                yield
        pipe.append(("commit", None))

    def warpgroup(u, sub):
        for t in range(n_tiles):
            g = 2 * t + u
            while not st_full[g % STAGES].ready((g // STAGES) & 1):
                yield
            assert holds[g % STAGES] == g
            while not s_full[u].ready(t & 1):
                yield
            assert s_full[u].completed == t + 1
            assert tm_s[u][sub] == ("S", t) and tm_dp[u][sub] == ("dP", t), \
                f"scores of tile {t} half {u}: {tm_s[u][sub]}, {tm_dp[u][sub]}"
            assert holds[g % STAGES] == g, "statistics read from a refilled stage"
            dp_read[u][sub] = t
            if ds[u][sub] is not None:
                assert ds_done[u] == [ds[u][sub][1]] * 2, "dS^T overwritten before dK and dQ^T read it"
            ds[u][sub] = ("dS", t)
            tm_s[u][sub] = ("P", t)
            for _ in range(128):
                p_full[u].arrive()
            yield
            while not dq_full[u].ready(t & 1):
                yield
            assert dq_full[u].completed == t + 1
            assert tm_dp[u][sub] == ("dQ", t), f"read {tm_dp[u][sub]} as dQ^T of tile {t}"
            dq_taken[u][sub] = t
            for _ in range(128):
                dq_read[u].arrive()
            yield

    agents = {"tma": tma(), "mma": mma(), "wg00": warpgroup(0, 0), "wg01": warpgroup(0, 1),
              "wg10": warpgroup(1, 0), "wg11": warpgroup(1, 1)}
    for _ in range(400000):
        if not agents and not pipe:
            return
        choices = sorted(agents) + (["pipe"] if pipe else [])
        name = rnd.choice(choices)
        if name == "pipe":
            op = pipe[0]
            if op[0] == "commit" and op[1] is None:
                pipe.pop(0)
            else:
                execute_one()
            continue
        try:
            next(agents[name])
        except StopIteration:
            del agents[name]
    raise AssertionError(f"no progress with {n_tiles} tiles: {sorted(agents)} still waiting, "
                         f"{len(pipe)} ops queued")


@pytest.mark.parametrize("n_tiles", list(range(0, 10)) + [31, 32])
def test_every_schedule_finishes_with_the_right_operands(n_tiles):
    for seed in range(25):
        run(n_tiles, seed)


def test_planted_mistakes_are_caught():
    """A dP^T issued without waiting for the dQ^T readers lands on an unread dQ^T; a stage
    released before dK lets the TMA warp refill the Q half that dK still reads."""
    for kw, what in ((dict(skip_dq_read_wait=True), "dQ^T that was not read"),
                     (dict(early_release=True), "dK of half")):
        caught = 0
        for seed in range(40):
            try:
                run(4, seed, **kw)
            except AssertionError as e:
                assert what in str(e), str(e)
                caught += 1
        assert caught > 0, kw
