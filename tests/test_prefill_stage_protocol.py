"""The mbarrier protocol of the 256-row prefill kernel, modelled on the CPU.

A work item is two 128-row query tiles A and B over the n key blocks of the item. Agents,
each a program over phase-counting barriers, run one step at a time in random order:
  * the TMA warp loads Q_A and Q_B of an item once the last S MMA of each tile released
    it, then K(j), V(j) for every block into a ring of slots freed by the MMA warp;
  * the MMA warp issues S_q(j) = Q_q K(j)^T and O_q += P_q(j) V(j) in the kernel's order
    (S of the first block for both tiles; then per block: P.V of A, S of A's next block,
    P.V of B, S of B's next block), commits the barriers the kernel commits, and releases
    ring slots;
  * softmax warpgroup q turns each S_q into P_q, then, after the item's last P.V, reads
    O_q (the epilogue) and hands the buffer back.
The tensor pipe executes issued MMAs and commits in issue order at random later times
(a commit arrives once everything issued before it has executed). Every schedule must
finish, and every operand an MMA or the softmax reads must hold what it means: the
right K/V block in the ring slot, the right item's Q, P of the right block in the S
buffer, and an O buffer whose previous item the epilogue has already read.
(The model also takes per-tile spans of blocks, which the kernel does not use: with
each tile over the whole item it is the kernel's protocol.)
"""
import random

import pytest

NSLOT = 5


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


def spans(n, rnd):
    """Random per-tile spans [f, l] whose union is 0..n-1."""
    kind = rnd.randrange(4)
    if kind == 0 or n == 1:
        return [(0, n - 1), (0, n - 1)]
    if kind == 1:  # causal: A stops one block early
        return [(0, n - 2), (0, n - 1)]
    if kind == 2:  # window: A stops early, B starts late, overlapping
        a = rnd.randrange(0, n - 1)
        b = rnd.randrange(1, a + 2)
        return [(0, a), (b, n - 1)]
    a = rnd.randrange(0, n)  # one tile spans everything, the other a random piece
    b = rnd.randrange(a, n)
    return [(0, n - 1), (a, b)] if rnd.random() < 0.5 else [(a, b), (0, n - 1)]


def run(items, seed, release_only_with_b=False, s_before_pv=False):
    """Two mistakes can be planted in the model: release_only_with_b releases K(j+1) only
    when tile B computes S(j+1); s_before_pv issues tile A's S(j+1) before its P.V(j)."""
    rnd = random.Random(seed)
    full = [Bar(1) for _ in range(NSLOT)]
    empty = [Bar(1) for _ in range(NSLOT)]
    q_full, q_empty = [Bar(1), Bar(1)], [Bar(1), Bar(1)]
    s_full, p_full = [Bar(1), Bar(1)], [Bar(128), Bar(128)]
    pv_done, o_empty = [Bar(1), Bar(1)], [Bar(128), Bar(128)]
    ring = [None] * NSLOT          # what each slot holds: (item, block, "K"/"V")
    qbuf = [None, None]            # item whose Q tile each buffer holds
    sbuf = [None, None]            # ("S" or "P", item, block) in each tile's TMEM columns
    obuf = [None, None]            # item whose partial output each O buffer holds
    o_read = [-1, -1]              # last item whose O the epilogue has read
    pipe = []                      # issued, not yet executed tensor-pipe operations

    def issue(op):
        pipe.append(op)

    def execute_one():
        op = pipe.pop(0)
        kind = op[0]
        if kind == "commit":
            op[1].arrive()
        elif kind == "S":
            _, q, it, j, slot = op
            assert qbuf[q] == it, "S read a Q tile of another item"
            assert ring[slot] == (it, j, "K"), "S read the wrong K block"
            assert sbuf[q] is None or sbuf[q][0] == "P" and (sbuf[q][1], sbuf[q][2]) in pv_seen[q], \
                "S overwrote a P that its P.V had not read"
            sbuf[q] = ("S", it, j)
        elif kind == "PV":
            _, q, it, j, slot, acc = op
            assert sbuf[q] == ("P", it, j), "P.V read the wrong P"
            assert ring[slot] == (it, j, "V"), "P.V read the wrong V block"
            if acc:
                assert obuf[q] == it
            else:
                assert o_read[q] == it - 1 or obuf[q] is None, "P.V overwrote an unread O"
                obuf[q] = it
            pv_seen[q].add((it, j))

    pv_seen = [set(), set()]

    def tma():
        pos = 0
        for it, (n, sp) in enumerate(items):
            for q in range(2):
                if it > 0:
                    while not q_empty[q].ready((it - 1) & 1):
                        yield
                qbuf[q] = it
                q_full[q].arrive()
                yield
            for s in range(2 * n):
                slot, use = pos % NSLOT, pos // NSLOT
                while not empty[slot].ready((use & 1) ^ 1):
                    yield
                ring[slot] = (it, s // 2, "V" if s & 1 else "K")
                full[slot].arrive()
                pos += 1
                yield

    def mma():
        pos = 0
        tc = [0, 0]
        for it, (n, sp) in enumerate(items):
            f = [sp[0][0], sp[1][0]]
            l = [sp[0][1], sp[1][1]]
            slot = pos % NSLOT
            while not full[slot].ready((pos // NSLOT) & 1):
                yield
            for q in range(2):
                while not q_full[q].ready(it & 1):
                    yield
                if f[q] == 0:
                    issue(("S", q, it, 0, slot))
                    issue(("commit", s_full[q]))
                    if l[q] == 0:
                        issue(("commit", q_empty[q]))
            issue(("commit", empty[slot]))
            pos += 1
            for j in range(n):
                vslot, kslot = pos % NSLOT, (pos + 1) % NSLOT
                more = j + 1 < n
                while not full[vslot].ready((pos // NSLOT) & 1):
                    yield

                def pv_step(q):
                    while not p_full[q].ready(tc[q] & 1):
                        yield
                    if j == f[q] and it > 0:
                        while not o_empty[q].ready((it - 1) & 1):
                            yield
                    issue(("PV", q, it, j, vslot, j > f[q]))
                    if j == l[q]:
                        issue(("commit", pv_done[q]))
                    tc[q] += 1

                def s_step(q):
                    issue(("S", q, it, j + 1, kslot))
                    issue(("commit", s_full[q]))
                    if j + 1 == l[q]:
                        issue(("commit", q_empty[q]))

                if s_before_pv and more:
                    while not full[kslot].ready(((pos + 1) // NSLOT) & 1):
                        yield
                    if f[0] <= j + 1 <= l[0]:
                        s_step(0)
                if f[0] <= j <= l[0]:
                    yield from pv_step(0)
                if more and not s_before_pv:  # K(j+1) landed, whichever tile uses it
                    while not full[kslot].ready(((pos + 1) // NSLOT) & 1):
                        yield
                if more and f[0] <= j + 1 <= l[0] and not s_before_pv:
                    s_step(0)
                if f[1] <= j <= l[1]:
                    yield from pv_step(1)
                issue(("commit", empty[vslot]))
                if more:
                    if f[1] <= j + 1 <= l[1]:
                        s_step(1)
                    if not (release_only_with_b and not f[1] <= j + 1 <= l[1]):
                        issue(("commit", empty[kslot]))
                yield
                pos += 2 if j + 1 < n else 1

    def softmax(q):
        tc = 0
        for it, (n, sp) in enumerate(items):
            f, l = sp[q]
            for j in range(f, l + 1):
                while not s_full[q].ready(tc & 1):
                    yield
                assert sbuf[q] == ("S", it, j), f"softmax {q} read {sbuf[q]}, wanted S {it},{j}"
                sbuf[q] = ("P", it, j)
                for _ in range(128):
                    p_full[q].arrive()
                tc += 1
                yield
            while not pv_done[q].ready(it & 1):
                yield
            assert obuf[q] == it and all((it, j) in pv_seen[q] for j in range(f, l + 1))
            o_read[q] = it
            for _ in range(128):
                o_empty[q].arrive()
            yield

    agents = {"tma": tma(), "mma": mma(), "sm0": softmax(0), "sm1": softmax(1)}
    for _ in range(400000):
        if not agents and not pipe:
            return
        choices = sorted(agents) + (["pipe"] if pipe else [])
        name = rnd.choice(choices)
        if name == "pipe":
            execute_one()
            continue
        try:
            next(agents[name])
        except StopIteration:
            del agents[name]
    raise AssertionError(f"no progress: {sorted(agents)} still waiting, {len(pipe)} ops queued")


@pytest.mark.parametrize("seed", range(40))
def test_every_schedule_finishes_with_the_right_operands(seed):
    """The kernel's protocol: both tiles over every block of every item."""
    rnd = random.Random(1000 + seed)
    items = []
    for _ in range(rnd.randrange(1, 7)):
        n = rnd.randrange(1, 9)
        items.append((n, [(0, n - 1), (0, n - 1)]))
    for s in range(5):
        run(items, seed * 10 + s)


@pytest.mark.parametrize("seed", range(10))
def test_the_protocol_also_holds_for_per_tile_spans(seed):
    rnd = random.Random(2000 + seed)
    items = []
    for _ in range(rnd.randrange(1, 7)):
        n = rnd.randrange(1, 9)
        items.append((n, spans(n, rnd)))
    for s in range(3):
        run(items, seed * 10 + s)


def test_planted_mistakes_are_caught():
    """Scores issued over a P that its P.V has not read yet break an operand check; a K
    slot released only when tile B computes on it stalls the ring."""
    items = [(5, [(0, 4), (0, 4)]), (3, [(0, 2), (0, 2)])]
    run(items, 1)
    caught = 0
    for seed in range(20):
        try:
            run(items, seed, s_before_pv=True)
        except AssertionError as e:
            assert "P.V had not read" in str(e) or "wrong" in str(e)
            caught += 1
    assert caught > 0
    spanned = [(5, [(0, 4), (0, 1)]), (3, [(0, 2), (0, 2)])]
    with pytest.raises(AssertionError, match="no progress"):
        run(spanned, 1, release_only_with_b=True)
