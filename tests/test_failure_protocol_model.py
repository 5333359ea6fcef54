"""CPU models of the forward kernels' failure paths (sparse and dense).

Every mbarrier wait in the kernels is bounded: it gives up after a time limit,
or at its next poll once another role has raised the CTA's abort flag, and
the role then leaves by its exit path. Named barriers have no time limit, so
the warps that meet at one must all get there. This model runs the sparse
forward's roles warp by warp (the two softmax warpgroups as four warps each)
with waits that may give up at any moment -- a timeout racing a phase that
completes just after it -- and with the MMA warp stalled (the testing hook),
and requires every run to end, i.e. every warp to reach the kernel's closing
__syncthreads. The control flow from before the epilogue-consensus fix, where
a warp could leave the item loop before warpgroup 0's consensus, must be
caught hanging at the named barrier. The dense forward, whose two softmax
warpgroups each meet at an epilogue consensus for every item, is run the
same way.

CPU only; no kernel code is involved.
"""
import random

import pytest

from tests.protocol_sim import Bar, Deadlock, run

POLL_LIMIT = 400  # polls before a blocked wait runs out of time


class Ctl:
    def __init__(self, rnd, p_giveup, poll_limit):
        self.abort, self.rnd, self.p, self.limit = False, rnd, p_giveup, poll_limit


def bwait(ctl, bar, phase, abort_aware=True):
    """A bounded wait; returns True when the phase with parity phase & 1 is
    reported complete, False when it gives up (and then raises the abort flag)."""
    polls = 0
    while (bar.completed & 1) == (phase & 1):
        polls += 1
        if (abort_aware and ctl.abort) or ctl.rnd.random() < ctl.p or polls > ctl.limit:
            ctl.abort = True
            Bar.changes += 1
            return False
        yield
    return True


class NamedBar:
    """bar.red.and / bar.sync over n warps: no time limit."""

    def __init__(self, n):
        self.n, self.gen, self.count, self.acc, self.result = n, 0, 0, True, {}

    def and_(self, ok):
        g = self.gen
        self.acc = self.acc and ok
        self.count += 1
        Bar.changes += 1
        if self.count == self.n:
            self.result[g], self.gen, self.count, self.acc = self.acc, self.gen + 1, 0, True
        while self.gen == g:
            yield
        return self.result[g]


def sparse_fwd_failure_model(n_items, nch, seed, p_giveup, stall_mma=False, early_break=False,
                             nslot=5, kslots=2, poll_limit=POLL_LIMIT):
    """Runs to the end (or raises Deadlock); returns whether any wait gave up."""
    rnd = random.Random(seed)
    ctl = Ctl(rnd, p_giveup, poll_limit)
    vslots = nslot - kslots
    full = [Bar(1) for _ in range(nslot)]
    empty = [Bar(1) for _ in range(nslot)]
    q_full, q_empty, mma_done = Bar(1), Bar(1), Bar(1)
    s_full, pv_done = [Bar(1), Bar(1)], [Bar(1), Bar(1)]
    p_full = [Bar(4), Bar(4)]       # every warp of a warpgroup arrives
    merge, o1_free = Bar(4), Bar(4)
    nbar = NamedBar(4)              # warpgroup 0's epilogue barrier
    tma, mma, cpa = [], [], []

    def kslot(g):
        return g % kslots

    def vslot(g):
        return kslots + g % vslots

    def k_producer():
        ok, last, q_loads = True, -1, 0
        for r in range(n_items):
            if not ok:
                break

            def load_k(c):
                nonlocal last
                g = r * nch + c
                if g // kslots > 0:
                    res = yield from bwait(ctl, empty[kslot(g)], g // kslots - 1)
                    if not res:
                        return False
                tma.append(full[kslot(g)])
                last = g
                return True
            if r > 0:
                ok = yield from load_k(0)
                if not ok:
                    break
                ok = yield from bwait(ctl, q_empty, r - 1)
                if not ok:
                    break
            tma.append(q_full)
            q_loads += 1
            for c in range(1 if r > 0 else 0, nch):
                ok = yield from load_k(c)
                if not ok:
                    break
        # Closing waits for copies in flight: bounded, not cut short by the abort flag.
        for g in range(max(0, last - kslots + 1), last + 1):
            yield from bwait(ctl, full[kslot(g)], g // kslots, abort_aware=False)
        if q_loads:
            yield from bwait(ctl, q_full, q_loads - 1, abort_aware=False)

    def v_producer():
        ok, issued, signalled = True, 0, 0
        for r in range(n_items):
            for c in range(nch):
                if not ok:
                    break
                g = r * nch + c
                if g // vslots > 0:
                    ok = yield from bwait(ctl, empty[vslot(g)], g // vslots - 1)
                    if not ok:
                        break
                cpa.append([False, vslot(g)])
                issued += 1
                if issued - signalled > 1:
                    while not cpa[signalled][0]:
                        yield
                    full[cpa[signalled][1]].arrive()
                    signalled += 1
        while signalled < issued:
            while not cpa[signalled][0]:
                yield
            full[cpa[signalled][1]].arrive()
            signalled += 1

    def mma_warp():
        ok, p_cnt = not stall_mma, [0, 0]
        for r in range(n_items):
            if not ok:
                break
            ok = yield from bwait(ctl, q_full, r)
            if not ok:
                break
            s_left = [nch]

            def issue_s(c):
                g = r * nch + c
                mma.append(s_full[c & 1])
                mma.append(empty[kslot(g)])
                s_left[0] -= 1
                if s_left[0] == 0:
                    mma.append(q_empty)
            for c in range(min(2, nch)):
                g = r * nch + c
                ok = yield from bwait(ctl, full[kslot(g)], g // kslots)
                if not ok:
                    break
                issue_s(c)
            for c in range(nch if ok else 0):
                w, g = c & 1, r * nch + c
                ok = yield from bwait(ctl, p_full[w], p_cnt[w])
                if not ok:
                    break
                p_cnt[w] += 1
                ok = yield from bwait(ctl, full[vslot(g)], g // vslots)
                if not ok:
                    break
                mma.append(empty[vslot(g)])
                if c + 2 >= nch:
                    mma.append(pv_done[w])
                if c + 2 < nch:
                    ok = yield from bwait(ctl, full[kslot(g + 2)], (g + 2) // kslots)
                    if not ok:
                        break
                    issue_s(c + 2)
        mma.append(mma_done)
        yield from bwait(ctl, mma_done, 0, abort_aware=False)

    def softmax_warp(w, k):  # warp k of warpgroup w
        ok, s_cnt, pv_cnt = True, 0, 0
        my_n = (nch - w + 1) // 2 if nch > w else 0
        for rr in range(n_items):
            if not ok:
                break
            checked = w == 0 or rr == 0
            for _ in range(my_n):
                ok = yield from bwait(ctl, s_full[w], s_cnt)
                if not ok:
                    break
                s_cnt += 1
                if not checked:
                    ok = yield from bwait(ctl, o1_free, rr - 1)
                    if not ok:
                        break
                    checked = True
                p_full[w].arrive((w, k))
            if early_break and not ok:
                break  # the control flow before the fix
            if ok and my_n > 0:
                ok = yield from bwait(ctl, pv_done[w], pv_cnt)
                pv_cnt += 1
            if w == 1:
                if ok and not checked:
                    ok = yield from bwait(ctl, o1_free, rr - 1)
                if not ok:
                    break
                merge.arrive((w, k))
                continue
            if ok:
                ok = yield from bwait(ctl, merge, rr)
            ok = yield from nbar.and_(ok)
            if not ok:
                break
            for _ in range(2):  # the staging tile's two bar.sync of the epilogue
                yield from nbar.and_(True)
            o1_free.arrive((w, k))

    agents = [k_producer(), v_producer(), mma_warp()]
    agents += [softmax_warp(w, k) for w in (0, 1) for k in range(4)]
    run(agents, (tma, mma, cpa), rnd)
    return ctl.abort


@pytest.mark.parametrize("nch", [1, 2, 5])
def test_every_warp_leaves_when_waits_give_up(nch):
    gave_up = sum(sparse_fwd_failure_model(3, nch, seed, p_giveup=0.02) for seed in range(60))
    assert gave_up > 0  # the failure paths were exercised (and every run ended)


@pytest.mark.parametrize("nch", [1, 3])
def test_every_warp_leaves_with_the_mma_warp_stalled(nch):
    for seed in range(20):
        assert sparse_fwd_failure_model(2, nch, seed, p_giveup=0.0, stall_mma=True)


def test_normal_runs_finish_without_giving_up():
    for seed in range(20):
        assert not sparse_fwd_failure_model(3, 5, seed, p_giveup=0.0, poll_limit=10 ** 9)


def test_leaving_before_the_consensus_is_caught():
    hangs = 0
    for seed in range(300):
        try:
            sparse_fwd_failure_model(3, 2, seed, p_giveup=0.02, early_break=True)
        except Deadlock:
            hangs += 1
    assert hangs > 0


def dense_fwd_failure_model(items, seed, p_giveup, stall_mma=False, nslot=4):
    """The dense forward's roles with bounded waits (see the sparse model above):
    the producer, the MMA issuer and two softmax warpgroups of four warps,
    each warpgroup meeting at its own epilogue consensus for every item."""
    rnd = random.Random(seed)
    ctl = Ctl(rnd, p_giveup, POLL_LIMIT)
    kv_full = [Bar(1) for _ in range(nslot)]
    kv_empty = [Bar(1) for _ in range(nslot)]
    q_full, q_empty, mma_done = Bar(1), Bar(1), Bar(1)
    s_full, pv_done = [Bar(1), Bar(1)], [Bar(1), Bar(1)]
    p_full = [Bar(4), Bar(4)]
    nbar = [NamedBar(4), NamedBar(4)]
    tma, mma = [], []

    def producer():
        ok, issued, q_loads = True, 0, 0
        for r, (n0, n1, l0, l1) in enumerate(items):
            if not ok:
                break
            n_pos = 2 * (n1 - l0)

            def load_kv():
                nonlocal issued
                slot, rnd_ = issued % nslot, issued // nslot
                if rnd_ > 0:
                    res = yield from bwait(ctl, kv_empty[slot], rnd_ - 1)
                    if not res:
                        return False
                tma.append(kv_full[slot])
                issued += 1
                return True
            pre = 0 if r == 0 else min(2, n_pos)
            for _ in range(pre):
                ok = yield from load_kv()
                if not ok:
                    break
            if not ok:
                break
            if r > 0:
                ok = yield from bwait(ctl, q_empty, r - 1)
                if not ok:
                    break
            tma.append(q_full)
            q_loads += 1
            for _ in range(pre, n_pos):
                ok = yield from load_kv()
                if not ok:
                    break
        for pos in range(max(0, issued - nslot), issued):
            yield from bwait(ctl, kv_full[pos % nslot], pos // nslot, abort_aware=False)
        if q_loads:
            yield from bwait(ctl, q_full, q_loads - 1, abort_aware=False)

    def mma_warp():
        ok, ring, p_cnt = not stall_mma, 0, [0, 0]
        for r, (n0, n1, l0, l1) in enumerate(items):
            if not ok:
                break
            n_kv, jlo, jb = (n0, n1), (l0, l1), l0
            ok = yield from bwait(ctl, q_full, r)
            if not ok:
                break
            s_left = [(n0 - l0) + (n1 - l1)]

            def issue_s(t):
                mma.append(s_full[t])
                s_left[0] -= 1
                if s_left[0] == 0:
                    mma.append(q_empty)

            def wait_kv(idx):
                q = ring + idx
                res = yield from bwait(ctl, kv_full[q % nslot], q // nslot)
                return res
            ok = yield from wait_kv(0)
            if not ok:
                break
            issue_s(0)
            if jlo[1] == jb:
                issue_s(1)
            mma.append(kv_empty[ring % nslot])
            for j in range(jb, n1):
                v_ready = k_next = False
                for t in range(2):
                    if jlo[t] <= j < n_kv[t]:
                        ok = yield from bwait(ctl, p_full[t], p_cnt[t])
                        if not ok:
                            break
                        p_cnt[t] += 1
                        if not v_ready:
                            ok = yield from wait_kv(2 * (j - jb) + 1)
                            if not ok:
                                break
                            v_ready = True
                        if j + 1 == n_kv[t]:
                            mma.append(pv_done[t])
                    if j + 1 < n_kv[t] and j + 1 >= jlo[t]:
                        if not k_next:
                            ok = yield from wait_kv(2 * (j - jb) + 2)
                            if not ok:
                                break
                            k_next = True
                        issue_s(t)
                if not ok:
                    break
                mma.append(kv_empty[(ring + 2 * (j - jb) + 1) % nslot])
                if k_next:
                    mma.append(kv_empty[(ring + 2 * (j - jb) + 2) % nslot])
            ring += 2 * (n1 - jb)
        mma.append(mma_done)
        yield from bwait(ctl, mma_done, 0, abort_aware=False)

    def softmax_warp(t, k):  # warp k of warpgroup t
        ok, s_cnt = True, 0
        for item, it in enumerate(items):
            if not ok:
                break
            for _ in range(it[2 + t], it[t]):
                ok = yield from bwait(ctl, s_full[t], s_cnt)
                if not ok:
                    break
                s_cnt += 1
                p_full[t].arrive((t, k))
            if ok:
                ok = yield from bwait(ctl, pv_done[t], item)
            ok = yield from nbar[t].and_(ok)
            if ok:
                for _ in range(4):  # the epilogue's staging-tile bar.sync pairs (D = 128: two chunks)
                    yield from nbar[t].and_(True)

    agents = [producer(), mma_warp()] + [softmax_warp(t, k) for t in (0, 1) for k in range(4)]
    run(agents, (tma, mma, []), rnd)
    return ctl.abort


@pytest.mark.parametrize("paired", [False, True], ids=["consecutive", "paired"])
@pytest.mark.parametrize("S,causal,window", [(1024, True, 0), (640, False, 0), (1000, True, 200)])
def test_dense_forward_every_warp_leaves(S, causal, window, paired):
    from tests.test_dense_protocol_model import fwd_items
    items = fwd_items(S, causal, window, paired)
    gave_up = sum(dense_fwd_failure_model(items, seed, p_giveup=0.02) for seed in range(40))
    assert gave_up > 0
    for seed in range(10):
        assert dense_fwd_failure_model(items, seed, p_giveup=0.0, stall_mma=True)
