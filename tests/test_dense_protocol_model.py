"""CPU models of the dense kernels' barrier protocols, in the same form as
the sparse ones: the roles run as programs over mbarriers with the hardware's
parity semantics, copies and MMA commits complete asynchronously (TMA in any
order, MMA commits in issue order), and random interleavings must neither
pass a wait on the wrong phase nor deadlock.

Forward: the persistent kernel -- a producer that preloads the next item's
first K/V tiles before waiting for the Q buffer, MMA issue, and two softmax
warpgroups -- over the items of causal, non-causal, ragged and
sliding-window problems: with P over S and one issuer alternating the query
tiles (D = 128), and with P in columns of its own and one issuer per query
tile (D = 64). Backward: the
persistent key-tile CTA over lists of items (K/V replaced per item, the
three-stage Q/dO ring and every other barrier running on across items), in
both dQ modes (the P/dS warps reading dQ^T and staging it for one reduction
warp, as for D = 64; four drain warps, as for D = 128).

CPU only; no kernel code is involved.
"""
import random

import pytest

from tests.protocol_sim import Aliasing, Bar, By, Deadlock, run, wait


def test_barrier_flags_a_second_arrival_by_one_agent():
    """A count-2 barrier completes on two different agents' arrivals; the
    same agent arriving twice within one phase is an error."""
    b = Bar(2)
    b.arrive(0)
    b.arrive(1)
    assert b.completed == 1
    b.arrive(0)
    with pytest.raises(Aliasing):
        b.arrive(0)


def fwd_items(S, causal, window=0, paired=False):
    """(n_kv[0], n_kv[1], jlo[0], jlo[1]) of every item, longest first (a CTA
    that takes them all in that order). Unpaired, an item is two consecutive
    128-row tiles of one head; paired, the same 128 rows of two heads of one
    kv group, so both tiles need the same K/V tiles."""
    BQ = BK = 128
    nkv_all = (S + BK - 1) // BK

    def tile(qt0):
        n = min(qt0 // BK + 1, nkv_all) if causal else nkv_all
        return n, (min(max(0, qt0 - window + 1) // BK, n - 1) if window else 0)

    if paired:
        n_qt = (S + BQ - 1) // BQ
        return [(n, n, lo, lo) for n, lo in (tile((n_qt - 1 - i) * BQ) for i in range(n_qt))]
    n_qb = (S + 2 * BQ - 1) // (2 * BQ)
    items = []
    for i in range(n_qb):
        q0 = (n_qb - 1 - i) * 2 * BQ
        (n0, l0), (n1, l1) = tile(q0), tile(q0 + BQ)
        items.append((n0, n1, l0, l1))
    return items


def dense_fwd_model(items, nslot, win=False, seed=0, release_unused=False):
    rnd = random.Random(seed)
    kv_full = [Bar(1) for _ in range(nslot)]
    kv_empty = [Bar(1) for _ in range(nslot)]
    q_full, q_empty, mma_done = Bar(1), Bar(1), Bar(1)
    s_full, p_full, pv_done = [Bar(1), Bar(1)], [Bar(1), Bar(1)], [Bar(1), Bar(1)]
    tma, mma = [], []

    def producer():
        issued = q_loads = 0
        for r, (n0, n1, l0, l1) in enumerate(items):
            n_pos = 2 * (n1 - l0)

            def load_kv():
                nonlocal issued
                slot, rnd_ = issued % nslot, issued // nslot
                if rnd_ > 0:
                    yield from wait(kv_empty[slot], rnd_ - 1)
                tma.append(kv_full[slot])
                issued += 1
            pre = 0 if r == 0 else min(2, n_pos)
            for _ in range(pre):
                yield from load_kv()
            if r > 0:
                yield from wait(q_empty, r - 1)
            tma.append(q_full)
            q_loads += 1
            for _ in range(pre, n_pos):
                yield from load_kv()
        for pos in range(max(0, issued - nslot), issued):
            yield from wait(kv_full[pos % nslot], pos // nslot)
        yield from wait(q_full, q_loads - 1)

    def mma_warp():
        ring, p_cnt = 0, [0, 0]
        for r, (n0, n1, l0, l1) in enumerate(items):
            n_kv, jlo, jb = (n0, n1), (l0, l1), l0
            yield from wait(q_full, r)
            s_left = [(n0 - l0) + (n1 - l1)]

            def issue_s(t):
                mma.append(s_full[t])
                s_left[0] -= 1
                if s_left[0] == 0:
                    mma.append(q_empty)

            def wait_kv(idx):
                q = ring + idx
                yield from wait(kv_full[q % nslot], q // nslot)

            def slot(idx):
                return (ring + idx) % nslot
            yield from wait_kv(0)
            issue_s(0)
            if jlo[1] == jb:
                issue_s(1)
            mma.append(kv_empty[slot(0)])
            for j in range(jb, n1):
                v_ready = k_next = False
                for t in range(2):
                    if jlo[t] <= j < n_kv[t]:
                        yield from wait(p_full[t], p_cnt[t])
                        p_cnt[t] += 1
                        if not v_ready:
                            yield from wait_kv(2 * (j - jb) + 1)
                            v_ready = True
                        if j + 1 == n_kv[t]:
                            mma.append(pv_done[t])
                    if j + 1 < n_kv[t] and j + 1 >= jlo[t]:
                        if not k_next:
                            yield from wait_kv(2 * (j - jb) + 2)
                            k_next = True
                        issue_s(t)
                # With a window, a tile that skips j still leaves no copy in flight.
                if win and not v_ready:
                    yield from wait_kv(2 * (j - jb) + 1)
                if win and j + 1 < n1 and not k_next:
                    yield from wait_kv(2 * (j - jb) + 2)
                    k_next = True
                mma.append(kv_empty[slot(2 * (j - jb) + 1)])
                if k_next or release_unused:
                    mma.append(kv_empty[slot(2 * (j - jb) + 2)])
            ring += 2 * (n1 - jb)
        mma.append(mma_done)
        yield from wait(mma_done, 0)

    def softmax(t):
        s_cnt = 0
        for item, it in enumerate(items):
            n_kv, jlo = it[t], it[2 + t]
            for _ in range(jlo, n_kv):
                yield from wait(s_full[t], s_cnt)
                s_cnt += 1
                p_full[t].arrive()
            yield from wait(pv_done[t], item)

    return run([producer(), mma_warp(), softmax(0), softmax(1)], (tma, mma, []), rnd)


FWD_CASES = [
    (1024, True, 0), (1024, False, 0), (900, True, 0), (256, True, 0), (128, False, 0),
    (2048, True, 128), (1000, True, 200), (1024, True, 1), (640, True, 384),
]


@pytest.mark.parametrize("paired", [False, True], ids=["consecutive", "paired"])
@pytest.mark.parametrize("S,causal,window", FWD_CASES)
@pytest.mark.parametrize("nslot", [4, 8])
def test_dense_forward_protocol_is_sound(S, causal, window, nslot, paired):
    items = fwd_items(S, causal, window, paired)
    for seed in range(25):
        assert dense_fwd_model(items, nslot, win=window > 0, seed=seed)


def dense_fwd_sep_p_model(items, nslot, win=False, seed=0, skip_s_free=False, skip_pv_step=False,
                          release_count=2, wait_unread=True):
    """The forward when P_t has tensor-memory columns of its own (D = 64, where
    O_t takes 64 of its 128 columns and P_t the other 64): the softmax frees
    S_t as soon as it has read it (s_free), so the tile's MMA issuer runs S_t(j+1)
    while the exponentials of S_t(j) are computed; P_t(j) is stored only
    after P_t V(j-1) has read P_t(j-1) (pv_step, one commit per P V). The
    tensor-memory regions are tracked: a score product that lands on unread
    scores, a P store over a P that its product has not read, an O rescale or
    epilogue read before the last P V landed, or an item's first P V (which
    overwrites O) before the previous epilogue read O, raises Aliasing.
    Each query tile has its own MMA issuer (with its own in-order
    completions); ring slots, the Q buffer and the final drain complete once
    both issuers have committed (count 2); an issuer waits for every ring
    tile's copy before committing its release, including the tiles it does not
    read, so that its commit cannot land on the slot's previous phase. The
    ring is tracked too: a copy issued into a slot whose previous tile still
    has a pending read raises Aliasing. skip_s_free and skip_pv_step plant the
    two missing waits, release_count=1 a slot handed back on either issuer's
    commit, wait_unread=False releases of unread tiles without their waits."""
    rnd = random.Random(seed)
    kv_full = [Bar(1) for _ in range(nslot)]
    kv_empty = [Bar(release_count) for _ in range(nslot)]
    q_full, q_empty, mma_done = Bar(1), Bar(2), Bar(2)
    s_full, s_free = [Bar(1), Bar(1)], [Bar(1), Bar(1)]
    p_full, pv_step, pv_done = [Bar(1), Bar(1)], [Bar(1), Bar(1)], [Bar(1), Bar(1)]
    tma, mma = [], ([], [])
    # Per query tile: score tiles written / read, P tiles stored / read by P V,
    # and epilogues done.
    st = [{"s_w": 0, "s_r": 0, "p_w": 0, "p_r": 0, "epi": 0} for _ in range(2)]
    # Ring positions: the tiles whose products read each one, and those done.
    readers, done_reads = {}, {}
    base = 0
    for n0, n1, l0, l1 in items:
        for j in range(l0, n1):
            for t, (lo, n) in enumerate(((l0, n0), (l1, n1))):
                if lo <= j < n:
                    readers.setdefault(base + 2 * (j - l0), set()).add(t)
                    readers.setdefault(base + 2 * (j - l0) + 1, set()).add(t)
        base += 2 * (n1 - l0)

    def read_done(t, pos):
        done_reads.setdefault(pos, set()).add(t)

    class Done:  # an asynchronous MMA completing: check the regions, then signal
        def __init__(self, fn, bar):
            self.fn, self.bar = fn, bar

        def arrive(self):
            self.fn()
            self.bar.arrive()

    def s_lands(t, pos):
        def fn():
            if st[t]["s_w"] != st[t]["s_r"]:
                raise Aliasing(f"S_{t} product landed on scores not yet read")
            st[t]["s_w"] += 1
            read_done(t, pos)
        return fn

    def pv_lands(t, item, first, pos):
        def fn():
            read_done(t, pos)
            if st[t]["p_r"] + 1 != st[t]["p_w"]:
                raise Aliasing(f"P_{t} V read a P that was not (or no longer) there")
            if first and st[t]["epi"] != item:
                raise Aliasing(f"item {item}'s first P_{t} V overwrote O before the epilogue read it")
            st[t]["p_r"] += 1
        return fn

    def producer():
        issued = q_loads = 0
        for r, (n0, n1, l0, l1) in enumerate(items):
            n_pos = 2 * (n1 - l0)

            def load_kv():
                nonlocal issued
                slot, rnd_ = issued % nslot, issued // nslot
                if rnd_ > 0:
                    yield from wait(kv_empty[slot], rnd_ - 1)
                    prev = issued - nslot
                    if readers.get(prev, set()) - done_reads.get(prev, set()):
                        raise Aliasing(f"ring slot {slot} reloaded while tile {prev} has a pending read")
                tma.append(kv_full[slot])
                issued += 1
            pre = 0 if r == 0 else min(2, n_pos)
            for _ in range(pre):
                yield from load_kv()
            if r > 0:
                yield from wait(q_empty, r - 1)
            tma.append(q_full)
            q_loads += 1
            for _ in range(pre, n_pos):
                yield from load_kv()
        for pos in range(max(0, issued - nslot), issued):
            yield from wait(kv_full[pos % nslot], pos // nslot)
        yield from wait(q_full, q_loads - 1)

    def mma_warp(t):
        ring, p_cnt, s_iss, q = 0, 0, 0, mma[t]
        for r, it in enumerate(items):
            n1, jb = it[1], it[2]
            my_n, my_lo = it[t], it[2 + t]
            yield from wait(q_full, r)
            s_left = [my_n - my_lo]

            def issue_s(pos):
                nonlocal s_iss
                if s_iss > 0 and not skip_s_free:
                    yield from wait(s_free[t], s_iss - 1)
                s_iss += 1
                q.append(Done(s_lands(t, pos), s_full[t]))
                s_left[0] -= 1
                if s_left[0] == 0:
                    q.append(By(q_empty, t))

            def wait_kv(idx):
                pos = ring + idx
                yield from wait(kv_full[pos % nslot], pos // nslot)

            def slot(idx):
                return (ring + idx) % nslot
            if my_lo == jb or wait_unread:
                yield from wait_kv(0)
            if my_lo == jb:
                yield from issue_s(ring)
            q.append(By(kv_empty[slot(0)], t))
            for j in range(jb, n1):
                k_done = v_done = False
                if my_lo <= j + 1 < my_n:  # the next scores first
                    yield from wait_kv(2 * (j - jb) + 2)
                    k_done = True
                    yield from issue_s(ring + 2 * (j + 1 - jb))
                if my_lo <= j < my_n:
                    yield from wait_kv(2 * (j - jb) + 1)
                    v_done = True
                    yield from wait(p_full[t], p_cnt)
                    p_cnt += 1
                    q.append(Done(pv_lands(t, r, j == my_lo, ring + 2 * (j - jb) + 1), pv_step[t]))
                    if j + 1 == my_n:
                        q.append(pv_done[t])
                if wait_unread and not v_done:
                    yield from wait_kv(2 * (j - jb) + 1)
                if wait_unread and j + 1 < n1 and not k_done:
                    yield from wait_kv(2 * (j - jb) + 2)
                q.append(By(kv_empty[slot(2 * (j - jb) + 1)], t))
                if j + 1 < n1:
                    q.append(By(kv_empty[slot(2 * (j - jb) + 2)], t))
            ring += 2 * (n1 - jb)
        q.append(By(mma_done, t))
        yield from wait(mma_done, 0)

    def softmax(t):
        s_cnt = 0
        for item, it in enumerate(items):
            n_kv, jlo = it[t], it[2 + t]
            for _ in range(jlo, n_kv):
                yield from wait(s_full[t], s_cnt)
                s_cnt += 1
                if st[t]["s_r"] + 1 != st[t]["s_w"]:
                    raise Aliasing(f"softmax {t} read scores that were not there")
                st[t]["s_r"] += 1
                s_free[t].arrive()
                yield  # the exponentials
                if s_cnt > 1 and not skip_pv_step:
                    yield from wait(pv_step[t], s_cnt - 2)
                # O rescale and the P store: every earlier P V has landed.
                if st[t]["p_r"] != st[t]["p_w"]:
                    raise Aliasing(f"softmax {t} stored P (or rescaled O) under a pending P V")
                st[t]["p_w"] += 1
                p_full[t].arrive()
            yield from wait(pv_done[t], item)
            if st[t]["p_r"] != st[t]["p_w"]:
                raise Aliasing(f"epilogue {t} read O before its last P V landed")
            st[t]["epi"] += 1

    return run([producer(), mma_warp(0), mma_warp(1), softmax(0), softmax(1)], (tma, mma, []), rnd)


@pytest.mark.parametrize("paired", [False, True], ids=["consecutive", "paired"])
@pytest.mark.parametrize("S,causal,window", FWD_CASES)
@pytest.mark.parametrize("nslot", [4, 8])
def test_dense_forward_separate_p_protocol_is_sound(S, causal, window, nslot, paired):
    items = fwd_items(S, causal, window, paired)
    for seed in range(25):
        assert dense_fwd_sep_p_model(items, nslot, win=window > 0, seed=seed)


def test_separate_p_model_catches_the_missing_waits():
    """Without the s_free wait a score product lands on scores the softmax has
    not read; without the pv_step wait a P store overwrites a P that its
    product has not read; with ring slots handed back on one issuer's commit
    a slot's barrier completes twice per use (each in some interleaving)."""
    for kw in ({"skip_s_free": True}, {"skip_pv_step": True}, {"release_count": 1}):
        caught = 0
        for seed in range(30):
            try:
                dense_fwd_sep_p_model(fwd_items(1024, True), 8, seed=seed, **kw)
            except (Aliasing, Deadlock):
                caught += 1
        assert caught > 0, kw


def test_separate_p_model_catches_an_unwaited_release():
    """An issuer that commits the release of a ring tile it does not read
    without waiting for its copy can arrive twice on one phase of the slot's
    barrier (when it runs far enough ahead of the other issuer); the slot is
    then reloaded under the other tile's pending read."""
    caught = 0
    for seed in range(60):
        for S, window in ((1024, 0), (2048, 300)):
            try:
                dense_fwd_sep_p_model(fwd_items(S, True, window), 4, win=window > 0, seed=seed,
                                      wait_unread=False)
            except (Aliasing, Deadlock):
                caught += 1
    assert caught > 0


def dense_bwd_model(items, dq_in_compute, stages=3, seed=0, stage_last=True, early_kv=False, ring=4):
    """The persistent backward main kernel over one CTA's items (n_it of
    each): the producer takes each item's code and publishes it in a ring of
    `ring` slots that the other roles read (a read that finds a later item's
    code there is aliasing), K/V replaced per item after kv_free, the item's
    first query stages issued before that wait, per-item mma_done and dkv_free
    (the compute warps' dK/dV read-out before the next item's first dV/dK
    products). early_kv plants a mistake: the next item's K/V load does not
    wait; ring=1 another: a one-slot ring."""
    rnd = random.Random(seed)
    item_bar = [Bar(1) for _ in range(ring)]
    slot_item = [None] * ring

    def publish(ii):
        slot_item[ii % ring] = ii
        item_bar[ii % ring].arrive()

    def take(ii, who):
        yield from wait(item_bar[ii % ring], ii // ring)
        if slot_item[ii % ring] != ii:
            raise Aliasing(f"{who} read item slot {ii % ring} for item {ii}, found {slot_item[ii % ring]}")
    kv_full, kv_free, mma_done, fin = Bar(1), Bar(1), Bar(1), Bar(1)
    dkv_free = Bar(2)                         # both P/dS warp groups arrive
    st_full = [Bar(1) for _ in range(stages)]
    st_empty = [Bar(1) for _ in range(stages)]
    sdp_full, sdp_free = Bar(1), Bar(2)
    pds_full, pds_free = Bar(2), Bar(1)
    dq_full, dq_free = Bar(1), Bar(1)
    stg_full, stg_free = [Bar(1), Bar(1)], [Bar(1), Bar(1)]
    tma, mma = [], []
    state = {"kv_item": -1, "mma_item_reading_kv": None}

    class KvLoad:  # a K/V load landing: the buffer now holds item ii
        def __init__(self, ii):
            self.ii = ii

        def arrive(self):
            if state["mma_item_reading_kv"] is not None and state["mma_item_reading_kv"] != self.ii:
                raise Aliasing(f"K/V of item {self.ii} landed under item {state['mma_item_reading_kv']}'s products")
            state["kv_item"] = self.ii
            kv_full.arrive()

    class KvUse:  # an MMA reading K/V of item ii completes
        def __init__(self, ii, last, bar):
            self.ii, self.last, self.bar = ii, last, bar

        def arrive(self):
            if state["kv_item"] != self.ii:
                raise Aliasing(f"a product of item {self.ii} read item {state['kv_item']}'s K/V")
            if self.last:
                state["mma_item_reading_kv"] = None
            if self.bar is not None:
                self.bar.arrive()

    def producer():
        git, issued, kv_issued = 0, 0, 0
        for ii, n_it in enumerate(items):
            publish(ii)
            n_early = 0 if ii == 0 else min(stages, n_it)
            if ii == 0:
                tma.append(KvLoad(0))
                kv_issued += 1
            for it in range(n_it):
                if ii > 0 and it == n_early:
                    if not early_kv:
                        yield from wait(kv_free, ii - 1)
                    tma.append(KvLoad(ii))
                    kv_issued += 1
                gi = git + it
                s, rnd_ = gi % stages, gi // stages
                if rnd_ > 0:
                    yield from wait(st_empty[s], rnd_ - 1)
                tma.append(st_full[s])
                issued = gi + 1
            if ii > 0 and n_it <= n_early:
                if not early_kv:
                    yield from wait(kv_free, ii - 1)
                tma.append(KvLoad(ii))
                kv_issued += 1
            git += n_it
        publish(len(items))  # the end of the list
        for gi in range(max(0, issued - stages), issued):
            yield from wait(st_full[gi % stages], gi // stages)
        if kv_issued:
            yield from wait(kv_full, kv_issued - 1)

    def mma_warp():
        git = 0
        for ii, n_it in enumerate(items):
            yield from take(ii, "mma")
            yield from wait(kv_full, ii)
            yield from wait(st_full[git % stages], git // stages)
            if git > 0:
                yield from wait(sdp_free, git - 1)
            state["mma_item_reading_kv"] = ii
            mma.append(KvUse(ii, False, sdp_full))
            for it in range(n_it):
                gi = git + it
                if it + 1 < n_it:
                    yield from wait(st_full[(gi + 1) % stages], (gi + 1) // stages)
                    yield from wait(sdp_free, gi)
                    mma.append(KvUse(ii, False, sdp_full))
                yield from wait(pds_full, gi)
                if it == 0 and ii > 0:
                    yield from wait(dkv_free, ii - 1)
                mma.append(st_empty[gi % stages])
                if not dq_in_compute and gi >= 1:
                    yield from wait(dq_free, gi - 1)
                mma.append(KvUse(ii, it == n_it - 1, dq_full if not dq_in_compute else None))
                mma.append(pds_free)
            mma.append(kv_free)
            mma.append(mma_done)
            git += n_it
        yield from take(len(items), "mma")
        mma.append(fin)
        yield from wait(fin, 0)

    def compute(cg):
        def stage(gq):
            if gq >= 1:
                yield from wait(stg_free[cg], gq - 1)
            stg_full[cg].arrive()
        git = 0
        for ii, n_it in enumerate(items):
            yield from take(ii, f"compute {cg}")
            for it in range(n_it):
                gi = git + it
                yield from wait(sdp_full, gi)
                yield from wait(st_full[gi % stages], gi // stages)
                sdp_free.arrive(cg)
                if gi >= 1:
                    yield from wait(pds_free, gi - 1)
                if not dq_in_compute and gi >= 1:
                    yield from wait(dq_free, gi - 1)
                pds_full.arrive(cg)
                if dq_in_compute and it >= 1:
                    yield from stage(gi - 1)
            if dq_in_compute and n_it > 0 and stage_last:
                yield from wait(pds_free, git + n_it - 1)
                yield from stage(git + n_it - 1)
            yield from wait(mma_done, ii)
            dkv_free.arrive(cg)
            git += n_it
        yield from take(len(items), f"compute {cg}")

    def reduce_warp():
        gq = 0
        for ii, n_it in enumerate(items):
            yield from take(ii, "reduce")
            for _ in range(n_it):
                for half in range(2):
                    yield from wait(stg_full[half], gq)
                    stg_free[half].arrive()
                gq += 1
        yield from take(len(items), "reduce")

    def drain_warps():
        gi = 0
        for ii, n_it in enumerate(items):
            yield from take(ii, "drain")
            for _ in range(n_it):
                yield from wait(dq_full, gi)
                dq_free.arrive()
                gi += 1
        yield from take(len(items), "drain")

    agents = [producer(), mma_warp(), compute(0), compute(1)]
    agents.append(reduce_warp() if dq_in_compute else drain_warps())
    return run(agents, (tma, mma, []), rnd)


BWD_ITEM_LISTS = [[1], [2], [3], [4], [7], [16], [5, 1, 1], [1, 1, 1, 1], [2, 7, 3], [4, 4, 2, 1], [9, 3, 2, 2, 1]]


@pytest.mark.parametrize("items", BWD_ITEM_LISTS, ids=[",".join(map(str, x)) for x in BWD_ITEM_LISTS])
@pytest.mark.parametrize("dq_in_compute", [True, False])
def test_dense_backward_protocol_is_sound(items, dq_in_compute):
    for seed in range(40):
        assert dense_bwd_model(items, dq_in_compute, seed=seed)


def test_dense_models_catch_planted_mistakes():
    """The models are not vacuous: a forward MMA issuer that also releases
    the slot after an item's last V tile (which holds no K tile of this item)
    hands out a slot phase too early, and a backward whose P/dS warps never
    stage the last dQ tile leaves the reduction warp waiting."""
    for seed in range(10):
        with pytest.raises((Aliasing, Deadlock)):
            dense_fwd_model(fwd_items(1024, True), 4, seed=seed, release_unused=True)
    with pytest.raises(Deadlock):
        dense_bwd_model([3], True, seed=0, stage_last=False)
    # A next item's K/V load that does not wait for kv_free lands under the
    # previous item's products in some interleaving.
    caught = 0
    for seed in range(30):
        try:
            dense_bwd_model([4, 4], False, seed=seed, early_kv=True)
        except (Aliasing, Deadlock):
            caught += 1
    assert caught > 0
    # A one-slot ring of item codes: the producer publishes the next item's
    # code before a slower role has read the current one.
    caught = 0
    for seed in range(40):
        for dq_in_compute in (True, False):
            try:
                dense_bwd_model([1, 1, 3, 1], dq_in_compute, seed=seed, ring=1)
            except (Aliasing, Deadlock):
                caught += 1
    assert caught > 0



def dvec_model(items, nslot, seed=0, early_free=False):
    """The backward's Dvec pass: the forward's producer (Q and dO of both
    tiles per item, K/V ring), an MMA issuer that per key tile issues both
    tiles' S products (then hands K_j back) and both tiles' dP products (then
    hands V_j back), each tile's S/dP buffers reused only after its rows have
    read them; two row groups. early_free plants a mistake: the row groups
    hand their buffers back before reading them."""
    rnd = random.Random(seed)
    kv_full = [Bar(1) for _ in range(nslot)]
    kv_empty = [Bar(1) for _ in range(nslot)]
    q_full, q_empty, mma_done = Bar(1), Bar(1), Bar(1)
    sdp_full, sdp_free = [Bar(1), Bar(1)], [Bar(1), Bar(1)]
    tma, mma = [], []
    # Which product pair of tile t each buffer holds, to catch a read of a
    # buffer that the next pair has already overwritten.
    held = [None, None]

    class Overwritten(Exception):
        pass

    def producer():
        issued = q_loads = 0
        for r, (n0, n1, l0, l1) in enumerate(items):
            n_pos = 2 * (n1 - l0)

            def load_kv():
                nonlocal issued
                slot, rnd_ = issued % nslot, issued // nslot
                if rnd_ > 0:
                    yield from wait(kv_empty[slot], rnd_ - 1)
                tma.append(kv_full[slot])
                issued += 1
            pre = 0 if r == 0 else min(2, n_pos)
            for _ in range(pre):
                yield from load_kv()
            if r > 0:
                yield from wait(q_empty, r - 1)
            tma.append(q_full)
            q_loads += 1
            for _ in range(pre, n_pos):
                yield from load_kv()
        for pos in range(max(0, issued - nslot), issued):
            yield from wait(kv_full[pos % nslot], pos // nslot)
        yield from wait(q_full, q_loads - 1)

    class Write:
        """An MMA completion that overwrites tile t's buffers with pair n."""
        def __init__(self, t, n):
            self.t, self.n = t, n

        def arrive(self):
            held[self.t] = self.n
            Bar.changes += 1

    def mma_warp():
        ring, n_sdp = 0, [0, 0]
        for r, (n0, n1, l0, l1) in enumerate(items):
            n_kv, jlo, jb = (n0, n1), (l0, l1), l0
            yield from wait(q_full, r)
            left = (n0 - l0) + (n1 - l1)

            def wait_kv(idx):
                q = ring + idx
                yield from wait(kv_full[q % nslot], q // nslot)

            def slot(idx):
                return (ring + idx) % nslot
            for j in range(jb, n1):
                yield from wait_kv(2 * (j - jb))
                for t in range(2):
                    if jlo[t] <= j < n_kv[t]:
                        if n_sdp[t] > 0:
                            yield from wait(sdp_free[t], n_sdp[t] - 1)
                        mma.append(Write(t, n_sdp[t]))
                mma.append(kv_empty[slot(2 * (j - jb))])
                yield from wait_kv(2 * (j - jb) + 1)
                for t in range(2):
                    if jlo[t] <= j < n_kv[t]:
                        mma.append(sdp_full[t])
                        n_sdp[t] += 1
                        left -= 1
                        if left == 0:
                            mma.append(q_empty)
                mma.append(kv_empty[slot(2 * (j - jb) + 1)])
            ring += 2 * (n1 - jb)
        mma.append(mma_done)
        yield from wait(mma_done, 0)

    def rows(t):
        n_seen = 0
        for it in items:
            for _ in range(it[2 + t], it[t]):
                yield from wait(sdp_full[t], n_seen)
                if early_free:
                    sdp_free[t].arrive()
                    yield
                if held[t] != n_seen:
                    raise Overwritten(f"tile {t}: pair {n_seen} read after pair {held[t]} landed")
                if not early_free:
                    sdp_free[t].arrive()
                n_seen += 1

    agents = [producer(), mma_warp(), rows(0), rows(1)]
    try:
        return run(agents, (tma, mma, []), rnd)
    except Overwritten as e:
        from tests.protocol_sim import Aliasing
        raise Aliasing(str(e))


@pytest.mark.parametrize("paired", [False, True], ids=["consecutive", "paired"])
@pytest.mark.parametrize("S,causal,window", FWD_CASES)
@pytest.mark.parametrize("nslot", [3, 8])
def test_dvec_pass_protocol_is_sound(S, causal, window, nslot, paired):
    items = fwd_items(S, causal, window, paired)
    for seed in range(25):
        assert dvec_model(items, nslot, seed=seed)


def test_dvec_model_catches_an_early_buffer_release():
    from tests.protocol_sim import Aliasing
    caught = 0
    for seed in range(40):
        try:
            dvec_model(fwd_items(1024, True), 3, seed=seed, early_free=True)
        except Aliasing:
            caught += 1
    assert caught > 0
