"""CPU models of the sparse kernels' barrier protocols.

The kernel's roles (K producer, V producer, MMA issuer, two softmax
warpgroups) are written as programs over mbarriers with the hardware's wait
semantics: a wait for the phase with parity P succeeds when the barrier's
current phase parity differs from P. Copies (TMA, cp.async) and MMA commits
complete asynchronously -- TMA copies in any order, cp.async groups of one
thread in order, MMA commits in issue order -- and a random scheduler
interleaves everything. Each successful wait must be the completion of the
phase it was meant for (no parity aliasing), and every run must finish (no
deadlock). The same model with K and V sharing one ring under two producers
-- a layout that misbehaved on the GPU -- must be caught: the K producer's
closing wait for its last copies then targets slots that the V producer
reuses afterwards, so the phase it waits for has already been passed.

The backward's protocol (K producer with the token's Q/dO, V producer with
one slot, MMA issuer, compute warps) is modelled the same way; its first
version, one producer that waited for the previous token's products before
issuing anything for the next token, must deadlock as it did on the GPU.

CPU only; no kernel code is involved.
"""
import random

import pytest

from tests.protocol_sim import Aliasing, Bar, Deadlock, run, wait


def sparse_fwd_model(n_items, nch, nslot, kslots, shared_ring=False, seed=0):
    rnd = random.Random(seed)
    vslots = nslot - kslots
    full = [Bar(1) for _ in range(nslot)]
    empty = [Bar(1) for _ in range(nslot)]
    q_full, q_empty = Bar(1), Bar(1)
    s_full, p_full, pv_done = [Bar(1), Bar(1)], [Bar(1), Bar(1)], [Bar(1), Bar(1)]
    merge, o1_free = Bar(1), Bar(1)
    nonlocal_last = [-1]
    tma = []        # pending TMA completions (any order)
    mma = []        # pending MMA commits (issue order)
    cpa = []        # pending cp.async groups of the V producer (in order): [done, slot]

    def kslot(g):
        return (2 * g) % nslot if shared_ring else g % kslots

    def kround(g):
        return (2 * g) // nslot if shared_ring else g // kslots

    def vslot(g):
        return (2 * g + 1) % nslot if shared_ring else kslots + g % vslots

    def vround(g):
        return (2 * g + 1) // nslot if shared_ring else g // vslots

    def k_producer():
        for r in range(n_items):
            def load_k(c):
                g = r * nch + c
                if kround(g) > 0:
                    yield from wait(empty[kslot(g)], kround(g) - 1)
                tma.append(full[kslot(g)])
                nonlocal_last[0] = g
            if r > 0:
                yield from load_k(0)
                yield from wait(q_empty, r - 1)
            tma.append(q_full)
            for c in range(1 if r > 0 else 0, nch):
                yield from load_k(c)
        # Before exiting, the K producer waits for its last copies to land
        # (the kernel bounds this wait; here it must simply succeed). Its
        # last chunks are the ones whose slots nothing reuses afterwards --
        # unless another producer shares the slots.
        last = nonlocal_last[0]
        if shared_ring:  # the K chunks among the last nslot ring positions
            tail = [g for g in range(last + 1) if 2 * g >= 2 * last - nslot]
        else:            # the last kslots K chunks
            tail = range(max(0, last - kslots + 1), last + 1)
        for g in tail:
            yield from wait(full[kslot(g)], kround(g))

    def v_producer():
        issued = signalled = 0
        for r in range(n_items):
            for c in range(nch):
                g = r * nch + c
                if vround(g) > 0:
                    yield from wait(empty[vslot(g)], vround(g) - 1)
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
        p_cnt = [0, 0]
        for r in range(n_items):
            yield from wait(q_full, r)
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
                yield from wait(full[kslot(g)], kround(g))
                issue_s(c)
            for c in range(nch):
                w, g = c & 1, r * nch + c
                yield from wait(p_full[w], p_cnt[w])
                p_cnt[w] += 1
                yield from wait(full[vslot(g)], vround(g))
                mma.append(empty[vslot(g)])
                if c + 2 >= nch:
                    mma.append(pv_done[w])
                if c + 2 < nch:
                    g2 = g + 2
                    yield from wait(full[kslot(g2)], kround(g2))
                    issue_s(c + 2)

    def softmax(w):
        s_cnt = pv_cnt = 0
        my_n = (nch - w + 1) // 2 if nch > w else 0
        for rr in range(n_items):
            checked = w == 0 or rr == 0
            for _ in range(my_n):
                yield from wait(s_full[w], s_cnt)
                s_cnt += 1
                if not checked:
                    yield from wait(o1_free, rr - 1)
                    checked = True
                p_full[w].arrive()
            if my_n > 0:
                yield from wait(pv_done[w], pv_cnt)
                pv_cnt += 1
            if w == 1:
                if not checked:
                    yield from wait(o1_free, rr - 1)
                merge.arrive()
                continue
            yield from wait(merge, rr)
            o1_free.arrive()

    return run([k_producer(), v_producer(), mma_warp(), softmax(0), softmax(1)], (tma, mma, cpa), rnd)


CASES = [(n_items, nch) for n_items in (1, 2, 5) for nch in (1, 2, 3, 5, 9)]


@pytest.mark.parametrize("n_items,nch", CASES)
def test_sparse_forward_protocol_is_sound(n_items, nch):
    for seed in range(40):
        assert sparse_fwd_model(n_items, nch, nslot=5, kslots=2, seed=seed)


def test_sparse_forward_protocol_other_slot_splits():
    for nslot, kslots in ((4, 2), (8, 2), (8, 4)):
        for seed in range(20):
            assert sparse_fwd_model(4, 5, nslot, kslots, seed=seed)


def test_shared_ring_under_two_producers_is_caught():
    caught = 0
    for seed in range(200):
        try:
            sparse_fwd_model(6, 5, nslot=5, kslots=2, shared_ring=True, seed=seed)
        except (Aliasing, Deadlock):
            caught += 1
    assert caught > 0


def sparse_bwd_model(n_items, nch, kslots=2, single_producer_no_flush=False, seed=0):
    """The backward kernel's roles: K producer (Q/dO/row vectors per token, K
    chunks by TMA into kslots slots), V producer (cp.async into one slot, each
    chunk reported once it has landed), MMA issuer, and the compute warps
    (P/dS, then the drain). With single_producer_no_flush, one producer
    gathers K and V with cp.async into a shared ring of kslots + 1 slots,
    keeps one position in flight and waits for the previous token's products
    before issuing anything for the next token (the first version)."""
    rnd = random.Random(seed)
    nslot = kslots + 1
    vs = kslots
    full = [Bar(1) for _ in range(nslot)]
    empty = [Bar(1) for _ in range(nslot)]
    q_full, q_empty = Bar(1), Bar(1)
    sdp_full, pds_full, grads_full = Bar(1), Bar(1), Bar(1)
    dk_drained, dv_drained = Bar(1), Bar(1)
    tma, mma, cpa = [], [], []

    def kslot(g):
        return (2 * g) % nslot if single_producer_no_flush else g % kslots

    def kround(g):
        return (2 * g) // nslot if single_producer_no_flush else g // kslots

    def vslot(g):
        return (2 * g + 1) % nslot if single_producer_no_flush else vs

    def vround(g):
        return (2 * g + 1) // nslot if single_producer_no_flush else g

    def k_producer():
        last = -1
        for r in range(n_items):
            def load_k(c):
                nonlocal last
                g = r * nch + c
                if kround(g) > 0:
                    yield from wait(empty[kslot(g)], kround(g) - 1)
                tma.append(full[kslot(g)])
                last = g
            if r > 0:
                yield from load_k(0)
                yield from wait(q_empty, r - 1)
            tma.append(q_full)
            for c in range(1 if r > 0 else 0, nch):
                yield from load_k(c)
        for g in range(max(0, last - kslots + 1), last + 1):
            yield from wait(full[kslot(g)], kround(g))
        yield from wait(q_full, n_items - 1)

    def v_producer():
        for r in range(n_items):
            for c in range(nch):
                g = r * nch + c
                if g > 0:
                    yield from wait(empty[vs], g - 1)
                cpa.append([False, vs])
                while not cpa[-1][0]:
                    yield
                full[vs].arrive()

    def single_producer():
        issued, signalled, pend = 0, 0, []
        for r in range(n_items):
            if r > 0:
                yield from wait(q_empty, r - 1)
            tma.append(q_full)
            for pos in range(2 * nch):
                g, is_v = r * nch + pos // 2, pos & 1
                slot, rnd_ = (vslot(g), vround(g)) if is_v else (kslot(g), kround(g))
                if rnd_ > 0:
                    yield from wait(empty[slot], rnd_ - 1)
                cpa.append([False, slot])
                pend.append(len(cpa) - 1)
                issued += 1
                if issued - signalled > 1:
                    while not cpa[pend[signalled]][0]:
                        yield
                    full[cpa[pend[signalled]][1]].arrive()
                    signalled += 1
        while signalled < issued:
            while not cpa[pend[signalled]][0]:
                yield
            full[cpa[pend[signalled]][1]].arrive()
            signalled += 1

    def mma_warp():
        chunk = 0
        for r in range(n_items):
            yield from wait(q_full, r)
            for c in range(nch):
                g = r * nch + c
                if chunk > 0:
                    # S^T(c) overwrites the columns dK_(c-1) was drained from
                    yield from wait(dk_drained, chunk - 1)
                yield from wait(full[kslot(g)], kround(g))
                yield from wait(full[vslot(g)], vround(g))
                mma.append(sdp_full)
                mma.append(empty[vslot(g)])
                yield from wait(pds_full, chunk)
                if chunk > 0:
                    # dV_c (and a token's first dQ^T) overwrite dV_(c-1) / dq's columns
                    yield from wait(dv_drained, chunk - 1)
                mma.append(grads_full)
                mma.append(empty[kslot(g)])
                if c + 1 == nch:
                    mma.append(q_empty)
                chunk += 1

    def compute():
        chunk = 0
        for r in range(n_items):
            yield from wait(q_full, r)
            for c in range(nch):
                yield from wait(sdp_full, chunk)
                pds_full.arrive()
                yield from wait(grads_full, chunk)
                dk_drained.arrive()
                yield
                dv_drained.arrive()
                chunk += 1

    producers = [single_producer()] if single_producer_no_flush else [k_producer(), v_producer()]
    return run(producers + [mma_warp(), compute()], (tma, mma, cpa), rnd)


@pytest.mark.parametrize("n_items,nch", CASES)
def test_sparse_backward_protocol_is_sound(n_items, nch):
    for seed in range(40):
        assert sparse_bwd_model(n_items, nch, seed=seed)


def test_sparse_backward_protocol_more_k_slots():
    for seed in range(20):
        assert sparse_bwd_model(4, 5, kslots=3, seed=seed)


def test_single_producer_without_flush_deadlocks():
    """The first backward version stopped on its bounded waits whenever a CTA
    had more than one token; the model reproduces that."""
    with pytest.raises(Deadlock):
        sparse_bwd_model(3, 2, single_producer_no_flush=True, seed=0)
    assert sparse_bwd_model(1, 5, single_producer_no_flush=True, seed=0)  # one token: fine
