"""Shared pieces of the CPU protocol models (test infrastructure): mbarriers
with the hardware's phase and parity semantics, a checked wait, and a random
interleaver of role programs and asynchronous completions."""


class Bar:
    changes = 0  # every arrival counts as progress

    def __init__(self, count):
        self.count, self.pending, self.completed = count, count, 0
        self.arrived = set()

    def arrive(self, who=None):
        """One arrival. With `who` (the arriving agent), a second arrival by
        the same agent within one phase raises Aliasing: it would complete the
        phase without an agent that has not arrived yet."""
        if who is not None:
            if who in self.arrived:
                raise Aliasing(f"{who} arrived twice within one phase (phase {self.completed})")
            self.arrived.add(who)
        Bar.changes += 1
        self.pending -= 1
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count
            self.arrived = set()


class By:
    """An arrival on `bar` by agent `who`, for the asynchronous completion
    queues (a commit that arrives when the agent's earlier MMAs complete)."""

    def __init__(self, bar, who):
        self.bar, self.who = bar, who

    def arrive(self):
        self.bar.arrive(self.who)


class Aliasing(Exception):
    pass


class Deadlock(Exception):
    pass


def wait(bar, phase):
    """A generator step: block until the hardware would report the phase with
    parity phase & 1 complete; then check that it really is `phase`."""
    while (bar.completed & 1) == (phase & 1):
        yield
    if bar.completed != phase + 1:
        raise Aliasing(f"wait for phase {phase} passed with {bar.completed} phases completed")


def run(agents, queues, rnd):
    """Interleave the agents and the asynchronous completions; raise Deadlock
    when nothing changes for a long stretch. `mma` is one in-order queue of
    MMA completions, or a tuple of them (one per issuing thread: each in
    order, the queues in any interleaving)."""
    tma, mma, cpa = queues
    fifos = mma if isinstance(mma, tuple) else (mma,)
    live = list(range(len(agents)))
    idle = 0
    n_mma = lambda: sum(len(q) for q in fifos)
    while live or tma or n_mma() or any(not d for d, _ in cpa):
        before = (Bar.changes, len(tma), n_mma(), len(cpa), len(live))
        events = (["tma"] if tma else []) + (["mma"] if n_mma() else []) + \
                 (["cpa"] if any(not d for d, _ in cpa) else [])
        choice = rnd.choice(live + events)
        if choice == "tma":
            tma.pop(rnd.randrange(len(tma))).arrive()
        elif choice == "mma":
            rnd.choice([q for q in fifos if q]).pop(0).arrive()
        elif choice == "cpa":
            next(e for e in cpa if not e[0])[0] = True
            Bar.changes += 1
        else:
            try:
                next(agents[choice])
            except StopIteration:
                live.remove(choice)
        if (Bar.changes, len(tma), n_mma(), len(cpa), len(live)) == before:
            idle += 1
            if idle > 20000:
                raise Deadlock("every role waits and nothing is in flight")
        else:
            idle = 0
    return True
