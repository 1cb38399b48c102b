"""A small checker for mbarrier protocols, used by the protocol tests.

Barrier mimics an mbarrier: a count of arrivals completes a phase, and a
parity wait passes when the current phase parity differs from the awaited
one.  The checker raises Violation when a wait passes without exactly the
awaited phase completed (the waiter ran two phases ahead), when a wait meets a
barrier two phases beyond it, or when arrivals exceed a barrier's count.

run_roles() runs role generators under a random interleaving.  A role yields
actions:
  ("wait", barrier, phase)    wait for that phase (-1: the first, free use)
  ("arrive", barrier, units)  arrive
  ("tma", barrier)            a copy that lands later, in any order
  ("mma",) ("commit", barrier)  tensor-core products of the role, completing
                              in issue order; a commit arrives after all of
                              the role's earlier products
  ("pair", key)               meet the other role that yields the same key
Data versions (optional): ("mma", reads, writes) with lists of (region, tag)
checks at issue and again at completion that each region it reads holds that
tag, and stores its tags at completion (a third list, ("mma", reads, writes,
chained), names accumulator inputs written by the same role's earlier
products: products of one role execute in order, so those are checked at
completion only); ("tma", barrier, region, tag) stores
its tag when it lands; ("read", region, tag) and ("write", region, tag) are a
role's own accesses.  A read that meets another tag is a stale read or an
overwrite of data still in use.
Host logic only.
"""


class Violation(Exception):
    pass


class Barrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.done = 0      # completed phases
        self.pending = 0   # arrivals in the current phase

    def arrive(self, k=1):
        self.pending += k
        if self.pending > self.count:
            raise Violation(f"{self.name}: {self.pending} arrivals for a count of {self.count}")
        if self.pending == self.count:
            self.done += 1
            self.pending = 0

    def try_wait(self, m):
        """Wait for phase m (m = -1: nothing to wait for).  Hardware rule:
        pass when the current phase parity differs from m's parity."""
        parity = m & 1
        passes = (self.done & 1) != parity
        if passes and self.done != m + 1:
            raise Violation(f"{self.name}: wait for phase {m} passed with {self.done} completed")
        if not passes and self.done > m + 1:
            raise Violation(f"{self.name}: wait for phase {m} overtaken ({self.done} completed)")
        return passes




def run_roles(roles, bars, issuers, rng, max_events=200000):
    """Run role generators to the end under a random interleaving.  `issuers`
    names the roles whose products and commits complete in issue order."""
    nxt = {k: None for k in roles}
    regions = {}

    def check_reads(reads, when):
        for r, tag in reads:
            if regions.get(r) != tag:
                raise Violation(f"{r}: {when} expects {tag}, holds {regions.get(r)}")
    finished = set()
    tma = []                            # barriers of copies in flight (land in any order)
    fifo = {k: [] for k in issuers}     # per issuer: products and commits in issue order
    pair_seen = {}

    def step_role(k):
        if nxt[k] is None:
            try:
                nxt[k] = next(roles[k])
            except StopIteration:
                finished.add(k)
                return True
        act = nxt[k]
        kind = act[0]
        if kind == "wait":
            if not bars[act[1]].try_wait(act[2]):
                return False
        elif kind == "arrive":
            bars[act[1]].arrive(act[2])
        elif kind == "tma":
            tma.append(act)
        elif kind == "mma":
            if len(act) > 1:
                check_reads(act[1], "a product at issue")
            fifo[k].append(act)
        elif kind == "commit":
            fifo[k].append(act)
        elif kind == "read":
            check_reads([(act[1], act[2])], "a read")
        elif kind == "write":
            regions[act[1]] = act[2]
        elif kind == "pair":
            pair_seen.setdefault(act[1], set()).add(k)
            if len(pair_seen[act[1]]) < 2:
                nxt[k] = ("pairwait", act[1])
                return True
        elif kind == "pairwait":
            if len(pair_seen[act[1]]) < 2:
                return False
        nxt[k] = None
        return True

    # per-run speeds: some roles and engines run much slower than others, so
    # that one half can fall several tiles behind the other
    speed = {k: rng.choice([0.05, 0.2, 1.0, 1.0]) for k in roles}
    speed["tma"] = rng.choice([0.05, 0.3, 1.0])
    for k in issuers:
        speed[k + "_mma"] = rng.choice([0.05, 0.3, 1.0])

    def land(act):
        if len(act) > 2:
            regions[act[2]] = act[3]
        bars[act[1]].arrive(1)

    def fire(ev):
        if ev == "tma":
            land(tma.pop(rng.randrange(len(tma))))
            return True
        if ev.endswith("_mma"):
            act = fifo[ev[:-4]].pop(0)
            if act[0] == "commit":
                bars[act[1]].arrive(1)
            elif len(act) > 1:
                check_reads(act[1], "a product at completion")
                if len(act) > 3:
                    check_reads(act[3], "a chained product at completion")
                for r, tag in act[2]:
                    regions[r] = tag
            return True
        return step_role(ev)

    for _ in range(max_events):
        if len(finished) == len(roles) and not tma and not any(fifo.values()):
            return
        cands = [k for k in roles if k not in finished]
        if tma:
            cands.append("tma")
        cands += [f"{k}_mma" for k in fifo if fifo[k]]
        while cands:
            ev = rng.choices(cands, weights=[speed[c] for c in cands])[0]
            if fire(ev):
                break
            cands.remove(ev)
        else:
            stuck = {k: nxt[k] for k in roles if k not in finished}
            raise Violation(f"deadlock: {stuck}")
    raise Violation("did not finish")
