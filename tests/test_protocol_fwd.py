"""Model check of the forward kernel's mbarrier protocol at d_h <= 64.

The fused forward at d_h <= 64 runs seven roles over shared rings: a Q/K and
table producer, a V producer, two MMA issuers, two compute halves and the
asynchronous engines (TMA loads that land in any order, tensor-core products
that complete in issue order per issuing thread, their commits arriving after
every earlier product of that thread).  This file restates, role by role, the
waits, arrivals and commits the kernel performs (attn_fwd.cu, hybrid_fwd_kernel
with SPLIT) and runs them under random interleavings.

An mbarrier parity wait passes when the barrier's current phase parity differs
from the awaited one.  Such a wait is only right if, when it passes, exactly
the awaited phase has completed: one phase fewer (the waiter ran two phases
ahead) passes spuriously, one more (the waiter fell two behind) would block
on the wrong phase.  The checker asserts this at every wait, forbids arrivals
beyond a barrier's count, and requires every role to finish (no deadlock).

Two planted mistakes, both once in the kernel, must be caught: the S buffers
shared by both halves and chosen by the parity of a global tile count, and
the issuer of static products waiting on a P buffer before the previous
item's O.  Host logic only: no GPU.
"""

import random

import pytest

from protocol_model import Barrier, Violation, run_roles

QST, KST, VST, AST = 2, 4, 4, 4


def make_barriers(shared_s):
    b = {}
    def add(name, count):
        b[name] = Barrier(name, count)
    for s in range(QST):
        add(f"q_full{s}", 1); add(f"q_empty{s}", 2)
    for s in range(KST):
        add(f"k_full{s}", 1); add(f"k_empty{s}", 1)
    for s in range(VST):
        add(f"v_full{s}", 1); add(f"v_empty{s}", 1)
    for s in range(2):
        add(f"s_full{s}", 1); add(f"s_empty{s}", 1)   # one unit = a half's 128 threads
        add(f"p_full{s}", 2); add(f"p_empty{s}", 1)   # two units = 256 threads
    for s in range(AST):
        add(f"aux_full{s}", 1); add(f"aux_empty{s}", 2)
    add("o_full", 2); add("o_empty", 2)
    return b


# --------------------------------------------------------------- the roles
# Each role is a generator of actions (see protocol_model).  Data regions:
# Q{slot}, K{slot}, V{slot}, A{slot} (tables) in shared memory; S{g} (a half's
# S buffer), P{b}h0 / P{b}h1 (the two halves' columns of a P buffer), O0, O1
# in TMEM.  Tags name the item i and its key tile j (or static step).

def producer_qk(items):
    qc = ac = 0
    kn = [0, 0]
    for i, it in enumerate(items):
        if it["dyn"]:
            qs = qc % QST
            yield ("wait", f"q_empty{qs}", qc // QST - 1)
            qc += 1
            yield ("tma", f"q_full{qs}", f"Q{qs}", f"q{i}")
            for j in range(it["n"]):
                r = j & 1
                n = kn[r]
                kn[r] += 1
                slot = 2 * r + (n & 1)
                yield ("wait", f"k_empty{slot}", (n >> 1) - 1)
                yield ("tma", f"k_full{slot}", f"K{slot}", f"k{i}.{j}")
        else:
            for step in range(it["n"]):
                a = ac % AST
                yield ("wait", f"aux_empty{a}", ac // AST - 1)
                ac += 1
                yield ("tma", f"aux_full{a}", f"A{a}", f"a{i}.{step}")


def producer_v(items):
    vc = 0
    for i, it in enumerate(items):
        if it["dyn"]:
            for j in range(it["n"]):
                vs = vc % VST
                yield ("wait", f"v_empty{vs}", vc // VST - 1)
                vc += 1
                yield ("tma", f"v_full{vs}", f"V{vs}", f"v{i}.{j}")
        else:
            for step in range(it["n"]):
                if it["nb"] == 2 and (vc & 1):
                    vs = vc % VST
                    yield ("wait", f"v_empty{vs}", vc // VST - 1)
                    vc += 1
                    yield ("arrive", f"v_full{vs}", 1)
                for bb in range(it["nb"]):
                    vs = vc % VST
                    yield ("wait", f"v_empty{vs}", vc // VST - 1)
                    vc += 1
                    yield ("tma", f"v_full{vs}", f"V{vs}", f"v{i}.{step}.{bb}")


def pbuf(b, tag):
    return [(f"P{b}h0", tag), (f"P{b}h1", tag)]


def issuer(g, items, shared_s, late_o=False):
    qc = vc = sc = oc = kn = sn = ss = 0
    for i, it in enumerate(items):
        o_ready = [False]

        def wait_o():
            if not o_ready[0]:
                o_ready[0] = True
                yield ("wait", "o_empty", oc - 1)

        if it["dyn"]:
            n = it["n"]
            qs = qc % QST
            yield ("wait", f"q_full{qs}", qc // QST)
            qc += 1

            def issue_s(j):
                nonlocal kn, sn
                slot = 2 * g + (kn & 1)
                yield ("wait", f"k_full{slot}", kn >> 1)
                if shared_s:   # planted mistake: buffer by the parity of a global count
                    us = ss + j
                    yield ("wait", f"s_empty{us & 1}", (us >> 1) - 1)
                    buf = us & 1
                else:
                    yield ("wait", f"s_empty{g}", sn - 1)
                    buf = g
                yield ("mma", [(f"Q{qs}", f"q{i}"), (f"K{slot}", f"k{i}.{j}")],
                       [(f"S{buf}", f"s{i}.{j}")])
                yield ("commit", f"k_empty{slot}")
                yield ("commit", f"s_full{buf}")
                kn += 1
                sn += 1

            def issue_pv(j):
                u = sc + j
                vq = vc + j
                yield ("wait", f"v_full{vq % VST}", vq // VST)
                yield ("wait", f"p_full{u & 1}", u >> 1)
                acc = [(f"O{g}", f"o{i}.{j - 2}r")] if j > 1 else []
                yield ("mma", pbuf(u & 1, f"p{i}.{j}") + [(f"V{vq % VST}", f"v{i}.{j}")] + acc,
                       [(f"O{g}", f"o{i}.{j}")])
                yield ("commit", f"v_empty{vq % VST}")
                yield ("commit", f"p_empty{u & 1}")

            if g < n:
                yield from issue_s(g)
            for j in range(g, n, 2):
                if j + 2 < n:
                    yield from issue_s(j + 2)
                yield from wait_o()
                yield from issue_pv(j)
            yield ("commit", f"q_empty{qs}")
            vc += n
            ss += n
        else:
            outs = ["O0", "O1"][: it["nb"]]
            for step in range(it["n"]):
                u = sc + step
                if g == 1:
                    if it["nb"] == 2 and (vc & 1):
                        vc += 1
                    vc += it["nb"]
                    continue
                if late_o:   # planted mistake: the static P wait before the O wait
                    yield ("wait", f"p_full{u & 1}", u >> 1)
                    yield from wait_o()
                else:
                    yield from wait_o()
                    yield ("wait", f"p_full{u & 1}", u >> 1)
                # the group's O chain: products of this issuer, in order
                acc = [(o, f"st{i}.{step - 1}") for o in outs] if step > 0 else []
                writes = [(o, f"st{i}.{step}") for o in outs]
                if it["nb"] == 2:
                    if vc & 1:
                        yield ("wait", f"v_full{vc % VST}", vc // VST)
                        yield ("commit", f"v_empty{vc % VST}")
                        vc += 1
                    yield ("wait", f"v_full{vc % VST}", vc // VST)
                    yield ("wait", f"v_full{(vc + 1) % VST}", (vc + 1) // VST)
                    yield ("mma", pbuf(u & 1, f"g{i}.{step}") +
                           [(f"V{vc % VST}", f"v{i}.{step}.0"),
                            (f"V{(vc + 1) % VST}", f"v{i}.{step}.1")], writes, acc)
                    yield ("commit", f"v_empty{vc % VST}")
                    yield ("commit", f"v_empty{(vc + 1) % VST}")
                    vc += 2
                else:
                    yield ("wait", f"v_full{vc % VST}", vc // VST)
                    yield ("mma", pbuf(u & 1, f"g{i}.{step}") +
                           [(f"V{vc % VST}", f"v{i}.{step}.0")], writes, acc)
                    yield ("commit", f"v_empty{vc % VST}")
                    vc += 1
                yield ("commit", f"p_empty{u & 1}")
        sc += it["n"]
        yield from wait_o()
        yield ("commit", "o_full")
        oc += 1


def compute(hf, items, shared_s):
    ac = sc = oc = sn = ss = 0
    for i, it in enumerate(items):
        sc0 = sc
        n = it["n"]
        if it["dyn"]:
            for j in range(hf, n, 2):
                u = sc0 + j
                if shared_s:
                    us = ss + j
                    sb, ph = us & 1, us >> 1
                else:
                    sb, ph = hf, sn
                yield ("wait", f"s_full{sb}", ph)
                sn += 1
                yield ("read", f"S{sb}", f"s{i}.{j}")
                yield ("arrive", f"s_empty{sb}", 1)
                yield ("wait", f"p_empty{u & 1}", (u >> 1) - 1)
                yield ("write", f"P{u & 1}h0", f"p{i}.{j}")
                yield ("write", f"P{u & 1}h1", f"p{i}.{j}")
                if j > 1:   # a rescale of this half's O, in place
                    yield ("read", f"O{hf}", f"o{i}.{j - 2}")
                    yield ("write", f"O{hf}", f"o{i}.{j - 2}r")
                yield ("arrive", f"p_full{u & 1}", 2)
            ss += n
            reads = [("O0", f"o{i}.{(n - 1) // 2 * 2}")]
            if n > 1:
                reads.append(("O1", f"o{i}.{(n - 2) // 2 * 2 + 1}"))
        else:
            for step in range(n):
                u = sc0 + step
                a = ac % AST
                yield ("wait", f"aux_full{a}", ac // AST)
                yield ("read", f"A{a}", f"a{i}.{step}")
                yield ("wait", f"p_empty{u & 1}", (u >> 1) - 1)
                yield ("write", f"P{u & 1}h{hf}", f"g{i}.{step}")
                yield ("arrive", f"aux_empty{a}", 1)
                ac += 1
                yield ("arrive", f"p_full{u & 1}", 1)
            reads = [(o, f"st{i}.{n - 1}") for o in ["O0", "O1"][: it["nb"]]]
        sc = sc0 + n
        yield ("pair", i)   # the halves' max/sum exchange (named barriers)
        yield ("wait", "o_full", oc)
        for r, tag in reads:
            yield ("read", r, tag)
        yield ("arrive", "o_empty", 1)
        oc += 1


def run_model(items, rng, shared_s=False, late_o=False):
    roles = {
        "qk": producer_qk(items), "v": producer_v(items),
        "i0": issuer(0, items, shared_s, late_o), "i1": issuer(1, items, shared_s, late_o),
        "c0": compute(0, items, shared_s), "c1": compute(1, items, shared_s),
    }
    run_roles(roles, make_barriers(shared_s), ("i0", "i1"), rng)


def random_items(rng, n_items):
    items = []
    for _ in range(n_items):
        if rng.random() < 0.3:
            items.append({"dyn": False, "n": rng.randint(1, 6), "nb": rng.choice([1, 2, 2])})
        else:
            items.append({"dyn": True, "n": rng.randint(1, 7)})
    return items


@pytest.mark.parametrize("seed", range(40))
def test_forward_protocol_holds(seed):
    rng = random.Random(seed)
    for _ in range(5):
        run_model(random_items(rng, rng.randint(1, 14)), rng)


def test_planted_shared_s_buffers_are_caught():
    # The earlier protocol: both halves share the two S buffers, picked by the
    # parity of a global tile count, so the halves swap buffers after an
    # odd-length item.  Some interleaving must make a wait pass early.
    rng = random.Random(1234)
    caught = 0
    for _ in range(200):
        try:
            run_model(random_items(rng, rng.randint(2, 10)), rng, shared_s=True)
        except Violation:
            caught += 1
    assert caught >= 10


def test_planted_late_o_wait_is_caught():
    # Issuer 0 waits on a static step's P buffer before the previous item's O
    # has been read: the buffer's older use may belong to the other half's
    # last tile of a dynamic item that is not written yet.
    rng = random.Random(99)
    caught = 0
    for _ in range(200):
        try:
            run_model(random_items(rng, rng.randint(2, 12)), rng, late_o=True)
        except Violation:
            caught += 1
    assert caught >= 10


def test_long_odd_item_runs():
    # the prefill shape: runs of one- and three-tile items, static groups between
    rng = random.Random(7)
    for _ in range(20):
        items = []
        for _ in range(12):
            items.append({"dyn": True, "n": rng.choice([1, 3, 5])})
            if rng.random() < 0.3:
                items.append({"dyn": False, "n": rng.choice([1, 2, 3]), "nb": 2})
        run_model(items, rng)
