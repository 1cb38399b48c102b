"""Model check of the forward kernel's mbarrier protocol at d_h = 128.

At d_h = 128 (and in the transposed static-dV engine) the forward keeps three
128-column TMEM buffers shared by dynamic and static steps: a dynamic step's
S (then P over it), a static step's generated tile.  Warp 1 issues the score
products, warp 3 every P V product; both compute halves work on every step
(split by key columns).  Every use of a buffer completes one phase of both of
its barriers (a static use through warp 3's commits), so the roles count uses
uniformly.  This file restates the roles and runs them under random
interleavings with the checker of protocol_model (parity waits on exactly the
awaited phase, no over-arrival, no deadlock, data versions of the buffers and
shared-memory slots).

The score issuer takes part in every use of every buffer: for a static step
it waits for the buffer's previous use and grants it (s_full), and the compute
halves generate into the buffer only after that grant.  The earlier protocol,
in which the score issuer passed over static steps (the compute waited on the
buffer itself), must be caught: at the next dynamic item the score issuer
could then wait on a buffer two phases early.  Host logic only.
"""

import random

import pytest

from protocol_model import Barrier, Violation, run_roles

NB, KST, VST, AST = 3, 2, 3, 4


def make_barriers():
    b = {}
    def add(name, count):
        b[name] = Barrier(name, count)
    add("q_full", 1); add("q_empty", 1)
    for s in range(KST):
        add(f"k_full{s}", 1); add(f"k_empty{s}", 1)
    for s in range(VST):
        add(f"v_full{s}", 1); add(f"v_empty{s}", 1)
    for s in range(NB):
        add(f"s_full{s}", 1); add(f"s_empty{s}", 1); add(f"p_full{s}", 2)
    for s in range(AST):
        add(f"aux_full{s}", 1); add(f"aux_empty{s}", 2)
    add("o_full", 1); add("o_empty", 2)
    return b


def buf(b, tag):
    return [(f"B{b}h0", tag), (f"B{b}h1", tag)]


def producer_qk(items):
    qc = kc = ac = 0
    for i, it in enumerate(items):
        if it["dyn"]:
            yield ("wait", "q_empty", qc - 1)
            qc += 1
            yield ("tma", "q_full", "Q", f"q{i}")
            for j in range(it["n"]):
                ks = kc % KST
                yield ("wait", f"k_empty{ks}", kc // KST - 1)
                kc += 1
                yield ("tma", f"k_full{ks}", f"K{ks}", f"k{i}.{j}")
        else:
            for step in range(it["n"]):
                a = ac % AST
                yield ("wait", f"aux_empty{a}", ac // AST - 1)
                ac += 1
                yield ("tma", f"aux_full{a}", f"A{a}", f"a{i}.{step}")


def producer_v(items):
    vc = 0
    for i, it in enumerate(items):
        for j in range(it["n"]):
            vs = vc % VST
            yield ("wait", f"v_empty{vs}", vc // VST - 1)
            vc += 1
            yield ("tma", f"v_full{vs}", f"V{vs}", f"v{i}.{j}")


def s_issuer(items, skip_static=False, old=False):
    qc = kc = sc = 0
    for i, it in enumerate(items):
        if it["dyn"]:
            yield ("wait", "q_full", qc)
            qc += 1
            for j in range(it["n"]):
                u = sc + j
                ks = kc % KST
                yield ("wait", f"k_full{ks}", kc // KST)
                yield ("wait", f"s_empty{u % NB}", u // NB - 1)
                yield ("mma", [("Q", f"q{i}"), (f"K{ks}", f"k{i}.{j}")], buf(u % NB, f"s{i}.{j}"))
                yield ("commit", f"k_empty{ks}")
                yield ("commit", f"s_full{u % NB}")
                if j == it["n"] - 1:
                    yield ("commit", "q_empty")
                kc += 1
        elif not skip_static and not old:
            # a static step's buffer: granted once its previous use is done,
            # so this issuer takes part in every use of every buffer
            for step in range(it["n"]):
                u = sc + step
                yield ("wait", f"s_empty{u % NB}", u // NB - 1)
                yield ("arrive", f"s_full{u % NB}", 1)
        sc += it["n"]


def pv_issuer(items, old=False):
    vc = sc = oc = 0
    for i, it in enumerate(items):
        for j in range(it["n"]):
            u = sc + j
            b = u % NB
            vs = vc % VST
            yield ("wait", f"p_full{b}", u // NB)
            if j == 0:
                yield ("wait", "o_empty", oc - 1)
            yield ("wait", f"v_full{vs}", vc // VST)
            tag = f"p{i}.{j}" if it["dyn"] else f"g{i}.{j}"
            yield ("mma", buf(b, tag) + [(f"V{vs}", f"v{i}.{j}")], [("O", f"o{i}.{j}")],
                   [("O", f"o{i}.{j - 1}")] if j > 0 else [])
            yield ("commit", f"v_empty{vs}")
            vc += 1
            if old and not it["dyn"]:
                yield ("commit", f"s_full{b}")
            yield ("commit", f"s_empty{b}")
        sc += it["n"]
        yield ("commit", "o_full")
        oc += 1


def compute(hf, items, old=False):
    sc = ac = oc = 0
    h = f"h{hf}"
    for i, it in enumerate(items):
        for j in range(it["n"]):
            u = sc + j
            b = u % NB
            if it["dyn"]:
                yield ("wait", f"s_full{b}", u // NB)
                yield ("read", f"B{b}" + h, f"s{i}.{j}")
                yield ("pair", (i, j))          # the halves swap row maxima
                if j > 0:
                    # a rescale of O waits for the previous P V product
                    yield ("wait", f"s_empty{(u - 1) % NB}", (u - 1) // NB)
                yield ("write", f"B{b}" + h, f"p{i}.{j}")
                yield ("arrive", f"p_full{b}", 1)
            else:
                a = ac % AST
                yield ("wait", f"aux_full{a}", ac // AST)
                yield ("read", f"A{a}", f"a{i}.{j}")
                if old:
                    yield ("wait", f"s_empty{b}", u // NB - 1)
                else:
                    yield ("wait", f"s_full{b}", u // NB)   # the score issuer's grant
                yield ("write", f"B{b}" + h, f"g{i}.{j}")
                yield ("pair", (i, j, "aux"))   # both halves have read the tables
                yield ("arrive", f"aux_empty{a}", 1)
                ac += 1
                yield ("arrive", f"p_full{b}", 1)
        sc += it["n"]
        yield ("pair", (i, "epi"))
        yield ("wait", "o_full", oc)
        yield ("read", "O", f"o{i}.{it['n'] - 1}")
        yield ("arrive", "o_empty", 1)
        oc += 1


def run_model(items, rng, old=False):
    """old: the earlier protocol (the score issuer passes over static steps,
    the compute waits on the buffer itself, warp 3 completes both phases)."""
    roles = {
        "qk": producer_qk(items), "v": producer_v(items),
        "s": s_issuer(items, skip_static=old, old=old), "pv": pv_issuer(items, old),
        "c0": compute(0, items, old), "c1": compute(1, items, old),
    }
    run_roles(roles, make_barriers(), ("s", "pv"), rng)


def random_items(rng, n_items):
    items = []
    for _ in range(n_items):
        if rng.random() < 0.35:
            items.append({"dyn": False, "n": rng.randint(1, 9)})
        else:
            items.append({"dyn": True, "n": rng.randint(1, 7)})
    return items


@pytest.mark.parametrize("seed", range(40))
def test_forward_128_protocol_holds(seed):
    rng = random.Random(500 + seed)
    for _ in range(5):
        run_model(random_items(rng, rng.randint(1, 14)), rng)


def test_earlier_protocol_is_caught():
    # The earlier protocol: the score issuer passed over static steps, so at
    # the next dynamic item it could wait on a buffer two phases early.
    rng = random.Random(41)
    caught = 0
    for _ in range(300):
        try:
            run_model(random_items(rng, rng.randint(2, 12)), rng, old=True)
        except Violation:
            caught += 1
    assert caught >= 10
