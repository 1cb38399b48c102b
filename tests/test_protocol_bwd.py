"""Model check of the dynamic backward's mbarrier protocol at d_h <= 64.

The dynamic backward kernel (attn_bwd.cu, bwd_dynamic_kernel, the path that
keeps P^T in TMEM and alternates two dS^T tiles in shared memory) runs a
producer (K_J, V_J once per item; Q_I, dO_I, lse, D per step in a ring of
three), an issuer of S^T and dP^T, an issuer of dV, dK and dQ, two compute
halves (both on every step, split by query columns) and the dQ warps.  This
file restates each role's waits, arrivals and commits and runs them under
random interleavings with the checker of protocol_model: every parity wait
must pass on exactly the awaited phase, no barrier may see more arrivals
than its count, and every role must finish.  A planted mistake (both dS^T
tiles released through one barrier) must be caught.  Host logic only.
"""

import random

import pytest

from protocol_model import Barrier, Violation, run_roles

QST = 3


def make_barriers():
    b = {}
    def add(name, count):
        b[name] = Barrier(name, count)
    add("kv_full", 1); add("kv_empty", 1)
    for s in range(QST):
        add(f"q_full{s}", 1); add(f"q_empty{s}", 1)
    add("s_full", 1)
    add("p_full", 2)        # both halves (256 threads)
    add("p_empty0", 1); add("p_empty1", 1)
    add("dq_full", 1); add("dq_empty", 1)   # the dQ warps (128 threads)
    add("kd_full", 1); add("kd_empty", 2)
    add("s_free", 2)
    add("pt_empty", 1)
    return b


def producer(items):
    kvc = qc = 0
    for n in items:
        yield ("wait", "kv_empty", kvc - 1)
        kvc += 1
        yield ("tma", "kv_full")
        for _ in range(n):
            qs = qc % QST
            yield ("wait", f"q_empty{qs}", qc // QST - 1)
            qc += 1
            yield ("tma", f"q_full{qs}")


def s_issuer(items):
    kvc = qc = sfc = 0
    for idx, n in enumerate(items):
        yield ("wait", "kv_full", kvc)
        kvc += 1
        if idx > 0:   # the previous item's last scores have been loaded
            yield ("wait", "s_free", sfc)
            sfc += 1
        for t in range(n):
            if t > 0:
                yield ("wait", "s_free", sfc)
                sfc += 1
            qs = qc % QST
            yield ("wait", f"q_full{qs}", qc // QST)
            yield ("mma",)            # S^T, dP^T
            yield ("commit", "s_full")
            qc += 1


def grad_issuer(items, one_tile=False):
    kvc = qc = pc = dqc = kdc = 0
    for n in items:
        yield ("wait", "kv_full", kvc)
        kvc += 1
        for t in range(n):
            qs = qc % QST
            yield ("wait", "p_full", pc)
            if t == 0:
                yield ("wait", "kd_empty", kdc - 1)
            yield ("mma",)            # dV from P^T in TMEM
            yield ("commit", "pt_empty")
            yield ("mma",)            # dK from the dS^T tile
            yield ("commit", f"q_empty{qs}")
            qc += 1
            yield ("wait", "dq_empty", dqc - 1)
            yield ("mma",)            # dQ from the dS^T tile
            yield ("commit", "p_empty0" if one_tile or not (pc & 1) else "p_empty1")
            pc += 1
            yield ("commit", "dq_full")
            dqc += 1
        yield ("commit", "kd_full")
        yield ("commit", "kv_empty")
        kdc += 1


def compute(hf, items, one_tile=False):
    qc = sc = pc = kdc = 0
    for idx, n in enumerate(items):
        for t in range(n):
            qs = qc % QST
            yield ("wait", f"q_full{qs}", qc // QST)
            yield ("wait", "s_full", sc)
            # first chunk: P^T and the dS^T tile must be free
            yield ("wait", "pt_empty", pc - 1)
            # (planted: both tiles' releases land on one barrier, while the
            # wait keeps the per-tile phase count)
            tile = 0 if one_tile else (pc & 1)
            yield ("wait", f"p_empty{tile}", (pc >> 1) - 1)
            yield ("arrive", "s_free", 1)   # after the last chunk's loads
            yield ("arrive", "p_full", 1)
            qc += 1
            sc += 1
            pc += 1
        yield ("wait", "kd_full", kdc)
        yield ("arrive", "kd_empty", 1)
        kdc += 1


def dq_warps(items):
    dqc = 0
    for n in items:
        for _ in range(n):
            yield ("wait", "dq_full", dqc)
            yield ("arrive", "dq_empty", 1)
            dqc += 1


def run_model(items, rng, one_tile=False):
    roles = {
        "prod": producer(items), "s": s_issuer(items), "g": grad_issuer(items, one_tile),
        "c0": compute(0, items, one_tile), "c1": compute(1, items, one_tile),
        "dq": dq_warps(items),
    }
    run_roles(roles, make_barriers(), ("s", "g"), rng)


def random_items(rng, n_items):
    return [rng.randint(1, 7) for _ in range(n_items)]


@pytest.mark.parametrize("seed", range(40))
def test_backward_protocol_holds(seed):
    rng = random.Random(seed)
    for _ in range(5):
        run_model(random_items(rng, rng.randint(1, 14)), rng)


def test_planted_shared_tile_barrier_is_caught():
    # Both dS^T tiles released through one barrier while each wait still
    # counts that tile's own uses: the barrier runs two phases per tile use,
    # so a wait meets a phase it did not expect.  (The kernel gives each tile
    # its own barrier.)
    rng = random.Random(5)
    caught = 0
    for _ in range(200):
        try:
            run_model(random_items(rng, rng.randint(2, 10)), rng, one_tile=True)
        except Violation:
            caught += 1
    assert caught >= 10
