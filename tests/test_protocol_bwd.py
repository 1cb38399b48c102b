"""Model check of the dynamic backward's mbarrier protocols (d_h <= 64 and 128).

The dynamic backward kernel (attn_bwd.cu, bwd_dynamic_kernel, the path that
keeps P^T in TMEM and alternates two dS^T tiles in shared memory) runs a
producer (K_J, V_J once per item; Q_I, dO_I, lse, D per step in a ring of
three), an issuer of S^T and dP^T, an issuer of dV, dK and dQ, two compute
halves (both on every step, split by query columns) and the dQ warps.  This
file restates each role's waits, arrivals and commits and runs them under
random interleavings with the checker of protocol_model: every parity wait
must pass on exactly the awaited phase, no barrier may see more arrivals
than its count, and every role must finish.  A planted mistake (both dS^T
tiles released through one barrier) must be caught.

At d_h = 128 the kernel has no TMEM to spare: one warp issues every product,
P^T and dS^T go packed over the S^T columns the compute has read, and dQ
over the whole dP^T region.  dQ is staged for its reduce-adds in the step's
own Q/dO stage, once dV and dK have read it, and the dQ warps (not the
issuer) release the stage to the producer when the reduce-adds have read it.
The compute signals each of its two groups of query columns (p_full0,
p_full1): dV and dK take the first group's k-steps while the compute works on
the second.  The second model restates that path (QST = 2, dv_done / dk_done
/ dp_full / dq_empty), and three planted mistakes (the next dP^T issued
before dQ has left its columns; the dQ warps staging before dV has read dO;
the second group's products issued after the first group only) must be
caught.
Host logic only.
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
    for i, n in enumerate(items):
        yield ("wait", "kv_empty", kvc - 1)
        kvc += 1
        yield ("tma", "kv_full", "KV", f"kv{i}")
        for _ in range(n):
            qs = qc % QST
            yield ("wait", f"q_empty{qs}", qc // QST - 1)
            yield ("tma", f"q_full{qs}", f"Q{qs}", f"q{qc}")
            qc += 1


# Data regions (d_h <= 64): KV, Q{stage} in shared memory, DST{tile}h0/h1 (the
# halves' columns of a dS^T tile); in TMEM TS and TDP (S^T, dP^T, per half),
# TPT (P^T, per half), TDV, TDK, TDQ.
def halves(region, tag):
    return [(region + "h0", tag), (region + "h1", tag)]


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
            yield ("mma", [("KV", f"kv{idx}"), (f"Q{qs}", f"q{qc}")],
                   halves("TS", f"S{qc}") + halves("TDP", f"dP{qc}"))   # S^T, dP^T
            yield ("commit", "s_full")
            qc += 1


def grad_issuer(items, one_tile=False):
    kvc = qc = pc = dqc = kdc = 0
    for i, n in enumerate(items):
        yield ("wait", "kv_full", kvc)
        kvc += 1
        for t in range(n):
            qs = qc % QST
            u = qc
            tile = 0 if one_tile else (pc & 1)
            yield ("wait", "p_full", pc)
            if t == 0:
                yield ("wait", "kd_empty", kdc - 1)
            yield ("mma", halves("TPT", f"P{u}") + [(f"Q{qs}", f"q{u}")],
                   [("TDV", f"dv{i}.{t}")],
                   [("TDV", f"dv{i}.{t - 1}")] if t > 0 else [])     # dV from P^T in TMEM
            yield ("commit", "pt_empty")
            yield ("mma", halves(f"DST{pc & 1}", f"dS{u}") + [(f"Q{qs}", f"q{u}")],
                   [("TDK", f"dk{i}.{t}")],
                   [("TDK", f"dk{i}.{t - 1}")] if t > 0 else [])     # dK from the dS^T tile
            yield ("commit", f"q_empty{qs}")
            qc += 1
            yield ("wait", "dq_empty", dqc - 1)
            yield ("mma", halves(f"DST{pc & 1}", f"dS{u}") + [("KV", f"kv{i}")],
                   [("TDQ", f"dQ{u}")])                               # dQ
            yield ("commit", f"p_empty{tile}")
            pc += 1
            yield ("commit", "dq_full")
            dqc += 1
        yield ("commit", "kd_full")
        yield ("commit", "kv_empty")
        kdc += 1


def compute(hf, items, one_tile=False):
    qc = sc = pc = kdc = 0
    h = f"h{hf}"
    for i, n in enumerate(items):
        for t in range(n):
            qs = qc % QST
            u = qc
            yield ("wait", f"q_full{qs}", qc // QST)
            yield ("read", f"Q{qs}", f"q{u}")           # -lse, -D of the stage
            yield ("wait", "s_full", sc)
            yield ("read", "TS" + h, f"S{u}")
            yield ("read", "TDP" + h, f"dP{u}")
            # first chunk: P^T and the dS^T tile must be free
            yield ("wait", "pt_empty", pc - 1)
            # (planted: both tiles' releases land on one barrier, while the
            # wait keeps the per-tile phase count)
            tile = 0 if one_tile else (pc & 1)
            yield ("wait", f"p_empty{tile}", (pc >> 1) - 1)
            yield ("write", "TPT" + h, f"P{u}")
            yield ("write", f"DST{pc & 1}" + h, f"dS{u}")
            yield ("arrive", "s_free", 1)   # after the last chunk's loads
            yield ("arrive", "p_full", 1)
            qc += 1
            sc += 1
            pc += 1
        yield ("wait", "kd_full", kdc)
        yield ("read", "TDV" if hf == 0 else "TDK", f"{'dv' if hf == 0 else 'dk'}{i}.{n - 1}")
        yield ("arrive", "kd_empty", 1)
        kdc += 1


def dq_warps(items):
    dqc = 0
    for n in items:
        for _ in range(n):
            yield ("wait", "dq_full", dqc)
            yield ("read", "TDQ", f"dQ{dqc}")
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


# ------------------------------------------------------------ d_h = 128 path
QST128 = 2


def make_barriers_128():
    b = {}
    def add(name, count):
        b[name] = Barrier(name, count)
    add("kv_full", 1); add("kv_empty", 1)
    for s in range(QST128):
        add(f"q_full{s}", 3); add(f"q_empty{s}", 1)   # Q, dO and -lse/-D land
    add("s_full", 1); add("dp_full", 1)
    add("p_full0", 2); add("p_full1", 2)   # first / second group of each half done
    add("dq_full", 1)
    add("dq_empty", 1)                 # all of dQ taken from TMEM by the dQ warps
    add("kd_full", 1); add("kd_empty", 2)
    add("dv_done", 1); add("dk_done", 1)
    return b


def producer_128(items):
    kvc = qc = 0
    for i, n in enumerate(items):
        yield ("wait", "kv_empty", kvc - 1)
        kvc += 1
        yield ("tma", "kv_full", "KV", f"kv{i}")
        for _ in range(n):
            qs = qc % QST128
            yield ("wait", f"q_empty{qs}", qc // QST128 - 1)
            for part in ("Q", "O", "L"):
                yield ("tma", f"q_full{qs}", f"{part}{qs}", f"q{qc}")
            qc += 1


# A stage holds Q (region Q{s}), dO (O{s}) and the -lse/-D vectors (L{s}).
# TMEM regions.  Compute half h reads two groups of 32 query columns of S^T,
# g = a then b (TS{g}{h}), and the same groups of dP^T (TDP{g}{h}); into each
# S^T group it has read it writes its packed P^T (TS{g}{h}P, the group's first
# 16 columns) and dS^T (TS{g}{h}D, the other 16).  dQ then goes over the whole
# dP^T region.  DST{h} are the halves' columns of the shared dS^T tile.  Tags
# name the global step u.
def s_cols(tag):
    return [(f"TS{g}{h}{x}", tag) for g in "ab" for h in "01" for x in "PD"]


def dp_cols(tag):
    return [(f"TDP{g}{h}", tag) for g in "ab" for h in "01"]


def issuer_128(items, skip_dq_drain=False, skip_second_wait=False):
    kvc = qc = pc = dqc = kdc = dvc = dkc = 0

    def issue_st(q, i):
        yield ("wait", f"q_full{q % QST128}", q // QST128)
        yield ("mma", [("KV", f"kv{i}"), (f"Q{q % QST128}", f"q{q}")], s_cols(f"S{q}"))
        yield ("commit", "s_full")

    def issue_dpt(q, i):
        yield ("wait", f"q_full{q % QST128}", q // QST128)
        yield ("mma", [("KV", f"kv{i}"), (f"O{q % QST128}", f"q{q}")], dp_cols(f"dP{q}"))
        yield ("commit", "dp_full")

    for i, n in enumerate(items):
        yield ("wait", "kv_full", kvc)
        kvc += 1
        # the previous step's dV and dK have read P^T and dS^T (products of
        # this warp complete in issue order, so the wait is kept only to make
        # the order explicit), and dQ has left the dP^T columns
        if dkc > 0:
            yield ("wait", "dk_done", dkc - 1)
        yield from issue_st(qc, i)
        if dqc > 0 and not skip_dq_drain:
            yield ("wait", "dq_empty", dqc - 1)
        yield from issue_dpt(qc, i)
        for t in range(n):
            qs = qc % QST128
            u = qc
            # the k-steps of the first group of both halves (query columns
            # 0..63) while the compute works on the second
            yield ("wait", "p_full0", pc)
            if t == 0:
                yield ("wait", "kd_empty", kdc - 1)
            acc_v = [("TDV", f"dv{i}.{t - 1}")] if t > 0 else []
            acc_k = [("TDK", f"dk{i}.{t - 1}")] if t > 0 else []
            yield ("mma", [(f"TSa{h}P", f"P{u}") for h in "01"] + [(f"O{qs}", f"q{u}")],
                   [("TDV", f"dv{i}.{t}a")], acc_v)                      # dV, k-steps 0..3
            yield ("mma", [(f"TSa{h}D", f"dS{u}") for h in "01"] + [(f"Q{qs}", f"q{u}")],
                   [("TDK", f"dk{i}.{t}a")], acc_k)                      # dK, k-steps 0..3
            if not skip_second_wait:
                yield ("wait", "p_full1", pc)
            yield ("mma", [("DST0", f"dS{u}"), ("DST1", f"dS{u}"), ("KV", f"kv{i}")],
                   dp_cols(f"dQ{u}"))                           # dQ
            yield ("commit", "dq_full")
            dqc += 1
            yield ("mma", [(f"TSb{h}P", f"P{u}") for h in "01"] + [(f"O{qs}", f"q{u}")],
                   [("TDV", f"dv{i}.{t}")], [("TDV", f"dv{i}.{t}a")])   # dV, k-steps 4..7
            yield ("commit", "dv_done")
            dvc += 1
            yield ("mma", [(f"TSb{h}D", f"dS{u}") for h in "01"] + [(f"Q{qs}", f"q{u}")],
                   [("TDK", f"dk{i}.{t}")], [("TDK", f"dk{i}.{t}a")])   # dK, k-steps 4..7
            yield ("commit", "dk_done")
            dkc += 1
            # (the stage goes back to the producer from the dQ warps)
            qc += 1
            pc += 1
            if t + 1 < n:
                yield ("wait", "dk_done", dkc - 1)
                yield from issue_st(qc, i)
                if not skip_dq_drain:
                    yield ("wait", "dq_empty", dqc - 1)
                yield from issue_dpt(qc, i)
        yield ("commit", "kd_full")
        yield ("commit", "kv_empty")
        kdc += 1


def compute_128(hf, items):
    qc = sc = pc = kdc = 0
    h = f"{hf}"
    for i, n in enumerate(items):
        for _ in range(n):
            qs = qc % QST128
            u = qc
            yield ("wait", f"q_full{qs}", qc // QST128)
            yield ("read", f"L{qs}", f"q{u}")           # -lse, -D of the stage
            yield ("wait", "s_full", sc)
            for g in "ab":
                # P from this group of S^T, then dS from the same group of
                # dP^T; both packed over the S^T group just read
                yield ("read", f"TS{g}{h}P", f"S{u}")
                yield ("read", f"TS{g}{h}D", f"S{u}")
                yield ("write", f"TS{g}{h}P", f"P{u}")
                if g == "a":
                    yield ("wait", "dp_full", sc)
                yield ("read", f"TDP{g}{h}", f"dP{u}")
                yield ("write", f"TS{g}{h}D", f"dS{u}")
                # the previous step's dQ has read the dS^T tile: its commit
                # precedes this step's s_full, waited for above
                yield ("write", "DST" + h, f"dS{u}")
                yield ("arrive", f"p_full{0 if g == 'a' else 1}", 1)
            qc += 1
            sc += 1
            pc += 1
        yield ("wait", "kd_full", kdc)
        yield ("read", "TDV" if hf == 0 else "TDK", f"{'dv' if hf == 0 else 'dk'}{i}.{n - 1}")
        yield ("arrive", "kd_empty", 1)
        kdc += 1


def dq_warps_128(items, early_stage=False):
    dqc = 0
    u = 0
    for n in items:
        for _ in range(n):
            qs = u % QST128
            yield ("wait", "dq_full", dqc)
            # low 64 columns into registers, staged where dO was once dV
            # has read it (planted: not waited for)
            for g in "ab":
                yield ("read", f"TDP{g}0", f"dQ{u}")
            if not early_stage:
                yield ("wait", "dv_done", dqc)
            yield ("write", f"O{qs}", f"dQs{u}")
            # high 64 columns; all of dQ has then left TMEM.  Waiting for dK
            # first keeps dk_done from running two phases ahead of this wait.
            for g in "ab":
                yield ("read", f"TDP{g}1", f"dQ{u}")
            yield ("wait", "dk_done", dqc)
            yield ("arrive", "dq_empty", 1)
            yield ("write", f"Q{qs}", f"dQs{u}")
            # the tensor reduce-adds read the staged rows; then the stage
            # goes back to the producer
            yield ("read", f"O{qs}", f"dQs{u}")
            yield ("read", f"Q{qs}", f"dQs{u}")
            yield ("arrive", f"q_empty{qs}", 1)
            dqc += 1
            u += 1


def run_model_128(items, rng, skip_dq_drain=False, early_stage=False, skip_second_wait=False):
    roles = {
        "prod": producer_128(items), "g": issuer_128(items, skip_dq_drain, skip_second_wait),
        "c0": compute_128(0, items), "c1": compute_128(1, items),
        "dq": dq_warps_128(items, early_stage),
    }
    run_roles(roles, make_barriers_128(), ("g",), rng)


@pytest.mark.parametrize("seed", range(40))
def test_backward_128_protocol_holds(seed):
    rng = random.Random(1000 + seed)
    for _ in range(5):
        run_model_128(random_items(rng, rng.randint(1, 14)), rng)


def test_planted_skipped_dq_drain_is_caught():
    # The next step's dP^T issued without waiting for the dQ warps to take dQ
    # out of the dP^T columns: a dQ read then finds dP^T there, or the phases
    # of dq_empty run ahead of their waiter.
    rng = random.Random(17)
    caught = 0
    for _ in range(200):
        try:
            run_model_128(random_items(rng, rng.randint(2, 10)), rng, skip_dq_drain=True)
        except Violation:
            caught += 1
    assert caught >= 10


def test_planted_staging_before_dv_read_is_caught():
    # The dQ warps staging dQ over the stage before dV has read dO: a dV
    # product then reads staged dQ where it expects dO.
    rng = random.Random(23)
    caught = 0
    for _ in range(200):
        try:
            run_model_128(random_items(rng, rng.randint(2, 10)), rng, early_stage=True)
        except Violation:
            caught += 1
    assert caught >= 10


def test_planted_second_group_before_written_is_caught():
    # dQ and the second half of dV / dK issued after the first group only:
    # they read P^T / dS^T columns that still hold S^T.
    rng = random.Random(29)
    caught = 0
    for _ in range(200):
        try:
            run_model_128(random_items(rng, rng.randint(2, 10)), rng, skip_second_wait=True)
        except Violation:
            caught += 1
    assert caught >= 10
