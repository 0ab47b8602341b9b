"""CPU model of the barrier protocol of the dQ kernel (fine_bwd_dq_kernel).

Roles, as in the kernel: a TMA producer (Q and dO once; K(j) into stage
j % 3, one step ahead, then V(j) into the single V stage), one MMA-issuing
thread, and two compute warpgroups (one per key cube of a step).  Barriers:
  bar_qdo       Q, dO landed                      (TMA)
  bar_k[s]      K stage s landed                  (TMA)
  bar_kvfree[s] dQ(j) that read K stage s done    (commit)
  bar_v         the V stage landed                (TMA)
  bar_vfree     dP(j) that read V done            (commit)
  s_done        S(j) and dP(j) done               (commit after dP(j))
  s_free        S(j), dP(j) read into registers   (all compute threads)
  bar_ds[b]     dS(j) written into buffer b = j % 2   (all compute threads)
  ds_free[b]    dQ(j) that read buffer b done     (commit)
S(j) is issued once S(j-1) and dP(j-1) are read and K(j) landed; dP(j) after
S(j) once V(j) landed; dQ(j) once dS(j) is written.  The model asserts the
parity rule at every test, that no K or V stage, S/dP buffer or dS buffer is
overwritten before its last reader is done, that each product reads the
operands of its own step, and that every schedule terminates.
"""
import random

import pytest

KSTAGES = 3


def delay(rnd, hi):
    """Mostly short, sometimes long: a late TMA tile or a slow MMA group."""
    return rnd.randint(1, hi) if rnd.random() < 0.85 else rnd.randint(4 * hi, 12 * hi)


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.arrived, self.phases = name, count, 0, 0

    def arrive(self, n=1):
        self.arrived += n
        assert self.arrived <= self.count, self.name
        if self.arrived == self.count:
            self.arrived = 0
            self.phases += 1

    def test(self, k):
        assert k <= self.phases <= k + 1, (self.name, k, self.phases)
        return self.phases > k


def simulate(steps, seed, max_ticks=400000, drop=(), stall=0.1):
    """drop: waits left out on purpose (to show the model catches them);
    stall: how often the issuing thread stalls."""
    rnd = random.Random(seed)
    bar_qdo = Barrier("bar_qdo", 1)
    bar_k = [Barrier(f"bar_k{i}", 1) for i in range(KSTAGES)]
    kvfree = [Barrier(f"kvfree{i}", 1) for i in range(KSTAGES)]
    bar_v, vfree = Barrier("bar_v", 1), Barrier("vfree", 1)
    s_done, s_free = Barrier("s_done", 1), Barrier("s_free", 2)
    bar_ds = [Barrier(f"bar_ds{i}", 2) for i in range(2)]
    ds_free = [Barrier(f"ds_free{i}", 1) for i in range(2)]

    kring = [None] * KSTAGES     # stage -> [step, read by dQ]
    vstage = None                # [step, read by dP]
    s_buf = None                 # [step, warpgroups that read S and dP]
    ds_buf = [None, None]        # buffer -> [step, warpgroups that wrote it, read by dQ]
    pipe, loads = [], []

    prog = [("QdO", -1), ("K", 0)] if steps else []
    for j in range(steps):
        if j + 1 < steps:
            prog.append(("K", j + 1))
        prog.append(("V", j))
    pc = 0
    qdo_ok = False
    ns = npd = ng = 0
    comp_j = [0, 0]
    comp_pc = [0, 0]             # 0 wait S/dP, 1 write dS
    issuer_busy = 0              # the issuing thread shares its sub-partition: it stalls at times

    for tick in range(max_ticks):
        if pipe:                                     # tensor pipe, in order
            pipe[0][2] -= 1
            if pipe[0][2] <= 0:
                kind, j, _, bars = pipe.pop(0)
                if kind == "S":
                    assert kring[j % KSTAGES] is not None and kring[j % KSTAGES][0] == j, ("K for S", kring, j)
                    assert s_buf is None or s_buf[1] == {0, 1}, ("S/dP overwritten unread", s_buf, j)
                    s_buf = [j, set()]
                elif kind == "dP":
                    assert vstage is not None and vstage[0] == j, ("V for dP", vstage, j)
                    assert s_buf is not None and s_buf[0] == j
                    vstage[1] = True
                else:
                    b = j & 1
                    assert kring[j % KSTAGES] is not None and kring[j % KSTAGES][0] == j, ("K for dQ", kring, j)
                    assert ds_buf[b] is not None and ds_buf[b][0] == j and ds_buf[b][1] == {0, 1}, \
                        ("dQ reads incomplete dS", ds_buf[b], j)
                    kring[j % KSTAGES][1] = True
                    ds_buf[b][2] = True
                for bar in bars:
                    bar.arrive()
        for ld in list(loads):                       # TMA completions
            ld[2] -= 1
            if ld[2] <= 0:
                loads.remove(ld)
                kind, j = ld[0], ld[1]
                if kind == "QdO":
                    bar_qdo.arrive()
                elif kind == "K":
                    st = j % KSTAGES
                    assert kring[st] is None or kring[st][1], ("K stage overwritten before dQ read it", kring[st], j)
                    kring[st] = [j, False]
                    bar_k[st].arrive()
                else:
                    assert vstage is None or vstage[1], ("V stage overwritten before dP read it", vstage, j)
                    vstage = [j, False]
                    bar_v.arrive()
        if pc < len(prog) and rnd.random() < 0.5:    # producer
            kind, j = prog[pc]
            ready = True
            if kind == "K" and j >= KSTAGES and "kvfree" not in drop:
                ready = kvfree[j % KSTAGES].test(j // KSTAGES - 1)
            if kind == "V" and j >= 1 and "vfree" not in drop:
                ready = vfree.test(j - 1)
            if ready:
                loads.append([kind, j, delay(rnd, 10)])
                pc += 1
        if issuer_busy:
            issuer_busy -= 1
        elif steps and rnd.random() < 0.7:           # issuer
            if rnd.random() < stall:
                issuer_busy = delay(rnd, 4)
            if not qdo_ok:
                qdo_ok = bar_qdo.test(0)
            else:
                if ns < steps and ns == npd and (ns == 0 or "s_free" in drop or s_free.test(ns - 1)) and \
                        bar_k[ns % KSTAGES].test(ns // KSTAGES):
                    pipe.append(["S", ns, delay(rnd, 6), []])
                    ns += 1
                if npd < ns and bar_v.test(npd):
                    pipe.append(["dP", npd, delay(rnd, 6), [s_done, vfree]])
                    npd += 1
                if ng < npd and bar_ds[ng & 1].test(ng >> 1):
                    pipe.append(["dQ", ng, delay(rnd, 6), [kvfree[ng % KSTAGES], ds_free[ng & 1]]])
                    ng += 1
        for g in range(2):                           # compute warpgroups
            j = comp_j[g]
            if j >= steps or rnd.random() > 0.4:
                continue
            if comp_pc[g] == 0:
                if s_done.test(j):
                    assert s_buf is not None and s_buf[0] == j, ("S/dP buffer", s_buf, j)
                    s_buf[1].add(g)
                    s_free.arrive()
                    comp_pc[g] = 1
            else:
                b = j & 1
                if j < 2 or "ds_free" in drop or ds_free[b].test((j >> 1) - 1):
                    if ds_buf[b] is not None and ds_buf[b][0] != j:
                        assert ds_buf[b][2], ("dS overwritten before dQ read it", ds_buf[b], j)
                        ds_buf[b] = None
                    if ds_buf[b] is None:
                        ds_buf[b] = [j, set(), False]
                    ds_buf[b][1].add(g)
                    bar_ds[b].arrive()
                    comp_j[g] += 1
                    comp_pc[g] = 0
        if steps == 0:
            return tick
        if ng == steps and not pipe and comp_j == [steps, steps]:
            assert ds_free[(steps - 1) & 1].test((steps - 1) >> 1)   # epilogue wait
            return tick
    raise AssertionError(f"no progress: steps={steps} seed={seed} ns={ns} npd={npd} ng={ng} comp={comp_j}")


@pytest.mark.parametrize("steps", [0, 1, 2, 3, 4, 5, 7, 12, 31, 77])
def test_dq_protocol_random_schedules(steps):
    for seed in range(25):
        simulate(steps, seed)


@pytest.mark.parametrize("drop,steps,stall,seeds", [("kvfree", 12, 0.1, 60), ("vfree", 12, 0.1, 60),
                                                    ("s_free", 12, 0.1, 60), ("ds_free", 3, 0.7, 400)])
def test_model_catches_each_missing_wait(drop, steps, stall, seeds):
    """Leaving out any one of the waits makes some schedule fail.  The wait
    for dQ(j - 2) before dS(j) is written is implied by the K ring on every
    step but the last (V(j) is requested after K(j + 1), which reuses the K
    stage of step j - 2 and so waits for dQ(j - 2)); on the last step only
    that wait keeps dS(j) from overwriting dS(j - 2), and it takes a slow
    issuer to expose it."""
    caught = 0
    for seed in range(seeds):
        try:
            simulate(steps, seed, max_ticks=50000, drop=(drop,), stall=stall)
        except AssertionError:
            caught += 1
    assert caught > 0, drop
