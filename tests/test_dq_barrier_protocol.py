"""CPU model of the barrier protocol of the dQ kernel (fine_bwd_dq_kernel).

Roles, as in the kernel: a TMA producer (Q once, a 3-stage K ring, a 2-stage
V ring), two MMA-issuing threads (one issues S(j) then dP(j), the other
dQ(j)), and two compute warpgroups, which first write dO into TMEM (the A
operand of dP).  One S / dP buffer in TMEM is
released as soon as both warpgroups have read it into registers; dS(j) goes
into the single dS buffer once dQ(j - 1) has read it.  The barriers:
  bar_dot       dO written into TMEM                (both warpgroups -> issuer)
  bar_k[s]      K stage s landed                    (TMA -> issuer)
  bar_kvfree[s] dQ of the step in K stage s done    (commit -> producer)
  bar_v[s]      V stage s landed                    (TMA -> issuer)
  bar_vfree[s]  dP of the step in V stage s done    (commit -> producer)
  s_done        S(j), dP(j) done                    (commit -> compute)
  s_free        S(j), dP(j) read                    (both warpgroups -> issuer: S(j+1))
  bar_ds        dS(j) written                       (both warpgroups -> issuer: dQ(j))
  ds_free       dQ(j) done                          (commit -> compute: dS(j+1))
A parity wait for phase k is only correct while the barrier has completed k
or k + 1 phases; the model asserts that at every test, that no buffer or ring
stage is overwritten before its last reader is done, that every product reads
the step it belongs to, and that every schedule of random delays terminates.
The MMA groups of one issuing thread complete in the order issued; nothing
orders the two threads' groups, so the model runs them as two independent
queues.
"""
import random

import pytest

K_STAGES, V_STAGES = 3, 2


def delay(rnd, hi):
    """Mostly short, sometimes long: a late TMA tile or a slow MMA group."""
    return rnd.randint(1, hi) if rnd.random() < 0.85 else rnd.randint(4 * hi, 12 * hi)


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.arrived, self.phases = name, count, 0, 0

    def arrive(self):
        self.arrived += 1
        assert self.arrived <= self.count, self.name
        if self.arrived == self.count:
            self.arrived = 0
            self.phases += 1

    def test(self, k):
        """True once phase k has completed (mbarrier.test_wait.parity k & 1)."""
        assert k <= self.phases <= k + 1, (self.name, k, self.phases)
        return self.phases > k


def simulate(steps, seed, max_ticks=200000, drop=()):
    """drop: waits left out on purpose (to show the model catches them)."""
    rnd = random.Random(seed)
    bar_dot = Barrier("bar_dot", 2)
    bar_k = [Barrier(f"bar_k{i}", 1) for i in range(K_STAGES)]
    kvfree = [Barrier(f"kvfree{i}", 1) for i in range(K_STAGES)]
    bar_v = [Barrier(f"bar_v{i}", 1) for i in range(V_STAGES)]
    vfree = [Barrier(f"vfree{i}", 1) for i in range(V_STAGES)]
    s_done, s_free = Barrier("s_done", 1), Barrier("s_free", 2)
    bar_ds, ds_free = Barrier("bar_ds", 2), Barrier("ds_free", 1)
    kring = [None] * K_STAGES   # stage -> [step, read by dQ]
    vring = [None] * V_STAGES   # stage -> [step, read by dP]
    sbuf = None                 # ("S", j) after S(j) and dP(j); ("read", j) once both warpgroups read it
    dsbuf = None                # ("dS", j) once both warpgroups wrote it; ("read", j) after dQ(j)
    dot = 0                     # warpgroups that wrote dO
    read_by, wrote = {}, {}
    pipes, loads = {"A": [], "B": []}, []
    kload = vload = ns = npd = ng = 0
    computed = [0, 0]
    phase = [-1, -1]            # per warpgroup: -1 = write dO, 0 = read S/dP(j), 1 = write dS(j)
    for tick in range(max_ticks):
        for pipe in pipes.values():
            if not pipe or rnd.random() < 0.3:
                continue
            pipe[0][2] -= 1
            if pipe[0][2] <= 0:
                kind, j, _, bars = pipe.pop(0)
                if kind == "S":
                    assert kring[j % K_STAGES] is not None and kring[j % K_STAGES][0] == j, ("K", j)
                    assert sbuf is None or sbuf == ("read", j - 1), ("S overwritten before read", sbuf, j)
                    sbuf = ("S only", j)
                elif kind == "P":
                    assert dot == 2, "dP before dO was in TMEM"
                    assert vring[j % V_STAGES] is not None and vring[j % V_STAGES][0] == j, ("V", j)
                    assert sbuf == ("S only", j), ("dP without its S", sbuf, j)
                    vring[j % V_STAGES][1] = True
                    sbuf = ("S", j)
                else:
                    assert dsbuf == ("dS", j), (dsbuf, j)
                    assert kring[j % K_STAGES][0] == j
                    kring[j % K_STAGES][1] = True
                    dsbuf = ("read", j)
                for bar in bars:
                    bar.arrive()
        for load in list(loads):
            load[1] -= 1
            if load[1] <= 0:
                loads.remove(load)
                ring, st, j, bar = load[0], load[2], load[3], load[4]
                slot = (kring if ring == "K" else vring)
                assert slot[st] is None or slot[st][1], (ring + " stage overwritten before its reader", slot[st], j)
                slot[st] = [j, False]
                bar.arrive()
        if rnd.random() < 0.5:                       # producer: V(j), then K(j + 1)
            if vload < steps and vload <= kload - 1:
                st = vload % V_STAGES
                if vload < V_STAGES or "vfree" in drop or vfree[st].test(vload // V_STAGES - 1):
                    loads.append(["V", delay(rnd, 8), st, vload, bar_v[st]])
                    vload += 1
            elif kload < steps and kload <= vload:
                st = kload % K_STAGES
                if kload < K_STAGES or "kvfree" in drop or kvfree[st].test(kload // K_STAGES - 1):
                    loads.append(["K", delay(rnd, 8), st, kload, bar_k[st]])
                    kload += 1
        if rnd.random() < 0.7 and bar_dot.phases >= 1:  # issuer A: S(j), then dP(j)
            if ns < steps and ns == npd and (ns == 0 or "s_free" in drop or s_free.test(ns - 1)) and \
                    bar_k[ns % K_STAGES].test(ns // K_STAGES):
                pipes["A"].append(["S", ns, delay(rnd, 5), []])
                ns += 1
            elif npd < ns and bar_v[npd % V_STAGES].test(npd // V_STAGES):
                pipes["A"].append(["P", npd, delay(rnd, 5), [s_done, vfree[npd % V_STAGES]]])
                npd += 1
        if rnd.random() < 0.7 and ng < steps and bar_ds.test(ng):  # issuer B: dQ(j)
            pipes["B"].append(["Q", ng, delay(rnd, 5), [kvfree[ng % K_STAGES], ds_free]])
            ng += 1
        for g in range(2):
            if rnd.random() >= 0.4:
                continue
            if phase[g] == -1:
                dot += 1
                bar_dot.arrive()
                phase[g] = 0
                continue
            j = computed[g]
            if j >= steps:
                continue
            if phase[g] == 0:
                if s_done.test(j):
                    assert sbuf == ("S", j), (sbuf, j, g)
                    read_by.setdefault(j, set()).add(g)
                    if len(read_by[j]) == 2:
                        sbuf = ("read", j)
                    s_free.arrive()
                    phase[g] = 1
            elif j == 0 or "ds_free" in drop or ds_free.test(j - 1):
                assert dsbuf is None or dsbuf[0] == "read" or dsbuf == ("dS", j), \
                    ("dS written before dQ read the previous one", dsbuf, j)
                wrote.setdefault(j, set()).add(g)
                if len(wrote[j]) == 2:
                    dsbuf = ("dS", j)
                bar_ds.arrive()
                computed[g] += 1
                phase[g] = 0
        if ng == steps and not pipes["A"] and not pipes["B"] and computed == [steps, steps]:
            if steps:            # the epilogue's wait for the last dQ
                assert ds_free.test(steps - 1)
            return tick
    raise AssertionError(f"no progress: steps={steps} seed={seed} ns={ns} npd={npd} ng={ng} computed={computed}")


@pytest.mark.parametrize("steps", list(range(0, 10)) + [37, 116])
def test_dq_protocol_random_schedules(steps):
    for seed in range(40):
        simulate(steps, seed)


@pytest.mark.parametrize("drop", ["s_free", "ds_free", "kvfree", "vfree"])
def test_model_catches_each_missing_wait(drop):
    """The model is not vacuous: leaving out the wait for the S / dP buffer's
    readers, for the dS buffer's reader, or for a ring stage's, makes some
    schedule fail."""
    caught = 0
    for seed in range(60):
        try:
            simulate(12, seed, max_ticks=50000, drop=(drop,))
        except AssertionError:
            caught += 1
    assert caught > 0, drop
