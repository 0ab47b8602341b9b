"""CPU model of the barrier protocol of the dK/dV kernel (fine_bwd_kv_kernel).

The kernel runs four roles on shared-memory mbarriers: a TMA producer filling
a 4-stage Q/dO ring, two MMA-issuing threads (one issues S^T(j) and dP^T(j),
the other dV(j) and dK(j)), and two compute warpgroups.  One
S^T / dP^T buffer in TMEM is released as soon as both warpgroups have read it
into registers; P^T / dS^T go to one of two P buffers (b = j % 2), which the
dV / dK products read.  The barriers, per the kernel:
  full[s]       ring stage s landed                 (TMA -> issuer, compute)
  stage_free[s] dV/dK of the step in stage s done   (commit -> producer)
  s_done        S^T(j), dP^T(j) done                (commit -> compute)
  s_free        S^T(j), dP^T(j) read                (both warpgroups -> issuer: S^T(j+1))
  pds[b]        P^T(j), dS^T(j) written             (both warpgroups -> issuer: dV/dK(j))
  pbuf_free[b]  dV(j), dK(j) done                   (commit -> compute: P(j+2))
A parity wait for phase k is only correct while the barrier has completed k
or k + 1 phases; the model asserts that at every test, that S^T(j + 1) never
overwrites the buffer before both warpgroups read S^T(j), that P(j + 2) is
never written before dV/dK(j) read P buffer b, that dV/dK(j) read P(j), and
that every schedule of random delays terminates.  The MMA groups of one
issuing thread complete in the order issued; nothing orders the two threads'
groups, so the model runs them as two independent queues.
"""
import random

import pytest

STAGES = 4


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
    full = [Barrier(f"full{i}", 1) for i in range(STAGES)]
    stage_free = [Barrier(f"stage_free{i}", 1) for i in range(STAGES)]
    s_done = Barrier("s_done", 1)
    s_free = Barrier("s_free", 2)
    pds = [Barrier(f"pds{i}", 2) for i in range(2)]
    pbuf_free = [Barrier(f"pbuf_free{i}", 1) for i in range(2)]
    sbuf = None                  # the S^T / dP^T buffer: (content, step)
    pbuf = [None, None]          # P buffer -> (content, step)
    ring = [None] * STAGES       # stage -> [step, read by dV/dK]
    read_by, wrote = {}, {}      # step -> warpgroups that read S^T / wrote P^T
    pipes, loads = {"A": [], "B": []}, []   # each issuer's in-order MMA groups; TMA loads in flight
    produced = ns = ng = 0
    computed = [0, 0]
    phase = [0, 0]               # per warpgroup: 0 = read S^T(j), 1 = write P(j)
    for tick in range(max_ticks):
        for pipe in pipes.values():  # each issuer's groups: in order
            if not pipe or rnd.random() < 0.3:
                continue
            pipe[0][2] -= 1
            if pipe[0][2] <= 0:
                kind, j, _, bars = pipe.pop(0)
                assert ring[j % STAGES] is not None and ring[j % STAGES][0] == j, ("ring", ring[j % STAGES], j)
                if kind == "S":
                    assert sbuf is None or sbuf == ("read", j - 1), ("S^T overwritten before it was read", sbuf, j)
                    sbuf = ("S", j)
                else:
                    assert pbuf[j & 1] == ("P", j), (pbuf[j & 1], j)
                    pbuf[j & 1] = ("read", j)
                    ring[j % STAGES][1] = True
                for bar in bars:
                    bar.arrive()
        for load in list(loads):  # TMA completions
            load[1] -= 1
            if load[1] <= 0:
                loads.remove(load)
                st, j = load[0], load[2]
                assert ring[st] is None or ring[st][1], ("ring stage overwritten before dV/dK read it", ring[st], j)
                ring[st] = [j, False]
                full[st].arrive()
        if produced < steps and rnd.random() < 0.5:   # producer
            st = produced % STAGES
            if produced < STAGES or "stage_free" in drop or stage_free[st].test(produced // STAGES - 1):
                loads.append([st, delay(rnd, 8), produced])
                produced += 1
        if rnd.random() < 0.7 and ns < steps and (ns == 0 or "s_free" in drop or s_free.test(ns - 1)) and \
                full[ns % STAGES].test(ns // STAGES):   # issuer A: S^T(j), dP^T(j)
            pipes["A"].append(["S", ns, delay(rnd, 5), [s_done]])
            ns += 1
        if rnd.random() < 0.7 and ng < ns and pds[ng & 1].test(ng >> 1):   # issuer B: dV(j), dK(j)
            pipes["B"].append(["G", ng, delay(rnd, 5), [stage_free[ng % STAGES], pbuf_free[ng & 1]]])
            ng += 1
        for g in range(2):                            # compute warpgroups
            j = computed[g]
            if j >= steps or rnd.random() >= 0.4:
                continue
            b = j & 1
            if phase[g] == 0:
                if s_done.test(j) and full[j % STAGES].test(j // STAGES):
                    assert sbuf == ("S", j), (sbuf, j, g)
                    read_by.setdefault(j, set()).add(g)
                    if len(read_by[j]) == 2:
                        sbuf = ("read", j)
                    s_free.arrive()
                    phase[g] = 1
            elif j < 2 or "pbuf_free" in drop or pbuf_free[b].test((j >> 1) - 1):
                assert pbuf[b] is None or pbuf[b][0] == "read" or pbuf[b] == ("P", j), \
                    ("P buffer written before dV/dK read it", pbuf[b], j)
                wrote.setdefault(j, set()).add(g)
                if len(wrote[j]) == 2:
                    pbuf[b] = ("P", j)
                pds[b].arrive()
                computed[g] += 1
                phase[g] = 0
        if ng == steps and not pipes["A"] and not pipes["B"] and computed == [steps, steps]:
            if steps:            # the epilogue's wait for the last dV/dK
                assert pbuf_free[(steps - 1) & 1].test((steps - 1) >> 1)
            return tick
    raise AssertionError(f"no progress: steps={steps} seed={seed} ns={ns} ng={ng} computed={computed}")


@pytest.mark.parametrize("steps", list(range(0, 10)) + [37, 154])
def test_kv_protocol_random_schedules(steps):
    for seed in range(40):
        simulate(steps, seed)


@pytest.mark.parametrize("drop", ["s_free", "pbuf_free", "stage_free"])
def test_model_catches_each_missing_wait(drop):
    """The model is not vacuous: leaving out the wait for the S^T buffer's
    readers, for the P buffer's last reader, or for the ring stage's, makes
    some schedule fail."""
    caught = 0
    for seed in range(60):
        try:
            simulate(12, seed, max_ticks=50000, drop=(drop,))
        except AssertionError:
            caught += 1
    assert caught > 0, drop
