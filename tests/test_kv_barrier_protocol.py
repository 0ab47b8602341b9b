"""CPU model of the barrier protocol of the dK/dV kernel (fine_bwd_kv_kernel).

The kernel runs four roles on shared-memory mbarriers: a TMA producer filling
a 4-stage Q/dO ring, one MMA-issuing thread, and two compute warpgroups.  S^T
and dP^T are double-buffered in TMEM (buffer b = j % 2) and the compute warps
write P^T / dS^T over them.  The barriers, per the kernel:
  full[s]       ring stage s landed                (TMA -> issuer, compute)
  stage_free[s] dV/dK of the step in stage s done  (commit -> producer)
  s_done[b]     S^T(j), dP^T(j) done               (commit -> compute)
  pds[b]        P^T(j), dS^T(j) written            (both warpgroups -> issuer)
  buf_free[b]   dV(j), dK(j) done                  (commit -> issuer: S^T(j+2))
A parity wait for phase k is only correct while the barrier has completed k
or k + 1 phases; the model asserts that at every test, that S^T(j + 2) never
overwrites a buffer before dV/dK(j) read it, that dV/dK(j) read P^T(j), and
that every schedule of random delays terminates.  The tensor pipe executes
the issued MMA groups in order, as the hardware does.
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


def simulate(steps, seed, max_ticks=200000):
    rnd = random.Random(seed)
    full = [Barrier(f"full{i}", 1) for i in range(STAGES)]
    stage_free = [Barrier(f"stage_free{i}", 1) for i in range(STAGES)]
    s_done = [Barrier(f"s_done{i}", 1) for i in range(2)]
    pds = [Barrier(f"pds{i}", 2) for i in range(2)]
    buf_free = [Barrier(f"buf_free{i}", 1) for i in range(2)]
    tmem = [None, None]          # buffer -> (content, step)
    wrote = set()                # (step, warpgroup) that wrote P^T / dS^T
    pipe, loads = [], []         # in-order MMA groups; TMA loads in flight
    produced = ns = ng = 0
    computed = [0, 0]
    for tick in range(max_ticks):
        if pipe:                 # tensor pipe: in order
            pipe[0][2] -= 1
            if pipe[0][2] <= 0:
                kind, j, _, bars = pipe.pop(0)
                b = j & 1
                if kind == "S":
                    assert tmem[b] is None or tmem[b] == ("read", j - 2), (tmem[b], j)
                    tmem[b] = ("S", j)
                else:
                    assert tmem[b] == ("P", j), (tmem[b], j)
                    tmem[b] = ("read", j)
                for bar in bars:
                    bar.arrive()
        for load in list(loads):  # TMA completions
            load[1] -= 1
            if load[1] <= 0:
                loads.remove(load)
                full[load[0]].arrive()
        if produced < steps and rnd.random() < 0.5:   # producer
            st = produced % STAGES
            if produced < STAGES or stage_free[st].test(produced // STAGES - 1):
                loads.append([st, delay(rnd, 8)])
                produced += 1
        if rnd.random() < 0.7:                        # MMA issuer
            if ns < steps and (ns < 2 or buf_free[ns & 1].test((ns >> 1) - 1)) and \
                    full[ns % STAGES].test(ns // STAGES):
                pipe.append(["S", ns, delay(rnd, 5), [s_done[ns & 1]]])
                ns += 1
            elif ng < ns and pds[ng & 1].test(ng >> 1):
                pipe.append(["G", ng, delay(rnd, 5), [stage_free[ng % STAGES], buf_free[ng & 1]]])
                ng += 1
        for g in range(2):                            # compute warpgroups
            j = computed[g]
            if j < steps and rnd.random() < 0.4:
                b = j & 1
                if s_done[b].test(j >> 1) and full[j % STAGES].test(j // STAGES):
                    assert tmem[b] in (("S", j), ("P", j)), (tmem[b], j, g)
                    wrote.add((j, g))
                    if (j, 0) in wrote and (j, 1) in wrote:
                        tmem[b] = ("P", j)
                    pds[b].arrive()
                    computed[g] += 1
        if ng == steps and not pipe and computed == [steps, steps]:
            if steps:            # the epilogue's wait for the last dV/dK
                assert buf_free[(steps - 1) & 1].test((steps - 1) >> 1)
            return tick
    raise AssertionError(f"no progress: steps={steps} seed={seed} ns={ns} ng={ng} computed={computed}")


@pytest.mark.parametrize("steps", list(range(0, 10)) + [37, 154])
def test_kv_protocol_random_schedules(steps):
    for seed in range(40):
        simulate(steps, seed)


def test_model_catches_a_missing_buffer_wait():
    """The model is not vacuous: issuing S^T(j) without waiting for
    buf_free (dV/dK(j - 2)) is caught as an overwrite of unread P^T."""
    caught = 0
    for seed in range(40):
        try:
            _simulate_without_buf_free(12, seed)
        except AssertionError:
            caught += 1
    assert caught > 0


def _simulate_without_buf_free(steps, seed):
    rnd = random.Random(seed)
    s_done = [Barrier(f"s_done{i}", 1) for i in range(2)]
    tmem = [None, None]
    pipe, ns, ng, computed = [], 0, 0, 0
    ready = set()
    for _ in range(20000):
        if pipe:
            pipe[0][2] -= 1
            if pipe[0][2] <= 0:
                kind, j, _ = pipe.pop(0)
                b = j & 1
                if kind == "S":
                    assert tmem[b] is None or tmem[b] == ("read", j - 2), (tmem[b], j)
                    tmem[b] = ("S", j)
                    s_done[b].phases += 1
                else:
                    tmem[b] = ("read", j)
        if ns < steps and rnd.random() < 0.9:        # no buf_free wait
            pipe.append(["S", ns, rnd.randint(1, 3)])
            ns += 1
        if computed < steps and rnd.random() < 0.2 and s_done[computed & 1].phases > computed >> 1:
            ready.add(computed)
            computed += 1
        if ng in ready and rnd.random() < 0.5:
            pipe.append(["G", ng, rnd.randint(1, 3)])
            ng += 1
        if ng == steps and not pipe:
            return
