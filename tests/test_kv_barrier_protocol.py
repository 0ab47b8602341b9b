"""CPU model of the barrier protocol of the dK/dV kernel (fine_bwd_kv_kernel).

The kernel runs four roles on shared-memory mbarriers: a TMA producer filling
a 4-stage Q/dO ring, two MMA-issuing threads (one issues S^T(j), then
dP^T(j); the other dV(j), then dK(j)), and two compute warpgroups.  Step j
uses TMEM step buffer b = j % 2, in two halves: S^T(j) lands in one, dP^T(j)
in the other; each compute warpgroup reads its part of the S^T half and
writes P^T(j) over it, then reads its part of the dP^T half and writes
dS^T(j) over it; dV(j) reads P^T, dK(j) reads dS^T.  The barriers:
  full[s]         ring stage s landed                (TMA -> issuer, compute)
  stage_free[s]   dK of the step in stage s done     (commit -> producer)
  st_done[b]      S^T(j) done                        (commit -> compute)
  dpt_done[b]     dP^T(j) done                       (commit -> compute)
  p_ready[b]      P^T(j) written                     (both warpgroups -> dV(j))
  ds_ready[b]     dS^T(j) written                    (both warpgroups -> dK(j))
  st_free[b]      dV(j) done                         (commit -> S^T(j + 2))
  dpt_free[b]     dK(j) done                         (commit -> dP^T(j + 2); epilogue)
A parity wait for phase k is only correct while the barrier has completed k
or k + 1 phases; the model asserts that at every test, that no half is
overwritten by S^T / dP^T (j + 2) before its reader (dV / dK (j)) is done,
that a warpgroup reads its part of a half before anything overwrites it,
that dV / dK (j) read a complete P^T / dS^T (j), that no ring stage is
refilled before all four products of its step read it, and that every
schedule of random delays terminates.  The MMA groups of one issuing thread
complete in the order issued; nothing orders the two threads' groups, so
the model runs them as two independent queues.
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
    bars = {n: [Barrier(f"{n}{i}", c) for i in range(2)]
            for n, c in (("st_done", 1), ("dpt_done", 1), ("p_ready", 2), ("ds_ready", 2),
                         ("st_free", 1), ("dpt_free", 1))}
    # half h (0: S^T / P^T, 1: dP^T / dS^T) of buffer b -> per warpgroup state:
    # ("T", j) after S^T / dP^T (j); ("P", j) after that warpgroup wrote over it;
    # ("free", j) once dV / dK (j) read it
    half = [[[None, None], [None, None]] for _ in range(2)]
    ring = [None] * STAGES       # stage -> [step, products of the step that read it]
    pipes, loads = {"A": [], "B": []}, []
    produced = 0
    na = [0, 0]                  # issuer A: next step, next half (0: S^T, 1: dP^T)
    nb = [0, 0]                  # issuer B: next step, next product (0: dV, 1: dK)
    computed = [0, 0]
    phase = [0, 0]               # per warpgroup: 0 read S^T, 1 write P^T, 2 read dP^T, 3 write dS^T
    free_of = ("st_free", "dpt_free")
    done_of = ("st_done", "dpt_done")
    ready_of = ("p_ready", "ds_ready")
    for tick in range(max_ticks):
        for pipe in pipes.values():  # each issuer's groups: in order
            if not pipe or rnd.random() < 0.3:
                continue
            pipe[0][2] -= 1
            if pipe[0][2] <= 0:
                kind, j, _, done = pipe.pop(0)
                b, h = j & 1, kind[1]
                st = j % STAGES
                assert ring[st] is not None and ring[st][0] == j, ("ring", ring[st], j)
                ring[st][1] += 1
                if kind[0] == "T":
                    for g in range(2):
                        assert half[h][b][g] is None or half[h][b][g] == ("free", j - 2), \
                            ("overwrote a half its product had not read", h, half[h][b][g], j)
                    half[h][b] = [("T", j), ("T", j)]
                else:
                    assert half[h][b] == [("P", j), ("P", j)], ("product read an incomplete half", h, half[h][b], j)
                    half[h][b] = [("free", j), ("free", j)]
                for bar in done:
                    bar.arrive()
        for load in list(loads):  # TMA completions
            load[1] -= 1
            if load[1] <= 0:
                loads.remove(load)
                st, j = load[0], load[2]
                assert ring[st] is None or ring[st][1] == 4, ("ring stage overwritten before its readers", ring[st], j)
                ring[st] = [j, 0]
                full[st].arrive()
        if produced < steps and rnd.random() < 0.5:   # producer
            st = produced % STAGES
            if produced < STAGES or "stage_free" in drop or stage_free[st].test(produced // STAGES - 1):
                loads.append([st, delay(rnd, 8), produced])
                produced += 1
        j, h = na
        if rnd.random() < 0.7 and j < steps:          # issuer A: S^T(j), then dP^T(j)
            b = j & 1
            if (j < 2 or free_of[h] in drop or bars[free_of[h]][b].test((j >> 1) - 1)) and \
                    full[j % STAGES].test(j // STAGES):
                pipes["A"].append([("T", h), j, delay(rnd, 5), [bars[done_of[h]][b]]])
                na = [j + h, 1 - h]
        j, h = nb
        if rnd.random() < 0.7 and j < na[0] + na[1] and j < steps:   # issuer B: dV(j), then dK(j)
            b = j & 1
            if bars[ready_of[h]][b].test(j >> 1):
                done = [bars[free_of[h]][b]] + ([stage_free[j % STAGES]] if h == 1 else [])
                pipes["B"].append([("G", h), j, delay(rnd, 5), done])
                nb = [j + h, 1 - h]
        for g in range(2):                            # compute warpgroups
            j = computed[g]
            if j >= steps or rnd.random() >= 0.4:
                continue
            b, ph = j & 1, phase[g]
            h = ph >> 1
            if ph in (0, 2):
                if bars[done_of[h]][b].test(j >> 1) and full[j % STAGES].test(j // STAGES):
                    assert half[h][b][g] == ("T", j), ("half not there to read", h, half[h][b][g], j, g)
                    phase[g] += 1
            else:
                # the warpgroup overwrites only its own part, which it has read
                assert half[h][b][g] == ("T", j), (h, half[h][b][g], j, g)
                half[h][b][g] = ("P", j)
                bars[ready_of[h]][b].arrive()
                if ph == 3:
                    computed[g] += 1
                    phase[g] = 0
                else:
                    phase[g] = 2
        if nb[0] == steps and not pipes["A"] and not pipes["B"] and computed == [steps, steps]:
            if steps:            # the epilogue's wait for the last dK
                assert bars["dpt_free"][(steps - 1) & 1].test((steps - 1) >> 1)
            return tick
    raise AssertionError(f"no progress: steps={steps} seed={seed} na={na} nb={nb} computed={computed}")


@pytest.mark.parametrize("steps", list(range(0, 10)) + [37, 154])
def test_kv_protocol_random_schedules(steps):
    for seed in range(40):
        simulate(steps, seed)


@pytest.mark.parametrize("drop", ["st_free", "dpt_free", "stage_free"])
def test_model_catches_each_missing_wait(drop):
    """The model is not vacuous: leaving out the wait for a half's last
    reader (dV or dK of step j - 2) or for a ring stage's makes some
    schedule fail."""
    caught = 0
    for seed in range(60):
        try:
            simulate(12, seed, max_ticks=50000, drop=(drop,))
        except AssertionError:
            caught += 1
    assert caught > 0, drop
