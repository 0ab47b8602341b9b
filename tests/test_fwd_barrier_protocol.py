"""CPU model of the barrier protocol of the fine forward kernel (fine_fwd_kernel).

Roles, as in the kernel: two TMA producers (one loads K(j) into ring stage
j % nk, the other V(j) into stage j % nv, each in step order and
independently of the other), the MMA issue (one polling thread for both
kinds of group in the native-layout kernel; one thread for S and one for PV
in the others, whose groups nothing orders against each other), and eight
softmax warps, two per TMEM lane quarter (one per key cube of the step).  S(j) goes
into TMEM buffer j % 2, and P(j) is written over the first half of S(j):
each warp writes 32 of those 64 columns, one of which is its partner's half
of S(j), so it may only write once its partner holds that half in
registers.  Barriers:
  bar_qt        Q rows written into TMEM          (256 softmax threads)
  kfull/vfull   ring stage landed                 (TMA)
  kfree/vfree   S(j) / PV(j) that read the stage done   (commits)
  bar_s[b]      S(j) done, b = j % 2              (commit)
  pair[q]       row-max exchange of quarter q     (its two warps, 64 threads;
                                                   both have loaded S(j))
  bar_p[b]      P(j) written over S(j)            (256 threads)
  pv_done[b]    PV(j) done                        (commit; buffer b may take S(j + 2))
The issuer issues S(j) once PV(j - 2) is done and PV(j) once P(j) is
written.  A softmax warp that raises its row max first waits for PV(j - 1)
and then rescales O.  The model asserts the parity rule (a wait for phase k
sees k or k + 1 completed phases), that no ring stage or TMEM buffer is
overwritten before its reader is done, that P(j) is written over S(j) only
after both warps of the quarter read their halves, that PV(j) reads a
complete P(j), that O is rescaled only with PV(0..j-1) done and PV(j) not yet
issued, and that every schedule of random delays terminates.
"""
import random

import pytest

WARPS = 8          # softmax warps; warp w is in lane quarter w % 4
THREADS = 32 * WARPS


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


def simulate(steps, nk, nv, seed, max_ticks=400000, drop=(), two_issuers=False):
    """drop: waits left out on purpose (to show the model catches them).
    two_issuers: S and PV issued by two threads (the kernels that read
    reordered tiles), else by one polling thread (the native-layout kernel)."""
    rnd = random.Random(seed)
    bar_qt = Barrier("bar_qt", THREADS)
    kfull = [Barrier(f"kfull{i}", 1) for i in range(nk)]
    kfree = [Barrier(f"kfree{i}", 1) for i in range(nk)]
    vfull = [Barrier(f"vfull{i}", 1) for i in range(nv)]
    vfree = [Barrier(f"vfree{i}", 1) for i in range(nv)]
    bar_s = [Barrier(f"bar_s{i}", 1) for i in range(2)]
    pair = [Barrier(f"pair{q}", 64) for q in range(4)]
    bar_p = [Barrier(f"bar_p{i}", THREADS) for i in range(2)]
    pv_done = [Barrier(f"pv_done{i}", 1) for i in range(2)]

    kring = [None] * nk            # stage -> [step, consumed]
    vring = [None] * nv
    # TMEM buffer b -> [step, kind "S" / "P", warps that read S, warps that wrote P, read by PV];
    # warp w works on lane quarter w % 4, w and w ^ 4 are the two warps of a quarter
    buf = [None, None]
    pv_completed = -1              # last PV completed (in order)
    pv_issued = -1
    rescale = {}                   # (step, quarter) -> bool, the same for both warps of a quarter
    pipes, loads = {"S": [], "PV": []}, []
    if not two_issuers:
        pipes["PV"] = pipes["S"]          # one thread: one queue, in issue order

    progs = [[("K", j) for j in range(steps)], [("V", j) for j in range(steps)]]
    pcs = [0, 0]
    ns = npv = 0
    qt_ok = False
    warp_j = [0] * WARPS
    warp_pc = [0] * WARPS          # 0 wait S, 1 arrive pair, 2 wait pair, 3 rescale, 4 write P
    warp_qt = [False] * WARPS

    for tick in range(max_ticks):
        # tensor pipe: each issuing thread's groups complete in issue order;
        # nothing orders two threads' groups (one thread: a single queue)
        for pipe in {id(q): q for q in pipes.values()}.values():
            if not pipe or rnd.random() < 0.3:
                continue
            pipe[0][2] -= 1
            if pipe[0][2] <= 0:
                kind, j, _, bars = pipe.pop(0)
                b = j & 1
                if kind == "S":
                    st = j % nk
                    assert kring[st] is not None and kring[st][0] == j, ("K stage", kring[st], j)
                    assert buf[b] is None or (buf[b][0] == j - 2 and buf[b][4]), ("S over an unread P", buf[b], j)
                    kring[st][1] = True
                    buf[b] = [j, "S", set(), set(), False]
                else:
                    st = j % nv
                    assert vring[st] is not None and vring[st][0] == j, ("V stage", vring[st], j)
                    assert buf[b] is not None and buf[b][0] == j and len(buf[b][3]) == WARPS, \
                        ("PV reads incomplete P", buf[b], j)
                    vring[st][1] = True
                    buf[b][4] = True
                    assert pv_completed == j - 1
                    pv_completed = j
                for bar in bars:
                    bar.arrive()
        for ld in list(loads):
            ld[2] -= 1
            if ld[2] <= 0:
                loads.remove(ld)
                kind, j = ld[0], ld[1]
                ring, depth = (kring, nk) if kind == "K" else (vring, nv)
                st = j % depth
                assert ring[st] is None or ring[st][1], (kind, "stage overwritten before read", ring[st], j)
                ring[st] = [j, False]
                (kfull if kind == "K" else vfull)[st].arrive()
        # producers
        for pi in range(2):
            if pcs[pi] < len(progs[pi]) and rnd.random() < 0.5:
                kind, j = progs[pi][pcs[pi]]
                depth, free = (nk, kfree) if kind == "K" else (nv, vfree)
                st, use = j % depth, j // depth
                if use == 0 or (kind == "K" and "kfree" in drop) or free[st].test(use - 1):
                    loads.append([kind, j, delay(rnd, 10)])
                    pcs[pi] += 1
        # issuers: S(ns) once PV(ns - 2) is done and K(ns) has landed; PV(npv)
        # once P(npv) is written and V(npv) has landed.  One polling thread
        # tries S first; with two threads each goes on its own.
        s_go = steps and rnd.random() < 0.7
        pv_go = (rnd.random() < 0.7) if two_issuers else not s_go
        if s_go and not qt_ok:
            qt_ok = bar_qt.test(0)
        elif s_go and ns < steps and (ns < 2 or "pv_s" in drop or pv_done[ns & 1].test((ns >> 1) - 1)) and \
                kfull[ns % nk].test(ns // nk):
            pipes["S"].append(["S", ns, delay(rnd, 6), [bar_s[ns & 1], kfree[ns % nk]]])
            ns += 1
            pv_go = pv_go and two_issuers
        elif not two_issuers and s_go:
            pv_go = True
        if steps and pv_go and npv < ns and bar_p[npv & 1].test(npv >> 1) and vfull[npv % nv].test(npv // nv):
            pipes["PV"].append(["PV", npv, delay(rnd, 6), [vfree[npv % nv], pv_done[npv & 1]]])
            pv_issued = npv
            npv += 1
        # softmax warps
        for w in range(WARPS):
            if rnd.random() > 0.35:
                continue
            q = w % 4
            if not warp_qt[w]:
                warp_qt[w] = True
                bar_qt.arrive(32)
                continue
            j = warp_j[w]
            if j >= steps:
                continue
            b = j & 1
            if warp_pc[w] == 0:
                if bar_s[b].test(j >> 1):
                    # the lanes of a quarter are its own: only P written by
                    # the two warps of this quarter would overwrite this half
                    assert buf[b] is not None and buf[b][0] == j, ("S buffer", buf[b], j)
                    assert not (buf[b][3] & {q, q + 4}), ("S read after P was written over it", buf[b], j, w)
                    buf[b][2].add(w)
                    warp_pc[w] = 1
            elif warp_pc[w] == 1:
                pair[q].arrive(32)
                warp_pc[w] = 2
            elif warp_pc[w] == 2:
                if "pair" in drop or pair[q].test(j):
                    rescale.setdefault((j, q), j > 0 and rnd.random() < 0.3)
                    warp_pc[w] = 3
            elif warp_pc[w] == 3:
                if not rescale[(j, q)]:
                    warp_pc[w] = 4
                elif "rescale" in drop or pv_done[(j - 1) & 1].test((j - 1) >> 1):
                    assert pv_completed >= j - 1 and pv_issued < j, ("rescale of O", pv_completed, pv_issued, j)
                    warp_pc[w] = 4
            elif warp_pc[w] == 4:
                partner = w ^ 4
                assert buf[b][0] == j and partner in buf[b][2] and w in buf[b][2], \
                    ("P written over S its partner has not read", buf[b], j, w)
                buf[b][1] = "P"
                buf[b][3].add(w)
                bar_p[b].arrive(32)
                warp_j[w] += 1
                warp_pc[w] = 0
        if steps == 0:
            return tick
        if npv == steps and not pipes["S"] and not pipes["PV"] and all(x == steps for x in warp_j):
            assert pv_done[(steps - 1) & 1].test((steps - 1) >> 1)   # epilogue wait
            return tick
    raise AssertionError(f"no progress: steps={steps} nk={nk} nv={nv} seed={seed} ns={ns} npv={npv} warps={warp_j}")


@pytest.mark.parametrize("two_issuers", [False, True])
@pytest.mark.parametrize("nk,nv", [(1, 1), (2, 1), (2, 2), (3, 3), (3, 2)])
@pytest.mark.parametrize("steps", [0, 1, 2, 3, 4, 7, 12, 31])
def test_fwd_protocol_random_schedules(nk, nv, steps, two_issuers):
    for seed in range(12):
        simulate(steps, nk, nv, seed, two_issuers=two_issuers)


@pytest.mark.parametrize("two_issuers", [False, True])
@pytest.mark.parametrize("drop", ["kfree", "pv_s", "pair", "rescale"])
def test_model_catches_each_missing_wait(drop, two_issuers):
    """Leaving out any one of the waits makes some schedule fail."""
    caught = 0
    for seed in range(60):
        try:
            simulate(12, 2, 2, seed, max_ticks=50000, drop=(drop,), two_issuers=two_issuers)
        except AssertionError:
            caught += 1
    assert caught > 0, drop
