"""CPU model of the prefill kernel's synchronisation protocol (host logic, no GPU).

`prefill_kernel` (csrc/prefill.cu) coordinates seven roles through mbarriers:
the Q/K TMA producer, the V TMA producer, the correction warps, the single
tcgen05.mma issuer, and the softmax warps of each head, around an in-order
tensor pipe.  This model restates that handshake -- which role waits on which
barrier phase, who arrives, how many arrivals or transaction bytes complete a
phase, which commit follows which MMA -- and runs it under adversarial
scheduling (per-run role priorities, TMA copies landing out of order).  Every
shared-memory stage and TMEM buffer records what it holds, so each modelled
MMA and softmax pass checks that it reads the tile it should:

- K stage holds K(v) (corrected for a remote tile) when QK(v) runs;
- Q is the corrected Q in the remote phase and the reloaded exact Q after;
- V stage holds V(v) and P_n holds P_n(v) when PV_n(v) runs;
- QK_n(v+1) never overwrites a P_n that PV_n(v) has not consumed;
- no phase receives more arrivals than its count (a phase completing early
  is how a race shows up), and every role finishes (no deadlock).

The virtual-tile sequence (remote tiles, then exact tiles) comes from the
same classification the kernel uses (tile_class.cuh, restated below).
The planted-mistake test removes the wait that orders the correction warps'
last arrival and checks that the model then finds the race.
"""
import random

import pytest

KBM = KBN = 128


def tile_class(i0, j0, S, w, g):
    """0 masked, 1 exact, 2 remote, 3 band (both views) -- tile_class.cuh."""
    i1 = min(i0 + KBM, S) - 1
    j1 = min(j0 + KBN, S) - 1
    if j0 > i1:
        return 0
    if g == 1 or i1 - j0 < w:
        return 1
    if i0 - j1 >= w:
        return 2
    return 3


def visit(qt, S, w, g):
    """(NR, T): tiles [0, NR) have a remote part; T virtual tiles in all."""
    i0 = qt * KBM
    lo, hi = 0, qt
    while lo < hi:
        mid = (lo + hi) // 2
        if tile_class(i0, mid * KBN, S, w, g) == 2:
            lo = mid + 1
        else:
            hi = mid
    kb = lo
    lo, hi = kb, qt + 1
    while lo < hi:
        mid = (lo + hi) // 2
        if tile_class(i0, mid * KBN, S, w, g) == 1:
            hi = mid
        else:
            lo = mid + 1
    nr = lo
    return nr, nr + (qt + 1 - kb)


class Race(AssertionError):
    pass


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.phase = name, count, count, 0, 0

    def _complete_if_done(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self):
        if self.pending == 0:
            raise Race(f"{self.name}: arrival beyond the phase's count")
        self.pending -= 1
        self._complete_if_done()

    def arrive_expect_tx(self):
        self.tx += 1
        self.arrive()

    def complete_tx(self):
        self.tx -= 1
        self._complete_if_done()

    def ready(self, parity):
        # try_wait.parity: the phase with this parity has completed
        return (self.phase & 1) != parity


def run_cta(S, w, g, qt, NK, NV, NH, seed, last_arrival_waits=True):
    rnd = random.Random(seed)
    NR, T = visit(qt, S, w, g)
    B = {}

    def bar(name, count):
        B[name] = Bar(name, count)

    bar("QFULL", 1), bar("K0READY", 128), bar("QFREE", 1)
    for s in range(NK):
        bar(f"KFULL{s}", 1), bar(f"KEMPTY{s}", 1), bar(f"GO{s}", 128 + 128 + 1)
    for s in range(NV):
        bar(f"VFULL{s}", 1), bar(f"VEMPTY{s}", 1)
    for n in range(2):
        bar(f"SFULL{n}", 1), bar(f"PFULL{n}", 128), bar(f"ODONE{n}", 1)
    st = {"Q": None, "K": [None] * NK, "V": [None] * NV, "S": [None, None], "P": [None, None],
          "O": [[], []]}
    tma, pipe = [], []

    def wait(name, parity):
        while not B[name].ready(parity):
            yield "blocked"

    def arrive_n(name, k):
        for _ in range(k):
            B[name].arrive()

    def kprod():
        B["QFULL"].arrive_expect_tx()
        tma.append(("QFULL", lambda: st.__setitem__("Q", "exact")))
        for v in range(T):
            if v == NR and NR > 0:
                yield from wait("QFREE", 0)
                B["QFULL"].arrive_expect_tx()
                tma.append(("QFULL", lambda: st.__setitem__("Q", "reloaded")))
            sk = v % NK
            yield from wait(f"KEMPTY{sk}", ((v // NK) & 1) ^ 1)
            B[f"KFULL{sk}"].arrive_expect_tx()
            tma.append((f"KFULL{sk}", lambda sk=sk, v=v: st["K"].__setitem__(sk, (v, "raw"))))
            yield "step"

    def vprod():
        for v in range(T):
            sv = v % NV
            yield from wait(f"VEMPTY{sv}", ((v // NV) & 1) ^ 1)
            B[f"VFULL{sv}"].arrive_expect_tx()
            tma.append((f"VFULL{sv}", lambda sv=sv, v=v: st["V"].__setitem__(sv, v)))
            yield from wait(f"VFULL{sv}", (v // NV) & 1)
            B[f"GO{v % NK}"].arrive()
            yield "step"

    def correction():
        yield from wait("QFULL", 0)
        if NR > 0:
            st["Q"] = "corrected"
        for u in range(T + 1):
            if u < T:
                sk = u % NK
                yield from wait(f"KFULL{sk}", (u // NK) & 1)
                if st["K"][sk] != (u, "raw"):
                    raise Race(f"correction: K stage {sk} holds {st['K'][sk]}, not K({u})")
                if u < NR:
                    st["K"][sk] = (u, "corrected")
                if u == NR and NR > 0:
                    yield from wait("QFULL", 1)
            if u == T and last_arrival_waits and T - 1 >= NK:
                yield from wait(f"GO{(T - 1) % NK}", (((T - 1) // NK) & 1) ^ 1)
            arrive_n("K0READY" if u == 0 else f"GO{(u - 1) % NK}", 128)
            yield "step"

    def qk_op(v, n):
        def run():
            want = (v, "corrected" if v < NR else "raw")
            if st["K"][v % NK] != want:
                raise Race(f"QK{n}({v}): K stage holds {st['K'][v % NK]}, wants {want}")
            q_want = "corrected" if v < NR else ("reloaded" if NR > 0 else "exact")
            if st["Q"] != q_want:
                raise Race(f"QK{n}({v}): Q is {st['Q']}, wants {q_want}")
            if st["P"][n] not in (None, "consumed"):
                raise Race(f"QK{n}({v}): overwrites P{n}({st['P'][n]}) before its PV")
            st["S"][n], st["P"][n] = v, None
        return run

    def pv_op(v, n):
        def run():
            if st["V"][v % NV] != v:
                raise Race(f"PV{n}({v}): V stage holds {st['V'][v % NV]}")
            if st["P"][n] != v:
                raise Race(f"PV{n}({v}): P{n} holds {st['P'][n]}")
            st["P"][n] = "consumed"
            st["O"][n].append(v)
        return run

    def issuer():
        yield from wait("K0READY", 0)

        def qk(v, n):
            pipe.append(("mma", qk_op(v, n)))
            pipe.append(("commit", f"SFULL{n}"))
            if n == NH - 1:
                pipe.append(("commit", f"KEMPTY{v % NK}"))
                if v == NR - 1:
                    pipe.append(("commit", "QFREE"))
        for n in range(NH):
            qk(0, n)
        for v in range(T):
            for n in range(NH):
                if n == 0:
                    yield from wait(f"GO{v % NK}", (v // NK) & 1)
                else:
                    yield from wait(f"PFULL{n}", v & 1)
                pipe.append(("mma", pv_op(v, n)))
                pipe.append(("commit", f"ODONE{n}"))
                if n == NH - 1:
                    pipe.append(("commit", f"VEMPTY{v % NV}"))
                if v + 1 < T:
                    qk(v + 1, n)
                yield "step"

    def softmax(n):
        for v in range(T):
            yield from wait(f"SFULL{n}", v & 1)
            if st["S"][n] != v:
                raise Race(f"softmax{n}({v}): S holds {st['S'][n]}")
            st["P"][n] = v
            arrive_n(f"GO{v % NK}" if n == 0 else f"PFULL{n}", 128)
            yield "step"
        yield from wait(f"ODONE{n}", (T - 1) & 1)
        if st["O"][n] != list(range(T)):
            raise Race(f"epilogue{n}: O accumulated {st['O'][n]}")

    roles = {"kprod": kprod(), "vprod": vprod(), "correction": correction(), "issuer": issuer(),
             "softmax0": softmax(0)}
    if NH == 2:
        roles["softmax1"] = softmax(1)
    weight = {k: rnd.choice([0.05, 1.0, 20.0]) for k in list(roles) + ["tma", "pipe"]}
    idle = 0
    while roles or tma or pipe:
        choices = list(roles) + (["tma"] if tma else []) + (["pipe"] if pipe else [])
        choices.sort(key=lambda c: -rnd.random() ** (1.0 / weight[c]))
        moved = False
        for c in choices:
            if c == "tma":
                name, land = tma.pop(rnd.randrange(len(tma)) if rnd.random() < 0.3 else 0)
                land()
                B[name].complete_tx()
            elif c == "pipe":
                kind, x = pipe.pop(0)
                x() if kind == "mma" else B[x].arrive()
            else:
                try:
                    if next(roles[c]) == "blocked":
                        continue
                except StopIteration:
                    del roles[c]
            moved = True
            break
        idle = 0 if moved else idle + 1
        if idle > 3:
            raise Race(f"deadlock: {sorted(roles)} blocked (NR={NR}, T={T})")


def _group_factor(S, L):
    return 1 if S <= L else -(-S // L)


RINGS = [(3, 2, 2), (3, 3, 1), (4, 4, 2), (4, 4, 1)]  # (NK, NV, NH) for D = 128 / 64
SHAPES = [(700, 200, 150), (2048, 512, 128), (1300, 7, 129), (640, 100, 1), (1000, 300, 256),
          (900, 1000, 64), (1, 1, 1)]


@pytest.mark.parametrize("NK,NV,NH", RINGS)
@pytest.mark.parametrize("S,L,w", SHAPES)
def test_protocol_model_has_no_race_or_deadlock(NK, NV, NH, S, L, w):
    g = _group_factor(S, L)
    for qt in range(-(-S // KBM)):
        for seed in range(12):
            run_cta(S, w, g, qt, NK, NV, NH, seed)


def test_model_finds_the_race_without_the_last_arrival_wait():
    """Planted mistake: the correction warps' last arrival without its phase
    wait can complete a GO phase before head 0's softmax has written P."""
    found = 0
    for qt in range(2, 6):
        for seed in range(40):
            try:
                run_cta(700, 150, 4, qt, 3, 2, 2, seed, last_arrival_waits=False)
            except Race:
                found += 1
    assert found > 0


# ---------------------------------------------------------------- the pair kernel
def run_pair(S, w, g, qt, NK, NV, seed, last_arrival_waits=True):
    """prefill_pair_kernel: two CTAs (ranks 0, 1) of one cluster, two heads
    each.  Each CTA's producers load its own half of every K / V tile; the
    correction warps of each CTA correct their own K half; the issuer (rank 0)
    waits on rank 0's K0READY / GO / PFULL1, which count one arrival per warp of
    BOTH CTAs, and each commit arrives on the barrier of both CTAs.  The last
    correction arrival of each CTA waits on its own KEMPTY for QK(T - NK)."""
    rnd = random.Random(seed)
    NR, T = visit(qt, S, w, g)
    B = [{}, {}]

    def bar(r, name, count):
        B[r][name] = Bar(f"{name}@{r}", count)

    for r in range(2):
        bar(r, "QFULL", 1), bar(r, "K0READY", 8), bar(r, "QFREE", 1)
        for s in range(NK):
            bar(r, f"KFULL{s}", 1), bar(r, f"KEMPTY{s}", 1), bar(r, f"GO{s}", 18)
        for s in range(NV):
            bar(r, f"VFULL{s}", 1), bar(r, f"VEMPTY{s}", 1)
        for n in range(2):
            bar(r, f"SFULL{n}", 1), bar(r, f"PFULL{n}", 8), bar(r, f"ODONE{n}", 1)
    st = [{"Q": None, "K": [None] * NK, "V": [None] * NV, "S": [None, None], "P": [None, None],
           "O": [[], []]} for _ in range(2)]
    tma, pipe = [], []

    def wait(r, name, parity):
        while not B[r][name].ready(parity):
            yield "blocked"

    def kprod(r):
        B[r]["QFULL"].arrive_expect_tx()
        tma.append((r, "QFULL", lambda: st[r].__setitem__("Q", "exact")))
        for v in range(T):
            if v == NR and NR > 0:
                yield from wait(r, "QFREE", 0)
                B[r]["QFULL"].arrive_expect_tx()
                tma.append((r, "QFULL", lambda: st[r].__setitem__("Q", "reloaded")))
            sk = v % NK
            yield from wait(r, f"KEMPTY{sk}", ((v // NK) & 1) ^ 1)
            B[r][f"KFULL{sk}"].arrive_expect_tx()
            tma.append((r, f"KFULL{sk}", lambda sk=sk, v=v: st[r]["K"].__setitem__(sk, (v, "raw"))))
            yield "step"

    def vprod(r):
        for v in range(T):
            sv = v % NV
            yield from wait(r, f"VEMPTY{sv}", ((v // NV) & 1) ^ 1)
            B[r][f"VFULL{sv}"].arrive_expect_tx()
            tma.append((r, f"VFULL{sv}", lambda sv=sv, v=v: st[r]["V"].__setitem__(sv, v)))
            yield from wait(r, f"VFULL{sv}", (v // NV) & 1)
            B[0][f"GO{v % NK}"].arrive()
            yield "step"

    def correction(r):
        yield from wait(r, "QFULL", 0)
        if NR > 0:
            st[r]["Q"] = "corrected"
        for u in range(T + 1):
            if u < T:
                sk = u % NK
                yield from wait(r, f"KFULL{sk}", (u // NK) & 1)
                if st[r]["K"][sk] != (u, "raw"):
                    raise Race(f"correction@{r}: K stage {sk} holds {st[r]['K'][sk]}, not K({u})")
                if u < NR:
                    st[r]["K"][sk] = (u, "corrected")
                if u == NR and NR > 0:
                    yield from wait(r, "QFULL", 1)
            if u == T and last_arrival_waits and T - 1 >= NK:
                yield from wait(r, f"KEMPTY{(T - NK) % NK}", ((T - NK) // NK) & 1)
            for _ in range(4):  # one arrival per correction warp
                B[0]["K0READY" if u == 0 else f"GO{(u - 1) % NK}"].arrive()
            yield "step"

    def qk_op(v, n):
        def run():
            for r in range(2):
                want = (v, "corrected" if v < NR else "raw")
                if st[r]["K"][v % NK] != want:
                    raise Race(f"QK{n}({v}): K half @{r} holds {st[r]['K'][v % NK]}, wants {want}")
                q_want = "corrected" if v < NR else ("reloaded" if NR > 0 else "exact")
                if st[r]["Q"] != q_want:
                    raise Race(f"QK{n}({v}): Q @{r} is {st[r]['Q']}, wants {q_want}")
                if st[r]["P"][n] not in (None, "consumed"):
                    raise Race(f"QK{n}({v}): overwrites P{n}@{r} before its PV")
                st[r]["S"][n], st[r]["P"][n] = v, None
        return run

    def pv_op(v, n):
        def run():
            for r in range(2):
                if st[r]["V"][v % NV] != v:
                    raise Race(f"PV{n}({v}): V half @{r} holds {st[r]['V'][v % NV]}")
                if st[r]["P"][n] != v:
                    raise Race(f"PV{n}({v}): P{n}@{r} holds {st[r]['P'][n]}")
                st[r]["P"][n] = "consumed"
                st[r]["O"][n].append(v)
        return run

    def issuer():
        yield from wait(0, "K0READY", 0)

        def qk(v, n):
            pipe.append(("mma", qk_op(v, n)))
            pipe.append(("commit", f"SFULL{n}"))
            if n == 1:
                pipe.append(("commit", f"KEMPTY{v % NK}"))
                if v == NR - 1:
                    pipe.append(("commit", "QFREE"))
        for n in range(2):
            qk(0, n)
        for v in range(T):
            for n in range(2):
                yield from wait(0, f"GO{v % NK}" if n == 0 else "PFULL1", (v // NK) & 1 if n == 0 else v & 1)
                pipe.append(("mma", pv_op(v, n)))
                pipe.append(("commit", f"ODONE{n}"))
                if n == 1:
                    pipe.append(("commit", f"VEMPTY{v % NV}"))
                if v + 1 < T:
                    qk(v + 1, n)
                yield "step"

    def softmax(r, n):
        for v in range(T):
            yield from wait(r, f"SFULL{n}", v & 1)
            if st[r]["S"][n] != v:
                raise Race(f"softmax{n}@{r}({v}): S holds {st[r]['S'][n]}")
            st[r]["P"][n] = v
            for _ in range(4):  # one arrival per softmax warp
                B[0][f"GO{v % NK}" if n == 0 else "PFULL1"].arrive()
            yield "step"
        yield from wait(r, f"ODONE{n}", (T - 1) & 1)
        if st[r]["O"][n] != list(range(T)):
            raise Race(f"epilogue{n}@{r}: O accumulated {st[r]['O'][n]}")

    roles = {"issuer": issuer()}
    for r in range(2):
        roles.update({f"kprod{r}": kprod(r), f"vprod{r}": vprod(r), f"correction{r}": correction(r),
                      f"softmax0@{r}": softmax(r, 0), f"softmax1@{r}": softmax(r, 1)})
    weight = {k: rnd.choice([0.05, 1.0, 20.0]) for k in list(roles) + ["tma", "pipe"]}
    idle = 0
    while roles or tma or pipe:
        choices = list(roles) + (["tma"] if tma else []) + (["pipe"] if pipe else [])
        choices.sort(key=lambda c: -rnd.random() ** (1.0 / weight[c]))
        moved = False
        for c in choices:
            if c == "tma":
                r, name, land = tma.pop(rnd.randrange(len(tma)) if rnd.random() < 0.3 else 0)
                land()
                B[r][name].complete_tx()
            elif c == "pipe":
                kind, x = pipe.pop(0)
                if kind == "mma":
                    x()
                else:  # commits arrive on the barrier of both CTAs
                    B[0][x].arrive()
                    B[1][x].arrive()
            else:
                try:
                    if next(roles[c]) == "blocked":
                        continue
                except StopIteration:
                    del roles[c]
            moved = True
            break
        idle = 0 if moved else idle + 1
        if idle > 3:
            raise Race(f"deadlock: {sorted(roles)} blocked (NR={NR}, T={T})")


@pytest.mark.parametrize("S,L,w", SHAPES)
def test_pair_protocol_model_has_no_race_or_deadlock(S, L, w):
    g = _group_factor(S, L)
    for qt in range(-(-S // KBM)):
        for seed in range(8):
            run_pair(S, w, g, qt, 4, 4, seed)


def test_pair_model_finds_the_race_without_the_last_arrival_wait():
    """Planted mistake: without the KEMPTY wait, a CTA's last correction
    arrival can complete a GO phase early (a PV or QK then reads a stage that
    is not ready)."""
    found = 0
    for qt in range(2, 8):
        for seed in range(30):
            try:
                run_pair(3000, 300, 6, qt, 4, 4, seed, last_arrival_waits=False)
            except Race:
                found += 1
    assert found > 0
