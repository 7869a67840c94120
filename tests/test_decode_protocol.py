"""CPU model of the tensor-core decode kernel's synchronisation protocol
(host logic, no GPU).

`decode_tc_kernel` (csrc/decode.cu) coordinates six roles through mbarriers:
the K and V TMA producers, the correction warps, the single tcgen05.mma issuer
and the softmax warps, around an in-order tensor pipe.  This model restates
that handshake -- who waits on which barrier phase, who arrives, which commit
follows which MMA, and the issue order QK(v+1) before P.V(v) -- and runs it
under adversarial scheduling (per-run role priorities, TMA copies landing out
of order).  Every stage and buffer records what it holds, so each modelled MMA
and softmax pass checks that it reads what it should:

- a K stage holds K(v) raw for an exact QK, and corrected for the aliased QK;
  the tile the window edge crosses is read raw (its exact QK) before the
  correction rotates it;
- S buffer v % 2 holds S(v) when the softmax reads it;
- a P buffer is never rewritten before the P.V that reads it has run, and
  P.V(v) reads P(v) and V(v) (zeroed past the sequence on the paged batch's
  last tile);
- when the softmax rescales O at tile v, O holds exactly the tiles before v;
  at the epilogue it holds every tile;
- no phase receives more arrivals than its count, and every role finishes.

P.V(v) completes a phase of ODONE[v % 2]: with QK(v+1) issued before P.V(v)
the P.V of the last two tiles can both be in flight at the epilogue, and on a
single barrier no parity wait is right there -- one on the last phase alone
passes on the older one (the kernel's first version), and a wait on tile
T-2's phase first blocks when both phases completed before it (the second).
The planted-mistake tests run both single-barrier forms and check that the
model finds each.
"""
import random

import pytest

NS = 3
KEYS = 128


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


def tile_classes(j_begin, j_end, j_split):
    """0 exact, 1 remote, 2 crossed by the window edge -- as decode_tc_kernel."""
    out = []
    for j0 in range(j_begin, j_end, KEYS):
        out.append(0 if j0 >= j_split else (1 if j0 + KEYS <= j_split else 2))
    return out


def run_split(cls, seed, paged=False, odone="split"):
    """odone: "split" -- two P.V barriers, tile v's commit on ODONE[v % 2] (the
    kernel); "single_last" -- one barrier, the epilogue waiting on the last
    phase only; "single_both" -- one barrier, the epilogue waiting on tile
    T-2's phase and then tile T-1's."""
    rnd = random.Random(seed)
    T = len(cls)
    B = {}

    def bar(name, count):
        B[name] = Bar(name, count)

    for s in range(NS):
        bar(f"KFULL{s}", 1), bar(f"KEMPTY{s}", 1), bar(f"KREADY{s}", 4)
        bar(f"VFULL{s}", 1), bar(f"VEMPTY{s}", 1)
    for b in range(2):
        bar(f"SFULL{b}", 1), bar(f"PFULL{b}", 4)
    bar("ODONE0", 1), bar("ODONE1", 1), bar("QREADY", 4), bar("BANDQK", 1), bar("VREADY", 1)

    def odone_of(v):
        # (barrier, parity) of the phase that P.V(v) completes
        if odone == "split":
            return f"ODONE{v & 1}", (v >> 1) & 1
        return "ODONE0", v & 1
    st = {"K": [None] * NS, "V": [None] * NS, "S": [None, None], "Sx": [None, None],
          "P": ["consumed", "consumed"], "O": []}
    tma, pipe = [], []
    rescale_at = {v for v in range(1, T) if rnd.random() < 0.3}

    def wait(name, parity):
        while not B[name].ready(parity):
            yield "blocked"

    def arrive_n(name, k):
        for _ in range(k):
            B[name].arrive()

    def producer(kind):
        for v in range(T):
            s = v % NS
            yield from wait(f"{kind}EMPTY{s}", ((v // NS) & 1) ^ 1)
            B[f"{kind}FULL{s}"].arrive_expect_tx()
            tma.append((f"{kind}FULL{s}", lambda s=s, v=v: st[kind].__setitem__(s, (v, "raw"))))
            yield "step"
        if kind == "V" and paged:
            # the last tile's rows past the sequence are zeroed, then VREADY
            v = T - 1
            yield from wait(f"VFULL{v % NS}", (v // NS) & 1)
            if st["V"][v % NS] != (v, "raw"):
                raise Race(f"V zeroing: stage holds {st['V'][v % NS]}, not V({v})")
            st["V"][v % NS] = (v, "zeroed")
            B["VREADY"].arrive()

    def correction():
        for v in range(T):
            s = v % NS
            yield from wait(f"KFULL{s}", (v // NS) & 1)
            if cls[v] == 2:
                yield from wait("BANDQK", 0)
            if st["K"][s] != (v, "raw"):
                raise Race(f"correction: K stage {s} holds {st['K'][s]}, not K({v}) raw")
            if cls[v] != 0:
                st["K"][s] = (v, "corrected")
            arrive_n(f"KREADY{s}", 4)
            yield "step"

    def qk_op(v, group):
        def run():
            want = (v, "raw") if (cls[v] == 0 or group == 1) else (v, "corrected")
            if st["K"][v % NS] != want:
                raise Race(f"QK({v}) group {group}: K stage holds {st['K'][v % NS]}, wants {want}")
            # S(v) goes to buffer v % 2; the softmax must have finished S(v-2)
            if group == 0:
                st["S"][v & 1] = v
            else:
                st["Sx"][v & 1] = v
        return run

    def pv_op(v):
        def run():
            want_v = (v, "zeroed") if (paged and v == T - 1) else (v, "raw")
            if st["V"][v % NS] != want_v:
                raise Race(f"PV({v}): V stage holds {st['V'][v % NS]}, wants {want_v}")
            if st["P"][v & 1] != v:
                raise Race(f"PV({v}): P buffer holds {st['P'][v & 1]}")
            st["P"][v & 1] = "consumed"
            st["O"].append(v)
        return run

    def issuer():
        yield from wait("QREADY", 0)

        def qk_tile(v):
            s = v % NS
            if cls[v] == 2:
                yield from wait(f"KFULL{s}", (v // NS) & 1)
                pipe.append(("mma", qk_op(v, 1)))
                pipe.append(("commit", "BANDQK"))
            yield from wait(f"KREADY{s}", (v // NS) & 1)
            pipe.append(("mma", qk_op(v, 0)))
            pipe.append(("commit", f"SFULL{v & 1}"))
            pipe.append(("commit", f"KEMPTY{s}"))

        yield from qk_tile(0)
        for v in range(T):
            if v + 1 < T:
                yield from qk_tile(v + 1)
            yield from wait(f"PFULL{v & 1}", (v >> 1) & 1)
            if paged and v == T - 1:
                yield from wait("VREADY", 0)
            else:
                yield from wait(f"VFULL{v % NS}", (v // NS) & 1)
            pipe.append(("mma", pv_op(v)))
            pipe.append(("commit", f"VEMPTY{v % NS}"))
            pipe.append(("commit", odone_of(v)[0]))
            yield "step"

    def softmax():
        arrive_n("QREADY", 4)
        for v in range(T):
            yield from wait(f"SFULL{v & 1}", (v >> 1) & 1)
            if st["S"][v & 1] != v:
                raise Race(f"softmax({v}): S buffer holds {st['S'][v & 1]}")
            if cls[v] == 2 and st["Sx"][v & 1] != v:
                raise Race(f"softmax({v}): exact view holds {st['Sx'][v & 1]}")
            if v in rescale_at:
                yield from wait(*odone_of(v - 1))
                if st["O"] != list(range(v)):
                    raise Race(f"rescale at {v}: O holds tiles {st['O']}")
            if st["P"][v & 1] != "consumed":
                raise Race(f"softmax({v}): P buffer still holds P({st['P'][v & 1]})")
            st["P"][v & 1] = v
            arrive_n(f"PFULL{v & 1}", 4)
            yield "step"
        if odone == "single_both" and T >= 2:
            yield from wait(*odone_of(T - 2))
        yield from wait(*odone_of(T - 1))
        if st["O"] != list(range(T)):
            raise Race(f"epilogue: O holds tiles {st['O']}")

    roles = {"kprod": producer("K"), "vprod": producer("V"), "correction": correction(),
             "issuer": issuer(), "softmax": softmax()}
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
            raise Race(f"deadlock: {sorted(roles)} blocked (T={T})")


# (j_begin, j_end, j_split): splits of the 128K call, one crossed by the
# window edge, the last split's ragged tail, single tiles, plain (g = 1)
SPLITS = [
    (0, 7296, 126976),           # 57 remote tiles
    (124032, 131072, 126976),    # remote, the edge tile, exact
    (126976, 131072, 126976),    # edge on a tile boundary: exact only
    (0, 300, 200),               # three tiles, the edge inside the second
    (0, 1, 0),                   # one key
    (0, 128, 64),                # one tile, both views
    (0, 5000, 0),                # plain: every tile exact
]


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("j_begin,j_end,j_split", SPLITS)
def test_decode_protocol_model_has_no_race_or_deadlock(j_begin, j_end, j_split, paged):
    cls = tile_classes(j_begin, j_end, j_split)
    for seed in range(25):
        run_split(cls, seed, paged=paged)


def _races(odone):
    found = 0
    cls = tile_classes(0, 2048, 0)
    for seed in range(300):
        try:
            run_split(cls, seed, odone=odone)
        except Race:
            found += 1
    return found


def test_model_finds_the_epilogue_race_with_one_barrier_and_one_wait():
    """Planted mistake: with QK(v+1) issued before P.V(v), the P.V of the last
    two tiles can both be in flight at the epilogue; on one barrier a parity
    wait on the last phase then passes on the older one and reads O early."""
    assert _races("single_last") > 0


def test_model_finds_the_stall_with_one_barrier_and_two_waits():
    """Planted mistake: on one barrier, waiting first for tile T-2's phase
    blocks for good when both last phases completed before the wait (the
    parity then names the phase in progress); the kernel's bounded wait would
    time out.  Two barriers, one per tile parity, keep every wait at most one
    phase behind."""
    assert _races("single_both") > 0
