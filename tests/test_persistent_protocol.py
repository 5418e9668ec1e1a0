"""A model of the persistent forward kernel's barrier protocol, run on the CPU.

The persistent kernel (attention_forward_mbarrier_gb300/csrc/fmha_fwd_persistent.cuh)
keeps its mbarrier phases running across the work units a CTA takes, and a
parity wait (mbarrier.try_wait.parity) is only unambiguous while its barrier
is at most one phase away from the phase waited for: a waiter two phases
ahead sees a completed phase that is not its own, one two phases behind waits
for ever.  This test replays the roles' waits and signals in the order the
kernel issues them, for one CTA and a sequence of units, under random
interleavings: the producer (unit ring, Q loads after the QFree commit, K/V
ring loads after the step commit that frees the slot), the MMA thread (first
QK^T of a unit, per step PV then the next QK^T, SFull0 / QFree / OFinal /
step commits, the first PV of a tile after ODrained, the acknowledgement of
tile 1 without key blocks), the 8 softmax warps, an in-order tensor pipe and
TMA copies that land in any order.

Checked on every wait: the parity test gives the same answer as the phase
count (never premature, never stuck).  Checked on every access: ring slots are
not refilled while an MMA reads them, QK^T reads the right Q and K block, PV
reads the P of its own step and the right V block, P is not overwritten before
its PV, O is not overwritten before the epilogue has read it, and the
epilogue reads O after exactly the unit's PVs.  A variant with the step
commits on two barriers instead of four must fail, which shows the model can
find the ambiguity it guards against.
"""
import random

import pytest


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.done += 1
            self.pending = self.count


def simulate(units, seed, step_bars=4, ring=4):
    """Run one CTA over `units` (key blocks of tile 0, of tile 1); return violations."""
    rnd = random.Random(seed)
    viol = []
    bars = {}

    def bar(name, count=1):
        bars[name] = Bar(name, count)

    for t in (0, 1):
        for n in ("QFull", "OFinal", "QFree"):
            bar(f"{n}{t}")
        bar(f"PVReady{t}", 4)
        bar(f"ODrained{t}", 4)
    for s in range(ring):
        bar(f"KVFull{s}")
    for s in range(step_bars):
        bar(f"Step{s}")
    bar("SFull0")
    for s in range(4):
        bar(f"UnitFull{s}")
        bar(f"UnitFree{s}", 9)  # the MMA thread and 8 softmax warps
    unit_ring = {}
    pipe, tma = [], []
    st = {"slot": {}, "Q": {}, "S": {}, "P": {}, "O": {}, "readers": {}, "Oread": {}}

    def wait(name, k, who):
        b = bars[name]
        while True:
            res = (b.done & 1) != (k & 1)  # try_wait.parity on phase k
            if res and b.done <= k:
                viol.append(f"premature {who} on {name} phase {k} (completed {b.done})")
            if not res and b.done > k:
                viol.append(f"stuck {who} on {name} phase {k} (completed {b.done})")
            if b.done > k:
                return
            yield

    def step_bar(n):
        return f"Step{n % step_bars}", n // step_bars

    def producer():
        nu = ld = cbase = 0
        qloads = [0, 0]
        release = {}
        for ui, unit in enumerate(units + [None]):
            slot = nu % 4
            if nu >= 4:
                yield from wait(f"UnitFree{slot}", nu // 4 - 1, "producer")
            unit_ring[slot] = ui if unit is not None else -1
            bars[f"UnitFull{slot}"].arrive()
            nu += 1
            if unit is None:
                return
            n0, n1 = unit
            nkv = max(n0, n1)

            def load_q(t):
                if (n1 if t else n0) == 0:
                    return
                if qloads[t] > 0:
                    yield from wait(f"QFree{t}", qloads[t] - 1, "producer Q")
                if st["Q"].get(t, [None, 0])[1] > 0:
                    viol.append(f"Q{t} refilled while read")
                st["Q"][t] = [(ui, "loading"), 0]
                tma.append((f"QFull{t}", lambda t=t, ui=ui: st["Q"].__setitem__(t, [(ui, "ok"), 0])))
                qloads[t] += 1

            yield from load_q(0)
            for i in range(2 * nkv):
                if i == 1:
                    yield from load_q(1)
                g = ld
                ld += 1
                s = g % ring
                if g >= ring:
                    yield from wait(*step_bar(release[s]), "producer K/V")
                if st["readers"].get(s, 0) > 0:
                    viol.append(f"slot {s} refilled while read")
                st["slot"][s] = (ui, i, "loading")
                tma.append((f"KVFull{s}", lambda s=s, ui=ui, i=i: st["slot"].__setitem__(s, (ui, i, "ok"))))
                release[s] = cbase + (i >> 1) + (i & 1)  # K_b: commit b; V_b: commit b + 1
                yield
            cbase += nkv + 1 if nkv > 0 else 0

    def mma():
        nu = ld = cn = 0
        qn, pvn, on = [0, 0], [0, 0], [0, 0]
        while True:
            slot = nu % 4
            yield from wait(f"UnitFull{slot}", nu // 4, "mma")
            ui = unit_ring[slot]
            bars[f"UnitFree{slot}"].arrive()
            nu += 1
            if ui < 0:
                return
            n0, n1 = units[ui]
            nb, nkv = (n0, n1), max(n0, n1)
            if nkv == 0:
                continue

            def qk(t, j, s, ui=ui):
                st["readers"][s] = st["readers"].get(s, 0) + 1
                st["Q"][t][1] += 1

                def run():
                    if st["slot"][s] != (ui, 2 * j, "ok"):
                        viol.append(f"QK{t} reads K {st['slot'][s]}, wants {(ui, 2 * j)}")
                    if st["Q"][t][0] != (ui, "ok"):
                        viol.append(f"QK{t} reads Q {st['Q'][t][0]}")
                    if st["P"].get(t) not in (None, "consumed"):
                        viol.append(f"QK{t} overwrites unconsumed P {st['P'][t]}")
                    st["S"][t] = (ui, j)
                    st["P"][t] = None
                    st["readers"][s] -= 1
                    st["Q"][t][1] -= 1
                pipe.append(("mma", run))

            def pv(t, j, s, ui=ui):
                st["readers"][s] = st["readers"].get(s, 0) + 1

                def run():
                    if st["slot"][s] != (ui, 2 * j + 1, "ok"):
                        viol.append(f"PV{t} reads V {st['slot'][s]}")
                    if st["P"].get(t) != (ui, j):
                        viol.append(f"PV{t} reads P {st['P'].get(t)}, wants {(ui, j)}")
                    if j == 0:
                        if st["Oread"].get(t, True) is False:
                            viol.append(f"PV{t} overwrites O before the epilogue read it")
                        st["O"][t] = [ui, 1]
                        st["Oread"][t] = False
                    else:
                        st["O"][t][1] += 1
                    st["P"][t] = "consumed"
                    st["readers"][s] -= 1
                pipe.append(("mma", run))

            ks = ld % ring
            yield from wait(f"KVFull{ks}", ld // ring, "mma K0")
            for t in (0, 1):
                if nb[t] > 0:
                    yield from wait(f"QFull{t}", qn[t], "mma Q")
                    qn[t] += 1
                    qk(t, 0, ks)
                    if t == 0:
                        pipe.append(("commit", "SFull0"))
                    if nb[t] == 1:
                        pipe.append(("commit", f"QFree{t}"))
                    yield
            pipe.append(("commit", step_bar(cn)[0]))
            cn += 1
            for j in range(nkv):
                vidx = ld + 2 * j + 1
                yield from wait(f"KVFull{vidx % ring}", vidx // ring, "mma V")
                kidx = ld + 2 * j + 2
                k_ready = False
                for t in (0, 1):
                    if j >= nb[t]:
                        continue
                    yield from wait(f"PVReady{t}", pvn[t], f"mma P{t}")
                    pvn[t] += 1
                    if j == 0 and on[t] > 0:
                        yield from wait(f"ODrained{t}", on[t] - 1, "mma ODrained")
                    pv(t, j, vidx % ring)
                    if j + 1 < nb[t]:
                        if not k_ready:
                            yield from wait(f"KVFull{kidx % ring}", kidx // ring, "mma K")
                            k_ready = True
                        qk(t, j + 1, kidx % ring)
                        if t == 0:
                            pipe.append(("commit", "SFull0"))
                        if j + 2 == nb[t]:
                            pipe.append(("commit", f"QFree{t}"))
                    else:
                        pipe.append(("commit", f"OFinal{t}"))
                        on[t] += 1
                    yield
                if n1 == 0:  # tile 1 acknowledges the step it has no block for
                    yield from wait("PVReady1", pvn[1], "mma ack")
                    pvn[1] += 1
                pipe.append(("commit", step_bar(cn)[0]))
                cn += 1
                yield
            ld += 2 * nkv

    def softmax(t, warp):
        nu = cn = s0n = ofn = 0
        while True:
            slot = nu % 4
            yield from wait(f"UnitFull{slot}", nu // 4, f"softmax{t}")
            ui = unit_ring[slot]
            bars[f"UnitFree{slot}"].arrive()
            nu += 1
            if ui < 0:
                return
            n0, n1 = units[ui]
            nkv, nb = max(n0, n1), (n0, n1)[t]
            if t == 1 and nb == 0:
                for j in range(nkv):
                    yield from wait(*step_bar(cn + j), "softmax1 ack")
                    bars["PVReady1"].arrive()
                    yield
            for j in range(nb):
                if t == 1:
                    yield from wait(*step_bar(cn + j), "softmax1 S")
                else:
                    yield from wait("SFull0", s0n + j, "softmax0 S")
                if st["S"].get(t) != (ui, j):
                    viol.append(f"softmax{t} reads S {st['S'].get(t)}, wants {(ui, j)}")
                yield
                if warp == 0:
                    st["P"][t] = (ui, j)
                bars[f"PVReady{t}"].arrive()
                yield
            if nb > 0:
                yield from wait(f"OFinal{t}", ofn, f"softmax{t} O")
                ofn += 1
                if st["O"][t] != [ui, nb]:
                    viol.append(f"epilogue{t} reads O {st['O'][t]}, wants {[ui, nb]}")
                yield
                if warp == 0:
                    st["Oread"][t] = True
                bars[f"ODrained{t}"].arrive()
            cn += nkv + 1 if nkv > 0 else 0
            s0n += n0

    roles = [producer(), mma()] + [softmax(t, w) for t in (0, 1) for w in range(4)]
    alive = list(range(len(roles)))
    for _ in range(2_000_000):
        if not (alive or pipe or tma):
            return viol
        r = rnd.random()
        if r < 0.15 and pipe:
            kind, x = pipe.pop(0)
            if kind == "mma":
                x()
            else:
                bars[x].arrive()
        elif r < 0.25 and tma:
            name, land = tma.pop(rnd.randrange(len(tma)))
            land()
            bars[name].arrive()
        elif alive:
            i = rnd.choice(alive)
            try:
                next(roles[i])
            except StopIteration:
                alive.remove(i)
    viol.append("no progress")
    return viol


def unit_sequences():
    """Key blocks (tile 0, tile 1) per unit: tile 1 has the same or one more
    (causal), or none (its rows lie past the sequence end); units with no
    block at all; long and one-block units."""
    seqs = [
        [(1, 2), (3, 0), (1, 1), (2, 3), (0, 1), (0, 0), (5, 5), (1, 0), (1, 0), (1, 0), (2, 2), (1, 1)],
        [(1, 1)] * 12,
        [(1, 0)] * 10 + [(2, 3)] * 3,
        [(4, 5), (1, 2), (1, 0), (0, 0), (0, 1), (3, 4), (8, 9)],
    ]
    rnd = random.Random(1)
    for _ in range(16):
        us = []
        for _ in range(rnd.randrange(1, 15)):
            a = rnd.randrange(0, 6)
            r = rnd.random()
            us.append((a, 0) if r < 0.25 and a > 0 else (a, a + (1 if r > 0.5 else 0)))
        seqs.append(us)
    return seqs


@pytest.mark.parametrize("idx", range(20))
def test_persistent_protocol_is_unambiguous_and_hazard_free(idx):
    units = unit_sequences()[idx]
    for seed in range(40):
        viol = simulate(units, seed)
        assert not viol, (units, seed, viol[:3])


def test_two_step_barriers_are_caught():
    # with the step commits on two barriers the producer can fall two phases
    # behind (short units): the model must report it
    found = any(simulate(units, seed, step_bars=2) for units in unit_sequences()[:4] for seed in range(10))
    assert found
