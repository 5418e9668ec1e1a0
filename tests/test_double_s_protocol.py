"""A model of the one-tile (head_dim 256) forward kernel's barrier protocol,
run on the CPU.

With one 128-row query tile per CTA the kernel keeps two S buffers in tensor
memory (attention_forward_mbarrier_gb300/csrc/fmha_fwd_kernel.cuh, the
double-buffered S schedule): the MMA thread issues groups g = 0 .. n + 1 of
PV(g - 2) (P from S buffer g % 2) then QK^T(g) (into the same buffer), with a
commit after the PV (VFree[m % 2]: V_m's slot is free) and one after the
QK^T (StepDone[g % 2]: S(g) ready, K_g's slot free); the producer loads the
ring in the order the groups read it (K_0, K_1, V_0, K_2, V_1, ..., V_(n-2),
V_(n-1)) into two slots, refilling a slot after the commit that frees it; the
four softmax warps take S(j) from StepDone, may rescale O once PV(j - 1) has
completed (VFree; it may still run when S(j) is ready), and hand P(j) off on
PVReady[j % 2] because they can run two blocks ahead of the PVs.

The model replays those waits and signals under random interleavings, with
an in-order tensor pipe and copies that land in any order.  Checked on every
parity wait: the parity test agrees with the phase count (never premature,
never stuck two phases behind).  Checked on every access: a slot is not
refilled while an MMA reads it, QK^T and PV read the right blocks, PV reads
the P of its own block, QK^T does not overwrite an unread P, the O rescale
sees PV(j - 1) done and no PV runs during it, and the epilogue reads O after
the last PV.  A variant with a single P barrier must fail (the softmax two
blocks ahead makes its parity ambiguous), which shows the model finds what
it guards against.
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


def ring_block(idx, n):
    """Ring load idx -> ('K' or 'V', key block), the kernel's order."""
    if idx == 0:
        return ("K", 0)
    if n == 1:
        return ("V", 0)
    if idx == 1:
        return ("K", 1)
    if idx == 2 * n - 1:
        return ("V", n - 1)
    r = idx - 2
    return ("V", r >> 1) if r % 2 == 0 else ("K", (r >> 1) + 2)


def release(idx, n):
    """(barrier, phase) after which load idx's slot is free: K_g by the commit
    after QK^T(g) (StepDone[g % 2]), V_m by the commit after PV(m)
    (VFree[m % 2])."""
    kind, blk = ring_block(idx, n)
    if kind == "K":
        return f"SD{blk & 1}", blk >> 1
    return f"VF{blk & 1}", blk >> 1


def simulate(n, seed, p_rescale, p_barriers=2):
    rnd = random.Random(seed)
    bars = {}
    problems = []

    def bar(name, count=1):
        bars[name] = Bar(name, count)

    for name in ("QFull", "KV0", "KV1", "SD0", "SD1", "VF0", "VF1", "OF"):
        bar(name)
    for b in range(p_barriers):
        bar(f"PV{b}", 4)

    def ready(name, k, who):
        b = bars[name]
        seen = (b.done & 1) != (k & 1)
        if seen and b.done <= k:
            problems.append(f"premature {who} {name} phase {k} (done {b.done})")
        if not seen and b.done > k + 1:
            problems.append(f"stuck {who} {name} phase {k} (done {b.done})")
        return b.done > k

    def wait(name, k, who):
        while not ready(name, k, who):
            yield

    def p_bar(m):
        return (f"PV{m % p_barriers}", m // p_barriers)

    pipe, copies = [], []
    st = {"slot": {}, "readers": {0: 0, 1: 0}, "S": {}, "P": {}, "O": None, "o_busy": 0}

    def producer():
        copies.append(("QFull", lambda: None))
        for idx in range(2 * n):
            if idx >= 2:
                yield from wait(*release(idx - 2, n), "producer")
            s = idx % 2
            if st["readers"][s]:
                problems.append(f"slot {s} refilled while read (load {idx})")
            blk = ring_block(idx, n)
            st["slot"][s] = (blk, "loading")
            copies.append((f"KV{s}", lambda s=s, blk=blk: st["slot"].__setitem__(s, (blk, "ok"))))
            yield

    def mma():
        yield from wait("QFull", 0, "mma")
        for g in range(n + 2):
            if g >= 2:
                m = g - 2
                vidx = 2 + 2 * m if m < n - 1 else (1 if n == 1 else 2 * n - 1)
                yield from wait(f"KV{vidx % 2}", vidx // 2, "mma V")
                yield from wait(*p_bar(m), "mma P")
                vs = vidx % 2
                st["readers"][vs] += 1

                def pv(m=m, vs=vs):
                    if st["slot"][vs] != (("V", m), "ok"):
                        problems.append(f"PV({m}) reads {st['slot'][vs]}")
                    if st["P"].get(m % 2) != m:
                        problems.append(f"PV({m}) reads P {st['P'].get(m % 2)}")
                    if st["o_busy"]:
                        problems.append(f"PV({m}) during an O rescale")
                    st["O"] = m
                    st["P"][m % 2] = "used"
                    st["readers"][vs] -= 1

                pipe.append(("mma", pv))
                pipe.append(("commit", f"VF{m & 1}"))
                if m == n - 1:
                    pipe.append(("commit", "OF"))
            if g < n:
                kidx = g if g < 2 else 2 * g - 1
                yield from wait(f"KV{kidx % 2}", kidx // 2, "mma K")
                ks = kidx % 2
                st["readers"][ks] += 1

                def qk(g=g, ks=ks):
                    if st["slot"][ks] != (("K", g), "ok"):
                        problems.append(f"QK({g}) reads {st['slot'][ks]}")
                    if st["P"].get(g % 2) not in (None, "used"):
                        problems.append(f"QK({g}) overwrites the unread P {st['P'][g % 2]}")
                    st["S"][g % 2] = g
                    st["readers"][ks] -= 1

                pipe.append(("mma", qk))
                pipe.append(("commit", f"SD{g & 1}"))
            yield

    def softmax(w):
        for j in range(n):
            yield from wait(f"SD{j & 1}", j >> 1, f"softmax {w}")
            if st["S"].get(j % 2) != j:
                problems.append(f"softmax {w} reads S {st['S'].get(j % 2)} for block {j}")
            yield
            if j > 0 and rnd.random() < p_rescale:
                yield from wait(f"VF{(j - 1) & 1}", (j - 1) >> 1, f"softmax {w} rescale")
                if st["O"] != j - 1:
                    problems.append(f"rescale at block {j} sees O after PV({st['O']})")
                st["o_busy"] += 1
                yield
                st["o_busy"] -= 1
            if w == 0:
                st["P"][j % 2] = j
            bars[p_bar(j)[0]].arrive()
            yield
        yield from wait("OF", 0, f"softmax {w} epilogue")
        if st["O"] != n - 1:
            problems.append("epilogue reads O before the last PV")

    roles = [producer(), mma()] + [softmax(w) for w in range(4)]
    alive = list(range(len(roles)))
    for _ in range(500_000):
        if not (alive or pipe or copies):
            break
        r = rnd.random()
        if r < 0.2 and pipe:
            kind, x = pipe.pop(0)
            if kind == "mma":
                x()
            else:
                bars[x].arrive()
            continue
        if r < 0.3 and copies:
            name, land = copies.pop(rnd.randrange(len(copies)))
            land()
            bars[name].arrive()
            continue
        if alive:
            i = rnd.choice(alive)
            try:
                next(roles[i])
            except StopIteration:
                alive.remove(i)
    else:
        problems.append("no progress")
    return problems


@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 18])
def test_double_s_protocol(n):
    for seed in range(30):
        for p_rescale in (0.0, 0.5, 1.0):
            problems = simulate(n, seed, p_rescale)
            assert not problems, (n, seed, p_rescale, problems[:3])


def test_single_p_barrier_is_caught():
    found = any(simulate(n, seed, 0.0, p_barriers=1) for n in (2, 4, 8) for seed in range(40))
    assert found
