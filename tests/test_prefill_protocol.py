"""CPU replay of the prefill kernel's barrier protocol (TMA producer, MMA issuer, two softmax
slots; K/V ring of 2 stages), with random interleavings.  Every parity wait must observe exactly
the phase it expects: a barrier two phases ahead of its waiter would let a parity wait pass on
the wrong phase.  Slot key-tile ranges cover overlapping, nested and disjoint cases (window
masks give the two slots disjoint ranges); the producer and the MMA walk only the tiles some
slot needs, as the kernel does.  Walking the whole span, including tiles no slot needs, fails
this replay."""
import itertools
import random

import pytest

NS = 2
class Bar:
    def __init__(s, count): s.count, s.pend, s.phase = count, count, 0   # phase = completed phases
    def arrive(s):
        s.pend -= 1
        if s.pend == 0: s.phase += 1; s.pend = s.count
    def ready(s, parity, expect_idx):
        # waiter expects completion #expect_idx (0-based); parity = expect_idx & 1
        assert parity == expect_idx & 1
        if s.phase > expect_idx + 1: raise AssertionError(f"ambiguous: phase {s.phase} vs expect {expect_idx}")
        return s.phase >= expect_idx + 1

def run(js, j0, j1, seed):
    rnd = random.Random(seed)
    act = lambda s, j: js[s] is not None and js[s][0] <= j < js[s][1]
    needed = [j for j in range(j0, j1) if act(0, j) or act(1, j)]
    kv_full = [Bar(1) for _ in range(NS)]; kv_free = [Bar(1) for _ in range(NS)]
    s_full = [Bar(1), Bar(1)]; p_full = [Bar(1), Bar(1)]; pv_done = [Bar(1), Bar(1)]
    # generators = threads; yield a predicate to wait on
    def producer():
        for it, j in enumerate(needed):
            st = it % NS
            if it >= NS:
                yield lambda: kv_free[st].ready((it // NS - 1) & 1, it // NS - 1)
            yield "load", (st, it)
    pending_loads = []
    def mma():
        yield lambda: kv_full[0].ready(0, 0)
        for s in range(2):
            if act(s, needed[0]): s_full[s].arrive()   # S issue+commit (completion modelled instantly)
        for it, j in enumerate(needed):
            st = it % NS
            jn = needed[it + 1] if it + 1 < len(needed) else None
            landed = False
            for s in range(2):
                if act(s, j):
                    k = j - js[s][0]
                    yield lambda k=k, s=s: p_full[s].ready(k & 1, k)
                    pv_done[s].arrive()
                if jn is not None and act(s, jn):
                    if not landed:
                        yield lambda it=it: kv_full[(it + 1) % NS].ready(((it + 1) // NS) & 1, (it + 1) // NS)
                        landed = True
                    s_full[s].arrive()
            kv_free[st].arrive()
    def softmax(s):
        if js[s] is None: return
        nk = js[s][1] - js[s][0]
        for k in range(nk):
            yield lambda k=k: s_full[s].ready(k & 1, k)
            if k >= 1 and rnd.random() < 0.3:
                yield lambda k=k: pv_done[s].ready((k - 1) & 1, k - 1)
            p_full[s].arrive()
        yield lambda: pv_done[s].ready((nk - 1) & 1, nk - 1)
    threads = {"prod": producer(), "mma": mma(), "s0": softmax(0), "s1": softmax(1)}
    waiting = {}
    done = set()
    steps = 0
    while len(done) < len(threads):
        steps += 1
        if steps > 100000: raise AssertionError("deadlock")
        # TMA loads land at random times
        if pending_loads and rnd.random() < 0.5:
            st, it = pending_loads.pop(0); kv_full[st].arrive()
        name = rnd.choice([n for n in threads if n not in done])
        if name in waiting:
            if not waiting[name](): continue
            del waiting[name]
        try:
            ev = next(threads[name])
        except StopIteration:
            done.add(name); continue
        if isinstance(ev, tuple):
            pending_loads.append(ev[1])
        else:
            waiting[name] = ev
    while pending_loads:
        st, it = pending_loads.pop(0); kv_full[st].arrive()



def _cases():
    out = []
    for a0, a1, b0, b1 in itertools.product(range(0, 5), range(1, 6), range(0, 5), range(1, 6)):
        if a1 > a0 and b1 > b0:
            out.append(((a0, a1), (b0, b1)))
    return out


@pytest.mark.parametrize("seed", [0, 1])
def test_protocol_phases_stay_in_step(seed):
    for ra, rb in _cases():
        run([ra, rb], min(ra[0], rb[0]), max(ra[1], rb[1]), seed)
        run([ra, None], ra[0], ra[1], seed)
