"""CPU replay of the persistent prefill kernel's barrier protocol, with random interleavings.

Roles: the TMA producer, the MMA issuer and the two softmax slots (each slot's four warps act
as one party).  A CTA walks a list of work units; each unit has a key-tile range per slot
(slot 1 may be empty), and the K and V rings of 2 stages each run on across units
(a K stage frees after its tile's Q K^T, a V stage after its P V).  Tensor-core
operations complete in issue order, some time after they are issued; TMA loads land at random
times.  Every parity wait must observe exactly the phase it expects: a barrier two phases
ahead of its waiter would let a parity wait pass on the wrong phase, and a wait that can never
be satisfied is a deadlock.  Both the TMA-staged Q and the thread-staged Q (permuted rows) are
replayed.  Slot key-tile ranges cover overlapping, nested and disjoint cases (window masks give
the two slots disjoint ranges); the producer and the MMA walk only the tiles some slot needs,
as the kernel does."""
import itertools
import random

import pytest

NS = 2


class Bar:
    def __init__(s, count):
        s.count, s.pend, s.phase = count, count, 0   # phase = completed phases

    def arrive(s):
        s.pend -= 1
        assert s.pend >= 0
        if s.pend == 0:
            s.phase += 1
            s.pend = s.count

    def ready(s, expect_idx):
        # the waiter expects completion #expect_idx (0-based) and waits on parity expect_idx & 1
        if s.phase > expect_idx + 1:
            raise AssertionError(f"ambiguous parity wait: phase {s.phase}, expected completion {expect_idx}")
        return s.phase >= expect_idx + 1


def needed_tiles(u):
    act = lambda s, j: u[s] is not None and u[s][0] <= j < u[s][1]
    lo = min(r[0] for r in u if r is not None)
    hi = max(r[1] for r in u if r is not None)
    return [j for j in range(lo, hi) if act(0, j) or act(1, j)], act


def run(units, seed, gather=False, slow_mma=True, walk_all=False, ns=NS):
    rnd = random.Random(seed)
    k_full = [Bar(1) for _ in range(ns)]; k_free = [Bar(1) for _ in range(ns)]
    v_full = [Bar(1) for _ in range(ns)]; v_free = [Bar(1) for _ in range(ns)]
    s_full = [Bar(1), Bar(1)]; p_full = [Bar(1), Bar(1)]; pv_done = [Bar(1), Bar(1)]
    q_full = [Bar(1), Bar(1)]; o_full = [Bar(1), Bar(1)]; o_free = [Bar(1), Bar(1)]
    q_free = Bar(1)
    tma_pending = []        # loads in flight (land in any order)
    mma_pending = []        # tensor-core completions (land in issue order)

    def mma_done(bar):
        if slow_mma:
            mma_pending.append(bar)
        else:
            bar.arrive()

    def producer():
        it = 0
        for nu, u in enumerate(units):
            tiles, act = needed_tiles(u)
            if not gather:
                if nu > 0:
                    yield lambda nu=nu: q_free.ready(nu - 1)
                for s in range(2):
                    if u[s] is not None:
                        yield ("load", q_full[s])
            walk = list(range(tiles[0], tiles[-1] + 1)) if walk_all else tiles
            for j in walk:
                st = it % ns
                if it >= ns:
                    yield lambda st=st, it=it: k_free[st].ready(it // ns - 1)
                yield ("load", k_full[st])
                if it >= ns:
                    yield lambda st=st, it=it: v_free[st].ready(it // ns - 1)
                yield ("load", v_full[st])
                it += 1

    def mma():
        it = 0
        ks = [0, 0]
        nus = [0, 0]
        for u in units:
            tiles, act = needed_tiles(u)
            walk = list(range(tiles[0], tiles[-1] + 1)) if walk_all else tiles
            nk = [0 if u[s] is None else u[s][1] - u[s][0] for s in range(2)]
            s_total = nk[0] + nk[1]
            issued = [0]

            def issue_s(s):
                mma_done(s_full[s])
                issued[0] += 1
                if issued[0] == s_total:
                    mma_done(q_free)

            for s in range(2):
                if u[s] is not None:
                    yield lambda s=s: q_full[s].ready(nus[s])
            yield lambda it=it: k_full[it % ns].ready(it // ns)
            for s in range(2):
                if act(s, walk[0]):
                    issue_s(s)
            mma_done(k_free[it % ns])
            for idx, j in enumerate(walk):
                jn = walk[idx + 1] if idx + 1 < len(walk) else None
                next_landed = v_landed = False
                for s in range(2):
                    if act(s, j):
                        k = j - u[s][0]
                        yield lambda s=s, k=k: p_full[s].ready(ks[s] + k)
                        if not v_landed:
                            yield lambda it=it: v_full[it % ns].ready(it // ns)
                            v_landed = True
                        if k == 0 and nus[s] > 0:
                            yield lambda s=s: o_free[s].ready(nus[s] - 1)
                        mma_done(pv_done[s])
                        if j == u[s][1] - 1:
                            mma_done(o_full[s])
                    if jn is not None and act(s, jn):
                        if not next_landed:
                            yield lambda it=it: k_full[(it + 1) % ns].ready((it + 1) // ns)
                            next_landed = True
                        issue_s(s)
                # with walk_all, a tile neither slot needs frees its stages without waiting
                mma_done(v_free[it % ns])
                if jn is not None:
                    mma_done(k_free[(it + 1) % ns])
                it += 1
            for s in range(2):
                if u[s] is not None:
                    ks[s] += nk[s]
                    nus[s] += 1

    def softmax(s):
        ks = nus = 0
        for nu, u in enumerate(units):
            if u[s] is None:
                continue
            if gather:
                if nu > 0:
                    yield lambda nu=nu: q_free.ready(nu - 1)
                q_full[s].arrive()
            nk = u[s][1] - u[s][0]
            for k in range(nk):
                kk = ks + k
                yield lambda kk=kk: s_full[s].ready(kk)
                if k >= 1 and rnd.random() < 0.3:          # the row max grew: rescale O
                    yield lambda kk=kk: pv_done[s].ready(kk - 1)
                p_full[s].arrive()
            yield lambda: o_full[s].ready(nus)
            o_free[s].arrive()
            ks += nk
            nus += 1

    threads = {"prod": producer(), "mma": mma(), "s0": softmax(0), "s1": softmax(1)}
    waiting = {}
    done = set()
    steps = 0
    while len(done) < len(threads) or tma_pending or mma_pending:
        steps += 1
        if steps > 200000:
            raise AssertionError(f"deadlock: waiting {sorted(waiting)}")
        if tma_pending and rnd.random() < 0.4:
            tma_pending.pop(rnd.randrange(len(tma_pending))).arrive()
        if mma_pending and rnd.random() < 0.4:
            mma_pending.pop(0).arrive()
        live = [n for n in threads if n not in done]
        if not live:
            continue
        name = rnd.choice(live)
        if name in waiting:
            if not waiting[name]():
                continue
            del waiting[name]
        try:
            ev = next(threads[name])
        except StopIteration:
            done.add(name)
            continue
        if isinstance(ev, tuple):
            tma_pending.append(ev[1])
        else:
            waiting[name] = ev


def _ranges():
    return [(a, b) for a in range(0, 4) for b in range(a + 1, 5)]


def _unit_lists(seed, count):
    rnd = random.Random(1000 + seed)
    rs = _ranges()
    out = []
    for _ in range(count):
        n_units = rnd.randint(1, 4)
        units = []
        for _ in range(n_units):
            r0 = rnd.choice(rs)
            r1 = rnd.choice(rs) if rnd.random() < 0.8 else None
            units.append((r0, r1))
        out.append(units)
    return out


@pytest.mark.parametrize("seed", [0, 1])
def test_single_unit_phases_stay_in_step(seed):
    """One unit per CTA, every pair of slot ranges (and an empty slot 1)."""
    for ra, rb in itertools.product(_ranges(), repeat=2):
        run([(ra, rb)], seed)
        run([(ra, None)], seed, slow_mma=False)


@pytest.mark.parametrize("ns", [1, 2])
@pytest.mark.parametrize("gather", [False, True])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_persistent_unit_walk_phases_stay_in_step(seed, gather, ns):
    """Several units per CTA: the rings (one or two stages), the per-slot tile counters and the
    per-unit barriers (q_full, q_free, o_full, o_free) carry their phases across units."""
    for i, units in enumerate(_unit_lists(seed, 150)):
        run(units, seed * 1000 + i, gather=gather, ns=ns)


def test_replay_catches_a_walk_over_unneeded_tiles():
    """The fault once met on the GPU: producer and MMA walked every tile of the union span
    (the slots' ranges are disjoint under a window mask) and the MMA marked the stages of tiles
    neither slot needs free without waiting for them to land, so the ring's barriers ran two
    phases ahead of the producer.  The replay must report it (under most interleavings)."""
    failures = 0
    for i in range(100):
        try:
            run([((0, 1), (4, 5))] * 3, i, walk_all=True)
        except AssertionError:
            failures += 1
    assert failures >= 50
