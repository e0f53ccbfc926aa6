"""CPU replay of the tcgen05 verify kernel's barrier protocol, with random interleavings.

Roles: the TMA producer, the MMA issuer and the softmax warps of the two slots (each slot acts
as one party).  A CTA walks a list of work units of n >= 1 key tiles; tile e of a unit belongs
to slot e & 1.  K and V run through rings of 2 and 3 stages (the kernel; 3 and 2 are replayed
too) across units; the
query rows of consecutive units alternate between two buffers and come either by TMA (the
producer, once the unit two back has run its last Q K^T) or from slot 1's threads (right after
it has published the previous unit's row statistics).  At a unit's end slot 1 publishes its
row max and sum once slot 0 has read the previous unit's (o_free), and slot 0 waits for both
slots' last P V and for slot 1's statistics before it frees both O accumulators.  Tensor-core
operations complete in issue order, some time after they are issued; TMA loads land at random
times.  Every parity wait must observe exactly the phase it expects (a barrier two phases
ahead of its waiter would let a parity wait pass on the wrong phase), and no wait may be left
unsatisfiable (a deadlock)."""
import random

import pytest

RINGS = [(2, 3), (3, 2)]      # (K stages, V stages): the kernel's, and the swapped depths


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


def tiles(n, s):
    return (n - s + 1) // 2


def run(units, seed, tma_q=True, ragged=(), rescale_p=0.3, drop_o_free_waits=False, rings=(2, 3)):
    NK, NV = rings
    rnd = random.Random(seed)
    k_full = [Bar(1) for _ in range(NK)]; k_free = [Bar(1) for _ in range(NK)]
    v_full = [Bar(1) for _ in range(NV)]; v_free = [Bar(1) for _ in range(NV)]
    s_full = [Bar(1), Bar(1)]; p_full = [Bar(1), Bar(1)]; pv_done = [Bar(1), Bar(1)]
    o_full = [Bar(1), Bar(1)]; o_free = [Bar(1), Bar(1)]
    q_full = [Bar(1), Bar(1)]; q_free = [Bar(1), Bar(1)]
    ml_ready = Bar(1)
    tma_pending, mma_pending = [], []

    def mma_done(bar):
        mma_pending.append(bar)

    def producer():
        kn = vn = qn = 0
        for n in units:
            if tma_q:
                j = qn & 1
                if qn >= 2:
                    yield lambda j=j, qn=qn: q_free[j].ready((qn - 2) >> 1)
                yield ("load", q_full[j])
                qn += 1
            for _ in range(n):
                if kn >= NK:
                    yield lambda kn=kn: k_free[kn % NK].ready(kn // NK - 1)
                yield ("load", k_full[kn % NK])
                kn += 1
                if vn >= NV:
                    yield lambda vn=vn: v_free[vn % NV].ready(vn // NV - 1)
                yield ("load", v_full[vn % NV])
                vn += 1

    def mma():
        it, ks, nu = 0, [0, 0], 0
        for n in units:
            qb = nu & 1
            yield lambda qb=qb, nu=nu: q_full[qb].ready(nu >> 1)

            def issue_s(e, it=it, n=n, qb=qb):
                st = (it + e) % NK
                yield lambda: k_full[st].ready((it + e) // NK)
                mma_done(s_full[e & 1])
                mma_done(k_free[st])
                if e == n - 1:
                    mma_done(q_free[qb])

            yield from issue_s(0)
            if n > 1:
                yield from issue_s(1)
            for e in range(n):
                s, j, sv = e & 1, e >> 1, (it + e) % NV
                yield lambda s=s, j=j, ks=list(ks): p_full[s].ready(ks[s] + j)
                yield lambda sv=sv, e=e: v_full[sv].ready((it + e) // NV)
                if j == 0 and nu > 0 and not drop_o_free_waits:
                    yield lambda s=s, nu=nu: o_free[s].ready(nu - 1)
                mma_done(pv_done[s])
                mma_done(v_free[sv])
                if e + 2 >= n:
                    mma_done(o_full[s])
                if e + 2 < n:
                    yield from issue_s(e + 2)
            it += n
            ks[0] += tiles(n, 0)
            ks[1] += tiles(n, 1)
            nu += 1

    def softmax(s):
        it = ks = nus = nus1 = nu = 0
        if s == 1 and not tma_q and units:
            q_full[0].arrive()                      # the first unit's rows
        for ui, n in enumerate(units):
            ns = tiles(n, s)
            for j in range(ns):
                e, kk = 2 * j + s, ks + j
                yield lambda kk=kk: s_full[s].ready(kk)
                if ui in ragged and e == n - 1:     # zero the V rows past the chunk first
                    ve = it + e
                    yield lambda ve=ve: v_full[ve % NV].ready(ve // NV)
                if j >= 1 and rnd.random() < rescale_p:   # the row max grew: rescale O
                    yield lambda kk=kk: pv_done[s].ready(kk - 1)
                p_full[s].arrive()
            has1 = tiles(n, 1) > 0
            if s == 1:
                if nu > 0 and not drop_o_free_waits:
                    yield lambda nu=nu: o_free[1].ready(nu - 1)
                ml_ready.arrive()
                if not tma_q and ui + 1 < len(units):
                    j = (nu + 1) & 1
                    if nu >= 1:
                        yield lambda j=j, nu=nu: q_free[j].ready((nu - 1) >> 1)
                    q_full[j].arrive()
            else:
                yield lambda nus=nus: o_full[0].ready(nus)
                yield lambda nu=nu: ml_ready.ready(nu)
                if has1:
                    yield lambda nus1=nus1: o_full[1].ready(nus1)
                o_free[0].arrive()
                o_free[1].arrive()
            it += n
            ks += ns
            nus += 1 if ns > 0 else 0
            nus1 += 1 if has1 else 0
            nu += 1

    threads = {"prod": producer(), "mma": mma(), "s0": softmax(0), "s1": softmax(1)}
    waiting, done = {}, set()
    steps = 0
    while len(done) < len(threads) or tma_pending or mma_pending:
        steps += 1
        if steps > 400000:
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


def _unit_lists(seed, count):
    rnd = random.Random(2000 + seed)
    return [[rnd.randint(1, 6) for _ in range(rnd.randint(1, 6))] for _ in range(count)]


@pytest.mark.parametrize("rings", RINGS)
@pytest.mark.parametrize("tma_q", [True, False])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_verify_unit_walk_phases_stay_in_step(seed, tma_q, rings):
    """Random unit lists (1 to 6 tiles per unit, odd counts leave slot 1 a tile short, a single
    tile leaves it none), both query paths, ragged last tiles and random O rescales."""
    for i, units in enumerate(_unit_lists(seed, 120)):
        rnd = random.Random(i)
        ragged = {u for u in range(len(units)) if rnd.random() < 0.5}
        run(units, seed * 1000 + i, tma_q=tma_q, ragged=ragged, rings=rings)


def test_single_tile_units_leave_slot_one_idle():
    """Units of one tile: slot 1 only publishes empty statistics and (fp32 rows) stages queries."""
    for i in range(50):
        run([1] * 7, i, tma_q=False)
        run([1] * 7, i, tma_q=True)


def test_replay_catches_missing_o_free_waits():
    """The replay must catch a planted mistake: the MMA starting a slot's first P V of a unit and
    slot 1 publishing its statistics without waiting for slot 0 to have read the previous unit's
    O and statistics.  With units of one or two tiles slot 1 then runs a unit ahead of slot 0's
    read-out, and slot 0's waits on o_full / ml_ready find those barriers two phases ahead."""
    failures = 0
    for i in range(100):
        try:
            run([2, 2, 1, 2, 2, 1, 2], i, tma_q=True, drop_o_free_waits=True)
        except AssertionError:
            failures += 1
    assert failures >= 30
