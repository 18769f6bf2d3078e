"""CPU model of the forward kernel's wind-down after a device-side wait gives up.

Every wait of the tensor-core kernels is bounded: it returns "done" when its phase has
completed, or "gave up" once its CTA's abort flag is raised or its own time limit runs out
(the first wait to run out raises the flag).  A role whose wait gave up stops its loop;
then the producer drains the copies it issued and each MMA issuer commits and waits for
its products (drain waits ignore the abort flag and have a fixed 4 s bound), and only then
is tensor and shared memory released.  In the CTA-pair form the two CTAs each have their
own abort flag and meet at a cluster barrier before either frees its memory.

This model replays the forward's roles (attn_fwd_tc.cu) with that control flow: the
producer(s), the even CTA's two issuers and every softmax warp, each wait able to give up
whenever the kernel's wait could.  Two scenarios:
  * forced: the test knob ra_debug_force_timeout, where each issuer first waits on a
    barrier nothing arrives on, so it always gives up before issuing any product (this is
    what the GPU failure test runs);
  * random: any wait that is blocked may run out of time at any step (a wait limit far
    shorter than some hand-off), anywhere in the run.
For every schedule the model requires that all roles of all CTAs reach the closing
barrier, that no drain wait is left waiting for an event that can no longer come (it
would sit out its 4 s bound), and that when the CTAs pass the closing barrier no copy is
still landing in shared memory or on a barrier and no product is still running.  Planted
wind-down mistakes must be caught.
"""
import random
from collections import defaultdict

import pytest

from test_protocol_model import Bar, ProtocolError, require


class Sim:
    """Random-schedule engine for roles with bounded waits.  Actions a role yields:
      ("bwait", bar, k, cta)      bounded wait; the role is sent True (phase k done) or False
      ("dwait", bar, k)           drain wait: blocks until phase k is done
      ("do", fn)                  run fn now
      ("copy", bar, k, cta, fn)   start a copy into CTA `cta`'s shared memory whose bytes
                                  count toward phase k of bar; fn on landing
      ("mma", issuer, fn)         issue a product (completes in issue order)
      ("commit", issuer, arrivals) arrive on each (bar, phase) once earlier products completed
      ("cbar", name)              barrier of every role (__syncthreads plus the cluster barrier)
    """

    def __init__(self, rng, ncta, p_timeout):
        self.rng, self.p_timeout = rng, p_timeout
        self.abort = [False] * ncta
        self.copies = []
        self.tc = defaultdict(list)
        self.exits = 0

    def run(self, roles, exit_name="exit", max_steps=400000):
        rng = self.rng
        n = len(roles)
        state = [None] * n
        send = [None] * n
        alive = set(range(n))
        at_bar = defaultdict(set)

        done_at_entry = [False] * n

        def advance(i):
            try:
                state[i] = roles[i].send(send[i]) if state[i] is not None else next(roles[i])
            except StopIteration:
                alive.discard(i)
                state[i] = ("end",)
            send[i] = None
            # the kernel's wait tries the barrier once before it looks at the abort flag
            done_at_entry[i] = state[i][0] == "bwait" and state[i][1].test(state[i][2])

        for i in range(n):
            advance(i)
        for _ in range(max_steps):
            if not alive and not self.copies and not any(self.tc.values()):
                return
            choices, timeouts = [], []
            for i in alive:
                a = state[i]
                if a[0] == "bwait":
                    done = a[1].test(a[2])
                    if done or self.abort[a[3]]:
                        choices.append(("role", i))
                    else:
                        timeouts.append(("timeout", i))
                elif a[0] == "dwait":
                    if a[1].test(a[2]):
                        choices.append(("role", i))
                elif a[0] == "cbar":
                    if i not in at_bar[a[1]]:
                        choices.append(("role", i))
                else:
                    choices.append(("role", i))
            if self.copies:
                choices.append(("copy", None))
            choices += [("tc", g) for g, q in self.tc.items() if q]
            if timeouts and (not choices or rng.random() < self.p_timeout):
                choices += timeouts
            if not choices:
                stuck = [state[i] for i in alive]
                drains = [f"{a[1].name} phase {a[2]}" for a in stuck if a[0] == "dwait"]
                if drains:
                    raise ProtocolError("drain left waiting for an event that cannot come (it sits out its 4 s "
                                        "bound): " + ", ".join(drains))
                raise ProtocolError("deadlock: " + ", ".join(str(a[:3]) for a in stuck))
            kind, i = rng.choice(choices)
            if kind == "copy":
                bar, phase, cta, fn = self.copies.pop(rng.randrange(len(self.copies)))
                bar.complete_tx(phase, 1)
                if fn:
                    fn()
            elif kind == "tc":
                op, payload = self.tc[i].pop(0)
                if op == "mma":
                    payload()
                else:
                    for bar, phase in payload:
                        bar.arrive(phase)
            elif kind == "timeout":
                self.abort[state[i][3]] = True
                send[i] = False
                advance(i)
            else:
                a = state[i]
                if a[0] == "bwait":
                    done = a[1].test(a[2])
                    # done already when the wait began: done; done since, with the CTA's abort
                    # flag raised meanwhile: the kernel's wait may have seen either first
                    if done_at_entry[i] or not self.abort[a[3]]:
                        send[i] = done
                    else:
                        send[i] = done and rng.random() < 0.5
                    advance(i)
                elif a[0] == "cbar":
                    at_bar[a[1]].add(i)
                    if len(at_bar[a[1]]) == len(alive):
                        if a[1] == exit_name:
                            self.check_exit()
                        for j in list(at_bar[a[1]]):
                            advance(j)
                else:
                    if a[0] == "copy":
                        self.copies.append((a[1], a[2], a[3], a[4]))
                    elif a[0] == "mma":
                        self.tc[a[1]].append(("mma", a[2]))
                    elif a[0] == "commit":
                        self.tc[a[1]].append(("commit", a[2]))
                    elif a[0] == "do":
                        a[1]()
                    advance(i)
        raise ProtocolError("schedule did not finish")

    def check_exit(self):
        require(not self.copies, f"{len(self.copies)} copies still landing when the CTAs free their memory")
        require(not any(self.tc.values()), "tensor-core work still running when the CTAs free their memory")
        self.exits += 1


class FwdAbortModel:
    """One work item of the forward with the kernel's wind-down (attn_fwd_tc.cu): ncta CTAs
    (1, or a pair), two products, nst ring stages, nkt key tiles (nkt_g[g] for product g).

    form "reconcile": the kernel as it stands.  In a pair the odd producer publishes how
    many ring fills it issued; after a first closing cluster barrier the even producer,
    which owns the barriers both CTAs' copies complete on, arms the fills only the odd CTA
    issued (for the odd CTA's bytes alone) and completes the bytes of those only it issued,
    then drains every fill either issued; a second cluster barrier precedes freeing memory.
    Planted mistakes: "even_drains_own" (the earlier form: the even producer drains only the
    fills it issued), "no_producer_drain", "no_issuer_drain"."""

    NGROUP, WARPS = 2, 4

    def __init__(self, sim, ncta, nst, nkt, nkt_g, forced, form="reconcile"):
        self.sim, self.ncta, self.nst, self.nkt, self.nkt_g = sim, ncta, nst, nkt, nkt_g
        self.forced, self.form = forced, form
        n, G, W = ncta, self.NGROUP, self.WARPS
        self.q_full = Bar("q_full", 1)
        self.ring_full = [Bar(f"ring_full[{i}]", 1) for i in range(nst)]
        self.ring_empty = [[Bar(f"ring_empty[{i}]@{r}", G) for i in range(nst)] for r in range(n)]
        self.s_full = [[[Bar(f"s_full[{g}][{b}]@{r}", 1) for b in range(2)] for g in range(G)] for r in range(n)]
        self.s_empty = [[Bar(f"s_empty[{g}][{b}]", n * W) for b in range(2)] for g in range(G)]
        self.p_full = [Bar(f"p_full[{g}]", n * W) for g in range(G)]
        self.p_empty = [[Bar(f"p_empty[{g}]@{r}", 1) for g in range(G)] for r in range(n)]
        self.o_full = [[Bar(f"o_full[{g}]@{r}", 1) for g in range(G)] for r in range(n)]
        self.drain = [[Bar(f"drain[{g}]@{r}", 1) for g in range(G)] for r in range(n)]
        self.stage_use = [[-1] * nst for _ in range(n)]
        self.s_written = defaultdict(set)
        self.outstanding = defaultdict(int)   # per issuer
        self.issued = [0] * n

    def closing(self):
        if self.form == "reconcile":
            yield ("cbar", "A")
        yield ("cbar", "exit")

    def fills(self):
        out = [("K", j) for j in range(self.nkt)] + [("K", 0)]
        for j in range(1, self.nkt):
            out += [("K", j), ("V", j - 1)]
        return out + [("V", self.nkt - 1)]

    def producer(self, r):
        n, nst = self.ncta, self.nst
        arms = r == 0
        if arms:
            yield ("do", lambda: self.q_full.arrive(0, tx=n))
        yield ("copy", self.q_full, 0, r, None)
        issued = 0
        for it, _ in enumerate(self.fills()):
            st, use = it % nst, it // nst
            ok = yield ("bwait", self.ring_empty[r][st], use - 1, r)
            if not ok:
                break
            if arms:
                yield ("do", lambda st=st, use=use: self.ring_full[st].arrive(use, tx=n))

            def land(st=st, use=use):
                self.stage_use[r][st] = use
            yield ("copy", self.ring_full[st], use, r, land)
            issued += 1
        self.issued[r] = issued

        def drain_upto(total):
            yield ("dwait", self.q_full, 0)
            for st in range(nst):
                last = [f // nst for f in range(total) if f % nst == st]
                if last:
                    yield ("dwait", self.ring_full[st], last[-1])

        if self.form == "reconcile":
            yield ("cbar", "A")
            if arms:
                other = self.issued[n - 1]
                for f in range(min(issued, other), max(issued, other)):
                    st, use = f % nst, f // nst
                    if f >= issued:   # only the odd CTA issued it: arm for its bytes alone
                        yield ("do", lambda st=st, use=use: self.ring_full[st].arrive(use, tx=1))
                    else:             # only this CTA did: the odd CTA's bytes will not come
                        yield ("do", lambda st=st, use=use: self.ring_full[st].complete_tx(use, 1))
                yield from drain_upto(max(issued, other))
            yield ("cbar", "exit")
            return
        if arms and self.form != "no_producer_drain":
            yield from drain_upto(issued)
        yield ("cbar", "exit")

    def issuer(self, g):
        n, nst, nkt, nkt_g = self.ncta, self.nst, self.nkt, self.nkt_g[g]
        uses = [0, 0]

        def ring_wait(p):
            st, use = p % nst, p // nst
            ok = yield ("bwait", self.ring_full[st], use, 0)
            if ok:
                for r in range(n):
                    require(self.stage_use[r][st] == use, f"product reads stage {st} use {use} before CTA {r}'s copy")
            return ok

        def release(p):
            yield ("commit", g, [(self.ring_empty[r][p % nst], p // nst) for r in range(n)])

        def product(done):
            self.outstanding[g] += 1

            def complete():
                self.outstanding[g] -= 1
                done()
            return ("mma", g, complete)

        def mma_s(b):
            use = uses[b]
            ok = yield ("bwait", self.s_empty[g][b], use - 1, 0)
            if not ok:
                return False
            yield product(lambda: self.s_written[(g, b)].add(use))
            yield ("commit", g, [(self.s_full[r][g][b], use) for r in range(n)])
            uses[b] += 1
            return True

        def mma_pv(j):
            ok = yield ("bwait", self.p_full[g], j, 0)
            if not ok:
                return False
            yield product(lambda: None)
            yield ("commit", g, [(self.p_empty[r][g], j) for r in range(n)])
            return True

        ok = yield ("bwait", self.q_full, 0, 0)
        if ok and self.forced:   # the test knob: nothing arrives on this barrier before the commit below
            ok = yield ("bwait", self.drain[0][g], 0, 0)
        pos = 0
        for j in range(nkt):
            if not ok:
                break
            ok = yield from ring_wait(pos)
            if ok and j < nkt_g:
                ok = yield from mma_s(j & 1)
            if ok:
                yield from release(pos)
            pos += 1
        if ok:
            ok = yield from ring_wait(pos)
        if ok:
            ok = yield from mma_s(0)
        if ok:
            yield from release(pos)
        pos += 1
        for j in range(nkt):
            if not ok:
                break
            if j + 1 < nkt:
                kpos, pos = pos, pos + 1
                ok = yield from ring_wait(kpos)
                if ok and j + 1 < nkt_g:
                    ok = yield from mma_s(0)
                if ok:
                    yield from release(kpos)
            vpos, pos = pos, pos + 1
            if ok:
                ok = yield from ring_wait(vpos)
            if ok and j < nkt_g:
                ok = yield from mma_pv(j)
            if ok:
                yield from release(vpos)
        if ok:
            yield ("commit", g, [(self.o_full[r][g], 0) for r in range(n)])
        if self.form != "no_issuer_drain":
            yield ("commit", g, [(self.drain[r][g], 0) for r in range(n)])
            yield ("dwait", self.drain[0][g], 0)
        yield from self.closing()

    def softmax(self, r, g, w):
        nkt_g = self.nkt_g[g]
        ok = True

        def take(b, use):
            ok = yield ("bwait", self.s_full[r][g][b], use, r)
            if not ok:
                return False
            require(use in self.s_written[(g, b)], f"S[{g}][{b}] use {use} read before its product completed")
            yield ("do", lambda: self.s_empty[g][b].arrive(use))
            return True

        for j in range(nkt_g):
            if not ok:
                break
            ok = yield from take(j & 1, j >> 1)
        sidx = (nkt_g + 1) >> 1
        for j in range(nkt_g):
            if not ok:
                break
            ok = yield from take(0, sidx)
            if not ok:
                break
            sidx += 1
            ok = yield ("bwait", self.p_empty[r][g], j - 1, r)
            if not ok:
                break
            yield ("do", lambda j=j: self.p_full[g].arrive(j))
        if ok:
            ok = yield ("bwait", self.o_full[r][g], 0, r)
            if ok:
                require(self.outstanding[g] == 0, f"O[{g}] read while its products are outstanding")
        yield from self.closing()

    def idle(self):
        yield from self.closing()

    def roles(self):
        out = [self.producer(r) for r in range(self.ncta)] + [self.issuer(g) for g in range(self.NGROUP)]
        out += [self.idle() for _ in range(self.ncta - 1) for _ in range(self.NGROUP)]   # odd CTA's issuer warps
        return out + [self.softmax(r, g, w) for r in range(self.ncta) for g in range(self.NGROUP)
                      for w in range(self.WARPS)]


# (CTAs, ring stages, key tiles, key tiles of product 0)
ABORT_CONFIGS = [(1, 3, 1, 1), (1, 3, 4, 4), (1, 6, 5, 3), (2, 6, 1, 1), (2, 6, 4, 4), (2, 6, 9, 7), (2, 6, 2, 1)]


def _run(ncta, nst, nkt, nkt0, forced, seed, form="reconcile", p_timeout=0.01):
    rng = random.Random(seed)
    sim = Sim(rng, ncta, p_timeout)
    model = FwdAbortModel(sim, ncta, nst, nkt, (nkt0, nkt), forced, form)
    sim.run(model.roles())
    require(sim.exits == 1, "the CTAs never passed the closing barrier")
    return sim


@pytest.mark.parametrize("ncta,nst,nkt,nkt0", ABORT_CONFIGS)
def test_forced_timeout_winds_down_cleanly(ncta, nst, nkt, nkt0):
    """The GPU failure test's scenario: each issuer gives up before its first product."""
    for seed in range(150):
        sim = _run(ncta, nst, nkt, nkt0, True, seed * 31 + nkt)
        assert sim.abort[0]


@pytest.mark.parametrize("ncta,nst,nkt,nkt0", ABORT_CONFIGS)
def test_timeouts_anywhere_wind_down_cleanly(ncta, nst, nkt, nkt0):
    """Any blocked wait may run out at any moment, in either CTA, mid-run."""
    for seed in range(300):
        _run(ncta, nst, nkt, nkt0, False, seed * 17 + nkt, p_timeout=0.02)


def _wind_down_caught(ncta, nst, nkt, nkt0, forced, form, seeds=400):
    for seed in range(seeds):
        try:
            _run(ncta, nst, nkt, nkt0, forced, seed, form, p_timeout=0.02)
        except ProtocolError:
            return True
    return False


@pytest.mark.parametrize("form,ncta,forced", [("even_drains_own", 2, False), ("no_producer_drain", 1, True),
                                              ("no_producer_drain", 2, True), ("no_issuer_drain", 1, False),
                                              ("no_issuer_drain", 2, False)])
def test_planted_wind_down_mistakes_are_caught(form, ncta, forced):
    """Draining only the even CTA's own fills leaves it waiting for odd-CTA bytes that will
    not come, or frees memory with an odd-CTA copy still landing, when the two producers
    gave up after different numbers of fills; skipping the producer's drain frees memory
    under landing copies; skipping the issuers' drain frees it under running products."""
    assert _wind_down_caught(ncta, 6 if ncta == 2 else 3, 6, 4, forced, form)


def test_earlier_form_is_sound_under_the_forced_timeout():
    """With the test knob no product is issued, so both producers stop after the same fills:
    the earlier form winds down cleanly in that scenario (the GPU failure test's), and only
    timeouts in mid-run tell the two forms apart."""
    for seed in range(150):
        _run(2, 6, 5, 3, True, seed, "even_drains_own")
