"""CPU models of the tensor-core kernels' barrier protocols, run on random schedules.

The kernels hand work between roles only through mbarriers: TMA producers, MMA-issuing
threads and softmax warps.  Each model replays every role's waits, arrivals, copies,
products and commits in the kernel's order, with the hardware's rules:
  * a wait on phase k tests the parity of the barrier's phase counter, so it would pass
    wrongly if the barrier were one phase behind and block wrongly if it were two ahead;
  * a phase completes when its expected arrivals have come and its transaction bytes are in
    (copy bytes may land before the arming arrival);
  * copies and products complete asynchronously, a commit arrives once every product its
    thread issued before it has completed, and a commit of a CTA pair lands on both CTAs.
For every random schedule the engine checks that all roles finish (no deadlock), that every
wait sees exactly the phase it means, and that every arrival and copy lands in the phase it
is meant for; each model adds checks that no buffer is rewritten while a reader still needs
it.  Planted protocol mistakes must be caught.

Models: the forward (attn_fwd_tc.cu), as one CTA and as a CTA pair, and both kernels of
the backward (attn_bwd_tc.cu).
"""
import random
from collections import defaultdict

import pytest


class ProtocolError(AssertionError):
    pass


class Bar:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.pending, self.tx, self.completed = 0, 0, 0

    def _check_phase(self, phase, what):
        if self.completed != phase:
            raise ProtocolError(f"{self.name}: {what} for phase {phase} while the barrier is in phase {self.completed}")

    def _maybe_complete(self):
        if self.pending == self.count and self.tx == 0:
            self.pending, self.completed = 0, self.completed + 1

    def arrive(self, phase, tx=0):
        self._check_phase(phase, "arrival")
        self.tx += tx
        self.pending += 1
        self._maybe_complete()

    def complete_tx(self, phase, n):
        self._check_phase(phase, "copy completion")
        self.tx -= n
        self._maybe_complete()

    def test(self, k):
        """Hardware parity test for the completion of phase k (k = -1: the phase before the first)."""
        done = (self.completed & 1) != (k & 1)
        if done and self.completed != k + 1:
            raise ProtocolError(f"{self.name}: wait for phase {k} passed with {self.completed} phases completed")
        if not done and self.completed != k:
            raise ProtocolError(f"{self.name}: wait for phase {k} blocks with {self.completed} phases completed")
        return done


def require(cond, msg):
    if not cond:
        raise ProtocolError(msg)


def run_roles(roles, rng, max_steps=400000, slow=()):
    """Run role generators to completion on a random schedule.  Actions:
      ("wait", bar, k)            block until phase k of bar has completed
      ("do", fn)                  run fn now (an arrival, a state change, a check)
      ("copy", bar, k, fn)        start a copy whose bytes complete phase k of bar; fn on landing
      ("mma", issuer, fn)         issue a product; fn when it completes (in issue order)
      ("commit", issuer, arrivals) arrive on each (bar, phase) once the issuer's earlier products completed
    Roles listed in `slow` are scheduled only one time in fifty while anything else can move:
    a thread that falls far behind the others.
    """
    state = [None] * len(roles)
    alive = set(range(len(roles)))
    tc = defaultdict(list)
    copies = []

    def advance(i):
        try:
            state[i] = next(roles[i])
        except StopIteration:
            alive.discard(i)
            state[i] = None

    for i in range(len(roles)):
        advance(i)
    for _ in range(max_steps):
        if not alive and not copies and not any(tc.values()):
            return
        choices = [("role", i) for i in alive if state[i][0] != "wait" or state[i][1].test(state[i][2])]
        if copies:
            choices.append(("copy", None))
        choices += [("tc", g) for g, q in tc.items() if q]
        if not choices:
            raise ProtocolError("deadlock: " + ", ".join(
                f"{state[i][1].name} phase {state[i][2]}" for i in alive if state[i][0] == "wait"))
        if slow:
            fast = [c for c in choices if not (c[0] == "role" and c[1] in slow)]
            if fast and len(fast) < len(choices) and rng.random() < 0.98:
                choices = fast
        kind, i = rng.choice(choices)
        if kind == "copy":
            bar, phase, fn = copies.pop(rng.randrange(len(copies)))
            bar.complete_tx(phase, 1)
            if fn:
                fn()
        elif kind == "tc":
            op, payload = tc[i].pop(0)
            if op == "mma":
                payload()
            else:
                for bar, phase in payload:
                    bar.arrive(phase)
        else:
            a = state[i]
            if a[0] == "copy":
                copies.append((a[1], a[2], a[3]))
            elif a[0] == "mma":
                tc[a[1]].append(("mma", a[2]))
            elif a[0] == "commit":
                tc[a[1]].append(("commit", a[2]))
            elif a[0] == "do":
                a[1]()
            advance(i)
    raise ProtocolError("schedule did not finish")


# ---------------------------------------------------------------------------- forward

class ForwardModel:
    """One work item of the forward: NCTA CTAs (1, or a pair), two products (query tiles, or
    pairs of them), NST ring stages, and the key tiles each product takes (takes[g]: its causal
    range, less the tiles a tile live map shows fully masked).  The producer streams the tiles
    either product takes; a tile neither takes is in no pass."""

    NGROUP, WARPS = 2, 4

    def __init__(self, ncta, nst, takes, dead, mutation=None):
        self.ncta, self.nst, self.dead, self.mutation = ncta, nst, dead, mutation
        self.takes = [sorted(t) for t in takes]
        self.tiles = sorted(set(takes[0]) | set(takes[1]))   # the walk: tiles either product takes
        n, G, W = ncta, self.NGROUP, self.WARPS
        sw = W if mutation == "single_cta_counts" else n * W
        self.q_full = Bar("q_full", 1)
        self.ring_full = [Bar(f"ring_full[{i}]", 1) for i in range(nst)]
        self.ring_empty = [[Bar(f"ring_empty[{i}]@{r}", G) for i in range(nst)] for r in range(n)]
        self.s_full = [[[Bar(f"s_full[{g}][{b}]@{r}", 1) for b in range(2)] for g in range(G)] for r in range(n)]
        self.s_empty = [[Bar(f"s_empty[{g}][{b}]", sw) for b in range(2)] for g in range(G)]
        self.p_full = [Bar(f"p_full[{g}]", sw) for g in range(G)]
        self.p_empty = [[Bar(f"p_empty[{g}]@{r}", 1) for g in range(G)] for r in range(n)]
        self.o_full = [[Bar(f"o_full[{g}]@{r}", 1) for g in range(G)] for r in range(n)]
        self.stage_use = [[-1] * nst for _ in range(n)]   # use whose copy has landed, per CTA
        self.stage_readers = [defaultdict(int) for _ in range(nst)]
        self.s_written = defaultdict(set)    # (g, b) -> uses whose product completed
        self.s_readers = defaultdict(int)    # (g, b, use) -> warps reading
        self.s_tile = {}                     # (g, b, use) -> key tile whose scores the use holds
        self.p_written = defaultdict(set)    # (g, c) -> warps that wrote the c-th P tile
        self.p_tile = {}                     # (g, c) -> key tile of the c-th P tile
        self.pv_done = set()                 # (g, c): the c-th P V product completed (or was skipped)
        self.pv_issued = defaultdict(int)
        self.outstanding = defaultdict(int)

    def producer(self, r):
        n, nst, t = self.ncta, self.nst, self.tiles
        arms = r == 0
        if arms:
            yield ("do", lambda: self.q_full.arrive(0, tx=n))
        yield ("copy", self.q_full, 0, None)
        fills = [("K", j) for j in t]
        if t:
            fills.append(("K", t[0]))
            for i in range(1, len(t)):
                fills += [("K", t[i]), ("V", t[i - 1])]
            fills.append(("V", t[-1]))
        for it, _ in enumerate(fills):
            st, use = it % nst, it // nst
            yield ("wait", self.ring_empty[r][st], use - 1)
            for u, left in self.stage_readers[st].items():
                require(not (u < use and left), f"stage {st} refilled (use {use}) while use {u} still has readers")
            if arms:
                yield ("do", lambda st=st, use=use: self.ring_full[st].arrive(use, tx=n))

            def land(r=r, st=st, use=use):
                self.stage_use[r][st] = use
            yield ("copy", self.ring_full[st], use, land)

    def issuer(self, g):
        n, nst, t = self.ncta, self.nst, self.tiles
        mine = set(self.takes[g])
        yield ("wait", self.q_full, 0)
        uses = [0, 0]

        def ring_wait(p):
            st, use = p % nst, p // nst
            yield ("wait", self.ring_full[st], use)
            for r in range(n):
                require(self.stage_use[r][st] == use, f"product reads stage {st} use {use} before CTA {r}'s copy landed")

        def release(p):
            yield ("commit", g, [(self.ring_empty[r][p % nst], p // nst) for r in range(n)])

        def product(reads_stage, done):
            st, suse = reads_stage
            self.stage_readers[st][suse] += 1
            self.outstanding[g] += 1

            def complete():
                self.stage_readers[st][suse] -= 1
                self.outstanding[g] -= 1
                done()
            return ("mma", g, complete)

        def mma_s(p, b, j):
            use = uses[b]
            yield ("wait", self.s_empty[g][b], use - 1)
            require(not any(self.s_readers[(g, b, u)] for u in range(use)),
                    f"S[{g}][{b}] use {use} written while an earlier use is being read")
            require(not (b == 1 and self.pv_issued[g]), f"pass-1 S into O[{g}]'s columns after a P V product")
            self.s_tile[(g, b, use)] = j
            yield product((p % nst, p // nst), lambda: self.s_written[(g, b)].add(use))
            yield ("commit", g, [(self.s_full[r][g][b], use) for r in range(n)])
            uses[b] += 1

        def mma_pv(j, c, p):
            yield ("wait", self.p_full[g], c)
            require(len(self.p_written[(g, c)]) == n * self.WARPS, f"P V product {c} issued before every warp wrote P[{g}]")
            require(self.p_tile[(g, c)] == j, f"P V product of tile {j} reads the P tile of tile {self.p_tile[(g, c)]}")
            require(not any(self.s_readers[(g, 1, u)] for u in range(uses[1])),
                    f"P V product into O[{g}] while pass-1 scores in its columns are read")
            if (g, j) in self.dead:
                self.pv_done.add((g, c))
            else:
                self.pv_issued[g] += 1
                yield product((p % nst, p // nst), lambda: self.pv_done.add((g, c)))
            yield ("commit", g, [(self.p_empty[r][g], c) for r in range(n)])

        skip_wait = self.mutation == "release_without_fill"
        pos = 0
        c = 0
        for j in t:                                            # pass 1
            if not (skip_wait and j not in mine):
                yield from ring_wait(pos)
                if j in mine:
                    yield from mma_s(pos, c & 1, j)
                    c += 1
            yield from release(pos)
            pos += 1
        if t:                                                  # pass 2: S(t0)
            yield from ring_wait(pos)
            if t[0] in mine:
                yield from mma_s(pos, 0, t[0])
            yield from release(pos)
            pos += 1
        c = 0
        for i, j in enumerate(t):
            if i + 1 < len(t):
                jn = t[i + 1]
                if not (skip_wait and jn not in mine):
                    yield from ring_wait(pos)
                    if jn in mine:
                        yield from mma_s(pos, 0, jn)
                yield from release(pos)
                pos += 1
            if not (skip_wait and j not in mine):
                yield from ring_wait(pos)
                if j in mine:
                    yield from mma_pv(j, c, pos)
                    c += 1
            yield from release(pos)
            pos += 1
        yield ("commit", g, [(self.o_full[r][g], 0) for r in range(n)])

    def softmax(self, r, g, w):
        mine = self.takes[g]

        def take(b, use, j):
            yield ("wait", self.s_full[r][g][b], use)
            require(use in self.s_written[(g, b)], f"S[{g}][{b}] use {use} read before its product completed")
            require(self.s_tile[(g, b, use)] == j, f"S[{g}][{b}] use {use} holds tile {self.s_tile[(g, b, use)]}, "
                                                   f"read as tile {j}")
            self.s_readers[(g, b, use)] += 1
            yield ("do", lambda: None)
            self.s_readers[(g, b, use)] -= 1
            yield ("do", lambda: self.s_empty[g][b].arrive(use))

        for c, j in enumerate(mine):                           # pass 1
            if self.mutation == "tile_index_buffers":          # buffer and use by key tile, not by count
                yield from take(j & 1, j >> 1, j)
            else:
                yield from take(c & 1, c >> 1, j)
        sidx = (len(mine) + 1) >> 1
        for c, j in enumerate(mine):                           # pass 2
            yield from take(0, sidx, j)
            sidx += 1
            if self.mutation != "no_p_free_wait":
                yield ("wait", self.p_empty[r][g], c - 1)
            require(c == 0 or (g, c - 1) in self.pv_done, f"P[{g}] rewritten (tile {j}) before the previous P V product completed")
            self.p_written[(g, c)].add((r, w))
            self.p_tile[(g, c)] = j
            yield ("do", lambda c=c: self.p_full[g].arrive(c))
        yield ("wait", self.o_full[r][g], 0)
        require(self.outstanding[g] == 0, f"O[{g}] read while products are outstanding")

    def roles(self):
        out = [self.producer(r) for r in range(self.ncta)] + [self.issuer(g) for g in range(self.NGROUP)]
        return out + [self.softmax(r, g, w) for r in range(self.ncta) for g in range(self.NGROUP)
                      for w in range(self.WARPS)]


FWD_CONFIGS = [
    # (CTAs, ring stages, key tiles, key tiles of the shorter product, which product is shorter,
    # dead fraction).  Under a causal mask product 0 ends earlier (the kernel's order); the
    # configurations with product 1 shorter check that the protocol does not depend on which.
    (1, 3, 1, 1, 0, 0.0), (1, 3, 4, 4, 0, 0.0), (1, 3, 5, 4, 0, 0.3), (1, 6, 3, 3, 0, 0.5), (1, 6, 7, 6, 0, 0.0),
    (2, 6, 1, 1, 1, 0.0), (2, 6, 4, 4, 1, 0.0), (2, 6, 5, 4, 1, 0.3), (2, 6, 9, 8, 1, 0.2), (2, 6, 2, 1, 1, 0.0),
    (2, 6, 5, 3, 0, 0.3), (2, 6, 6, 5, 1, 0.0),
]


@pytest.mark.parametrize("ncta,nst,nkt,nshort,short,dead_frac", FWD_CONFIGS)
def test_forward_protocol_holds_on_random_schedules(ncta, nst, nkt, nshort, short, dead_frac):
    takes = (range(nshort), range(nkt)) if short == 0 else (range(nkt), range(nshort))
    for seed in range(60):
        rng = random.Random(seed * 1000 + nkt * 10 + ncta)
        dead = {(g, j) for g in range(2) for j in range(nkt) if rng.random() < dead_frac}
        run_roles(ForwardModel(ncta, nst, takes, dead).roles(), rng)
    # one role far behind the others: a producer, either issuer, a softmax warp
    for slow in (0, ncta, ncta + 1, ncta + 2):
        for seed in range(20):
            rng = random.Random(seed * 31 + slow)
            dead = {(g, j) for g in range(2) for j in range(nkt) if rng.random() < dead_frac}
            run_roles(ForwardModel(ncta, nst, takes, dead).roles(), rng, slow={slow})


@pytest.mark.parametrize("ncta,nst,nkt", [(1, 3, 6), (1, 6, 9), (2, 6, 6), (2, 6, 11)])
def test_forward_protocol_holds_with_tile_live_maps(ncta, nst, nkt):
    """Under an attention mask each product takes a subset of its range (the tiles the live map
    shows an allowed pair in): random subsets, often different for the two products, sometimes
    one or both empty."""
    for seed in range(80):
        rng = random.Random(seed * 7919 + nkt * 31 + ncta)
        hi = (rng.randint(0, nkt), nkt) if rng.random() < 0.5 else (nkt, rng.randint(0, nkt))
        takes = [{j for j in range(hi[g]) if rng.random() < 0.6} for g in range(2)]
        if seed % 9 == 0:
            takes[seed % 2] = set()
        if seed % 27 == 0:
            takes = [set(), set()]
        dead = {(g, j) for g in range(2) for j in range(nkt) if rng.random() < 0.2}
        run_roles(ForwardModel(ncta, nst, takes, dead).roles(), rng)


def _caught(make, seeds=300):
    for seed in range(seeds):
        try:
            run_roles(make().roles(), random.Random(seed))
        except ProtocolError:
            return True
    return False


@pytest.mark.parametrize("mutation,ncta,takes0,takes1", [("release_without_fill", 1, range(3), range(6)),
                                                         ("release_without_fill", 2, range(2), range(6)),
                                                         ("release_without_fill", 2, range(6), range(2)),
                                                         ("release_without_fill", 2, {0, 2, 5}, {1, 2, 3, 4}),
                                                         ("single_cta_counts", 2, range(3), range(3)),
                                                         ("no_p_free_wait", 1, range(4), range(4)),
                                                         ("no_p_free_wait", 2, {1, 3}, {0, 1, 3, 4}),
                                                         ("tile_index_buffers", 1, {0, 2, 3, 5}, {0, 2, 3, 5}),
                                                         ("tile_index_buffers", 2, {1, 2}, {0, 1, 2, 4})])
def test_planted_forward_protocol_mistakes_are_caught(mutation, ncta, takes0, takes1):
    """Releasing ring stages without waiting for their fill lets the issuer that skips tiles
    run a phase ahead; counting one CTA's warps on the pair's barriers completes a phase
    early; skipping the P-free wait rewrites P under a running product; picking a score buffer
    by key tile instead of by the product's own tile count breaks once the walk has holes."""
    assert _caught(lambda: ForwardModel(ncta, 6 if ncta == 2 else 3, (takes0, takes1), set(), mutation))


# ---------------------------------------------------------------------------- dK/dV kernel

class DkdvModel:
    """One key tile of the dK/dV kernel over nq query tiles: a producer (Q and dO tiles in
    rings of NQS and NDS slots, the per-query constants X and Y as bulk copies), issuer 0
    (S^T = K Q^T and dP^T = V dO^T), issuer 1 (dV += P^T dO, P^T read from tensor memory over
    the S^T columns, then dK += dS^T Q) and the softmax warps (P^T into tensor memory, dS^T
    into a shared tile).  P^T is handed over in two halves (the first and second 16 query
    columns of every warp, p_full[0] and p_full[1]); dV takes each half as it lands."""

    def __init__(self, nq, nqs, nds, warps=4, mutation=None):
        self.nq, self.nqs, self.nds, self.W, self.mutation = nq, nqs, nds, warps, mutation
        W = warps
        self.kv_full = Bar("kv_full", 1)
        self.q_full = [Bar(f"q_full[{i}]", 1) for i in range(nqs)]
        self.q_empty = [Bar(f"q_empty[{i}]", 2) for i in range(nqs)]
        self.do_full = [Bar(f"do_full[{i}]", 1) for i in range(nds)]
        self.do_empty = [Bar(f"do_empty[{i}]", 2) for i in range(nds)]
        self.st_full = Bar("st_full", 2)      # issuer 0's commit + the producer's arming for X
        self.dpt_full = Bar("dpt_full", 2)    # issuer 0's commit + the producer's arming for Y
        self.dpt_free = Bar("dpt_free", W)
        self.p_full = [Bar(f"p_full[{h}]", W) for h in range(2)]
        self.p_free = Bar("p_free", 1)
        self.acc_full = Bar("acc_full", 1)
        self.cx_empty = Bar("cx_empty", W)
        self.cy_empty = Bar("cy_empty", W)
        self.ds_full = Bar("ds_full", W)
        self.ds_free = Bar("ds_free", 1)
        # data state
        self.q_slot = [-1] * nqs          # tile whose Q has landed in each slot
        self.do_slot = [-1] * nds
        self.q_readers = defaultdict(int)  # tile -> products reading its Q
        self.do_readers = defaultdict(int)
        self.x_tile = self.y_tile = -1     # constants that have landed
        self.x_readers = defaultdict(int)
        self.y_readers = defaultdict(int)
        self.st_tile = -1                  # tile whose S^T product has completed (P^T then goes over it)
        self.st_readers = 0
        self.pt_written = defaultdict(set)   # (tile, half) -> warps that wrote that half of P^T
        self.dpt_tile, self.dpt_readers = -1, 0
        self.ds_written = defaultdict(set)
        self.ds_reading = -1               # tile whose dS^T the running dK product reads
        self.outstanding = 0

    def producer(self):
        nq, nqs, nds = self.nq, self.nqs, self.nds
        yield ("do", lambda: self.kv_full.arrive(0, tx=1))
        yield ("copy", self.kv_full, 0, None)
        for it in range(nq):
            qs, ds = it % nqs, it % nds
            yield ("wait", self.q_empty[qs], it // nqs - 1)
            require(not any(v for t, v in self.q_readers.items() if t < it and t % nqs == qs),
                    f"Q slot {qs} refilled (tile {it}) while read")
            yield ("do", lambda qs=qs, it=it: self.q_full[qs].arrive(it // nqs, tx=1))
            yield ("copy", self.q_full[qs], it // nqs, lambda qs=qs, it=it: self.q_slot.__setitem__(qs, it))
            yield ("wait", self.cx_empty, it - 1)
            require(not any(v for t, v in self.x_readers.items() if t < it), f"X rewritten (tile {it}) while read")
            yield ("do", lambda it=it: self.st_full.arrive(it, tx=1))
            yield ("copy", self.st_full, it, lambda it=it: setattr(self, "x_tile", it))
            yield ("wait", self.do_empty[ds], it // nds - 1)
            require(not any(v for t, v in self.do_readers.items() if t < it and t % nds == ds),
                    f"dO slot {ds} refilled (tile {it}) while read")
            yield ("do", lambda ds=ds, it=it: self.do_full[ds].arrive(it // nds, tx=1))
            yield ("copy", self.do_full[ds], it // nds, lambda ds=ds, it=it: self.do_slot.__setitem__(ds, it))
            yield ("wait", self.cy_empty, it - 1)
            if self.mutation != "y_before_dk":
                yield ("wait", self.ds_free, it - 1)
            require(not any(v for t, v in self.y_readers.items() if t < it), f"Y rewritten (tile {it}) while read")
            yield ("do", lambda it=it: self.dpt_full.arrive(it, tx=1))
            yield ("copy", self.dpt_full, it, lambda it=it: setattr(self, "y_tile", it))

    def _product(self, who, done):
        self.outstanding += 1

        def complete():
            self.outstanding -= 1
            done()
        return ("mma", who, complete)

    def issuer0(self):
        nqs, nds = self.nqs, self.nds
        yield ("wait", self.kv_full, 0)
        for it in range(self.nq):
            qs, ds = it % nqs, it % nds
            yield ("wait", self.q_full[qs], it // nqs)
            yield ("wait", self.p_free, it - 1)
            require(self.q_slot[qs] == it, f"S^T of tile {it} issued before its Q landed")
            require(self.st_readers == 0 and (it == 0 or self.pt_read_done),
                    f"S^T of tile {it} overwrites the S^T/P^T columns while in use")
            self.q_readers[it] += 1

            def s_done(it=it):
                self.q_readers[it] -= 1
                self.st_tile = it
                self.pt_read_done = False
            yield self._product(0, s_done)
            yield ("commit", 0, [(self.st_full, it), (self.q_empty[qs], it // nqs)])
            yield ("wait", self.do_full[ds], it // nds)
            yield ("wait", self.dpt_free, it - 1)
            require(self.do_slot[ds] == it, f"dP^T of tile {it} issued before its dO landed")
            require(self.dpt_readers == 0, f"dP^T of tile {it} overwrites the dP^T columns while read")
            self.do_readers[it] += 1

            def dp_done(it=it):
                self.do_readers[it] -= 1
                self.dpt_tile = it
            yield self._product(0, dp_done)
            yield ("commit", 0, [(self.dpt_full, it), (self.do_empty[ds], it // nds)])

    def issuer1(self):
        nqs, nds = self.nqs, self.nds
        yield ("wait", self.kv_full, 0)
        for it in range(self.nq):
            qs, ds = it % nqs, it % nds
            yield ("wait", self.q_full[qs], it // nqs)
            yield ("wait", self.do_full[ds], it // nds)
            self.do_readers[it] += 1
            for h in range(2):
                if not (h == 1 and self.mutation == "dv_half_without_wait"):
                    yield ("wait", self.p_full[h], it)
                require(len(self.pt_written[(it, h)]) == self.W and self.st_tile == it,
                        f"dV (half {h}) of tile {it} issued before every warp wrote that half of P^T")

                def dv_done(it=it, h=h):
                    if h == 1:
                        self.do_readers[it] -= 1
                        self.pt_read_done = True
                yield self._product(1, dv_done)
            yield ("commit", 1, [(self.do_empty[ds], it // nds), (self.p_free, it)])
            yield ("wait", self.ds_full, it)
            require(len(self.ds_written[it]) == self.W, f"dK of tile {it} issued before every warp wrote dS^T")
            self.q_readers[it] += 1
            self.ds_reading = it

            def dk_done(it=it):
                self.q_readers[it] -= 1
                self.ds_reading = -1
            yield self._product(1, dk_done)
            yield ("commit", 1, [(self.q_empty[qs], it // nqs), (self.ds_free, it)])
        yield ("commit", 1, [(self.acc_full, 0)])

    def softmax(self, w):
        for it in range(self.nq):
            yield ("wait", self.st_full, it)
            require(self.st_tile == it and self.x_tile == it, f"warp reads S^T/X of tile {it} before they are in")
            self.st_readers += 1
            self.x_readers[it] += 1
            yield ("do", lambda: None)
            self.st_readers -= 1   # this warp's S^T columns are read: its P^T goes over them
            self.pt_written[(it, 0)].add(w)
            yield ("do", lambda it=it: self.p_full[0].arrive(it))
            yield ("do", lambda: None)
            self.x_readers[it] -= 1
            self.pt_written[(it, 1)].add(w)
            yield ("do", lambda it=it: (self.cx_empty.arrive(it), self.p_full[1].arrive(it)))
            yield ("wait", self.dpt_full, it)
            require(self.dpt_tile == it and self.y_tile == it, f"warp reads dP^T/Y of tile {it} before they are in")
            self.dpt_readers += 1
            yield ("do", lambda: None)
            self.dpt_readers -= 1
            yield ("do", lambda it=it: self.dpt_free.arrive(it))
            self.y_readers[it] += 1
            require(self.ds_reading < 0, f"dS^T tile rewritten (tile {it}) while dK of tile {self.ds_reading} reads it")
            self.ds_written[it].add(w)
            yield ("do", lambda: None)
            self.y_readers[it] -= 1
            yield ("do", lambda it=it: (self.cy_empty.arrive(it), self.ds_full.arrive(it)))
        if self.nq > 0:
            yield ("wait", self.acc_full, 0)
            require(self.outstanding == 0, "dK/dV accumulators read while products are outstanding")

    def roles(self):
        self.pt_read_done = False
        return [self.producer(), self.issuer0(), self.issuer1()] + [self.softmax(w) for w in range(self.W)]


# With an attention mask's tile live map the backward kernels walk only the tiles their tile
# takes and index every slot and phase by that count, so the protocol is this one over the
# count of taken tiles; 0 (a tile with nothing to take) is included.
@pytest.mark.parametrize("nq,nqs,nds", [(0, 2, 2), (1, 2, 2), (2, 2, 2), (5, 2, 2), (6, 3, 2), (7, 2, 3)])
def test_dkdv_protocol_holds_on_random_schedules(nq, nqs, nds):
    for seed in range(80):
        run_roles(DkdvModel(nq, nqs, nds).roles(), random.Random(seed * 100 + nq))
    # one role far behind the others: the producer, either issuer, a softmax warp
    for slow in (0, 1, 2, 3):
        for seed in range(40):
            run_roles(DkdvModel(nq, nqs, nds).roles(), random.Random(seed * 7 + slow), slow={slow})


def test_planted_dkdv_protocol_mistake_is_caught():
    """Issuing Y (and with it the dP^T-complete phase) before dK has read the previous dS^T
    tile lets a warp overwrite that tile under the running dK product."""
    assert _caught(lambda: DkdvModel(5, 2, 2, mutation="y_before_dk"))


def test_planted_dkdv_half_hand_off_mistake_is_caught():
    """Issuing the second half of dV on the first half's arrival reads P^T columns a slow
    warp has not written yet."""
    assert _caught(lambda: DkdvModel(4, 2, 2, mutation="dv_half_without_wait"))


# ---------------------------------------------------------------------------- dQ kernel

class DqModel:
    """One query tile of the dQ kernel over nkt key tiles: a producer (K and V tiles in rings
    of NKS and NVS slots), issuer 0 (S_j = Q K_j^T into score buffer j & 1, dP_j = dO V_j^T),
    issuer 1 (dQ += E_t K_t, E read from tensor memory) and the softmax warps (E_j written
    over the S_j columns they have read)."""

    def __init__(self, nkt, nks, nvs, warps=4, mutation=None):
        self.nkt, self.nks, self.nvs, self.W, self.mutation = nkt, nks, nvs, warps, mutation
        W = warps
        self.qdo_full = Bar("qdo_full", 1)
        self.k_full = [Bar(f"k_full[{i}]", 1) for i in range(nks)]
        self.k_empty = [Bar(f"k_empty[{i}]", 2) for i in range(nks)]   # S_j and dQ_j read K_j
        self.v_full = [Bar(f"v_full[{i}]", 1) for i in range(nvs)]
        self.v_empty = [Bar(f"v_empty[{i}]", 1) for i in range(nvs)]
        self.s_full = [Bar(f"s_full[{b}]", 1) for b in range(2)]
        self.e_free = [Bar(f"e_free[{b}]", 1) for b in range(2)]
        self.dp_full = Bar("dp_full", 1)
        self.dp_free = Bar("dp_free", W)
        # one barrier per score buffer; "single_e_full" plants the earlier form that shared one
        self.e_full = [Bar("e_full", W)] * 2 if mutation == "single_e_full" else [Bar(f"e_full[{b}]", W) for b in range(2)]
        self.dq_full = Bar("dq_full", 1)
        self.k_slot = [-1] * nks
        self.v_slot = [-1] * nvs
        self.k_readers = defaultdict(int)
        self.v_readers = defaultdict(int)
        self.buf = [("empty", -1), ("empty", -1)]   # score buffer b: ("S", j) or ("E", j)
        self.buf_readers = [0, 0]                   # warps reading S, or the dQ product reading E
        self.e_written = defaultdict(set)
        self.dp_tile, self.dp_readers = -1, 0
        self.outstanding = 0

    def producer(self):
        yield ("do", lambda: self.qdo_full.arrive(0, tx=1))
        yield ("copy", self.qdo_full, 0, None)
        for j in range(self.nkt):
            ks, vs = j % self.nks, j % self.nvs
            yield ("wait", self.k_empty[ks], j // self.nks - 1)
            require(not any(v for t, v in self.k_readers.items() if t < j and t % self.nks == ks),
                    f"K slot {ks} refilled (tile {j}) while read")
            yield ("do", lambda ks=ks, j=j: self.k_full[ks].arrive(j // self.nks, tx=1))
            yield ("copy", self.k_full[ks], j // self.nks, lambda ks=ks, j=j: self.k_slot.__setitem__(ks, j))
            yield ("wait", self.v_empty[vs], j // self.nvs - 1)
            require(not any(v for t, v in self.v_readers.items() if t < j and t % self.nvs == vs),
                    f"V slot {vs} refilled (tile {j}) while read")
            yield ("do", lambda vs=vs, j=j: self.v_full[vs].arrive(j // self.nvs, tx=1))
            yield ("copy", self.v_full[vs], j // self.nvs, lambda vs=vs, j=j: self.v_slot.__setitem__(vs, j))

    def _product(self, who, done):
        self.outstanding += 1

        def complete():
            self.outstanding -= 1
            done()
        return ("mma", who, complete)

    def issuer0(self):
        yield ("wait", self.qdo_full, 0)
        for j in range(self.nkt):
            ks, vs, sb = j % self.nks, j % self.nvs, j & 1
            yield ("wait", self.k_full[ks], j // self.nks)
            if self.mutation != "no_e_free_wait":
                yield ("wait", self.e_free[sb], (j >> 1) - 1)
            require(self.k_slot[ks] == j, f"S_{j} issued before K_{j} landed")
            require(self.buf_readers[sb] == 0 and (j < 2 or self.buf[sb] == ("E", j - 2) and self.e_read[j - 2]),
                    f"S_{j} overwrites score buffer {sb} while in use")
            self.k_readers[j] += 1

            def s_done(j=j, sb=sb):
                self.k_readers[j] -= 1
                self.buf[sb] = ("S", j)
            yield self._product(0, s_done)
            yield ("commit", 0, [(self.s_full[sb], j >> 1), (self.k_empty[ks], j // self.nks)])
            yield ("wait", self.v_full[vs], j // self.nvs)
            yield ("wait", self.dp_free, j - 1)
            require(self.v_slot[vs] == j, f"dP_{j} issued before V_{j} landed")
            require(self.dp_readers == 0, f"dP_{j} overwrites the dP columns while read")
            self.v_readers[j] += 1

            def dp_done(j=j):
                self.v_readers[j] -= 1
                self.dp_tile = j
            yield self._product(0, dp_done)
            yield ("commit", 0, [(self.v_empty[vs], j // self.nvs), (self.dp_full, j)])

    def issuer1(self):
        yield ("wait", self.qdo_full, 0)
        for t in range(self.nkt):
            ks, sb = t % self.nks, t & 1
            yield ("wait", self.e_full[sb], t if self.mutation == "single_e_full" else t >> 1)
            yield ("wait", self.k_full[ks], t // self.nks)
            require(len(self.e_written[t]) == self.W and self.buf[sb] == ("E", t), f"dQ_{t} issued before every warp wrote E")
            require(self.k_slot[ks] == t, f"dQ_{t} issued before K_{t} landed")
            self.k_readers[t] += 1
            self.buf_readers[sb] += 1

            def dq_done(t=t, sb=sb):
                self.k_readers[t] -= 1
                self.buf_readers[sb] -= 1
                self.e_read[t] = True
            yield self._product(1, dq_done)
            yield ("commit", 1, [(self.k_empty[ks], t // self.nks), (self.e_free[sb], t >> 1)])
        yield ("commit", 1, [(self.dq_full, 0)])

    def softmax(self, w):
        for j in range(self.nkt):
            sb = j & 1
            yield ("wait", self.s_full[sb], j >> 1)
            require(self.buf[sb] == ("S", j), f"warp reads S_{j} before its product completed")
            self.buf_readers[sb] += 1
            yield ("do", lambda: None)
            self.buf_readers[sb] -= 1
            yield ("wait", self.dp_full, j)
            require(self.dp_tile == j, f"warp reads dP_{j} before its product completed")
            self.dp_readers += 1
            yield ("do", lambda: None)
            self.dp_readers -= 1
            yield ("do", lambda j=j: self.dp_free.arrive(j))
            self.e_written[j].add(w)
            if len(self.e_written[j]) == self.W:
                self.buf[sb] = ("E", j)
            yield ("do", lambda j=j, sb=sb: self.e_full[sb].arrive(j if self.mutation == "single_e_full" else j >> 1))
        yield ("wait", self.dq_full, 0)
        require(self.outstanding == 0, "dQ accumulator read while products are outstanding")

    def roles(self):
        self.e_read = defaultdict(bool)
        return [self.producer(), self.issuer0(), self.issuer1()] + [self.softmax(w) for w in range(self.W)]


@pytest.mark.parametrize("nkt,nks,nvs", [(0, 2, 2), (1, 2, 2), (2, 2, 2), (5, 2, 2), (6, 3, 2), (7, 2, 3)])
def test_dq_protocol_holds_on_random_schedules(nkt, nks, nvs):
    for seed in range(80):
        run_roles(DqModel(nkt, nks, nvs).roles(), random.Random(seed * 100 + nkt))
    for slow in (0, 1, 2, 3):
        for seed in range(40):
            run_roles(DqModel(nkt, nks, nvs).roles(), random.Random(seed * 7 + slow), slow={slow})


@pytest.mark.parametrize("mutation", ["no_e_free_wait", "single_e_full"])
def test_planted_dq_protocol_mistakes_are_caught(mutation):
    """Issuing S_{j+2} without waiting for the dQ product that reads E_j from the same
    buffer overwrites E_j under that product.  One E-complete barrier for both buffers (the
    kernel's earlier form) lets a warp that has finished tile j + 1 arrive while a slower
    warp's arrival for tile j is still missing: the phase of tile j would complete early."""
    # three K stages, as in the kernel: with two, refilling K_{j+2} already waits for dQ_j
    assert _caught(lambda: DqModel(5, 3, 2, mutation=mutation))
