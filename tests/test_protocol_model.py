"""A CPU model of the tensor-core forward kernel's barrier protocol, run on random schedules.

The kernel (attn_fwd_tc.cu) hands work between roles only through mbarriers: a TMA producer
per CTA, one issuing thread per product g (in the even CTA of a CTA pair), and four softmax
warps per query tile.  The model replays each role's waits, arrivals, copies, products and
commits in the kernel's order, with the hardware's rules:
  * a wait on phase k tests the parity of the barrier's phase counter, so it would pass
    wrongly if the barrier were one phase behind and block wrongly if it were two ahead;
  * a phase completes when its expected arrivals have come and its transaction bytes are in
    (copy bytes may land before the arming arrival);
  * copies and products complete asynchronously, a commit arrives once every product its
    thread issued before it has completed, and a commit of a pair lands on both CTAs.
For every random schedule it checks that all roles finish (no deadlock), that every wait
sees exactly the phase it means, that every arrival and copy lands in the phase it is meant
for, and that no buffer is rewritten while a reader still needs it: ring stages (K and V
tiles), score buffers (including the O accumulator's columns used as the second pass-1
buffer), P tiles and O accumulators.  Two planted protocol mistakes must be caught.
"""
import random

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


class Model:
    """One work item: NCTA CTAs (1, or a pair), two products (query tiles, or pairs of them)."""

    NGROUP, WARPS = 2, 4

    def __init__(self, ncta, nst, nkt, nkt_g, dead, rng, mutation=None):
        self.ncta, self.nst, self.nkt, self.nkt_g, self.dead, self.rng = ncta, nst, nkt, nkt_g, dead, rng
        self.mutation = mutation
        n, G, W = ncta, self.NGROUP, self.WARPS
        sw = W if mutation == "single_cta_counts" else n * W
        # barriers that only the even CTA's copy is used of, and per-CTA barriers fed by commits
        self.q_full = Bar("q_full", 1)
        self.ring_full = [Bar(f"ring_full[{i}]", 1) for i in range(nst)]
        self.ring_empty = [[Bar(f"ring_empty[{i}]@{r}", G) for i in range(nst)] for r in range(n)]
        self.s_full = [[[Bar(f"s_full[{g}][{b}]@{r}", 1) for b in range(2)] for g in range(G)] for r in range(n)]
        self.s_empty = [[Bar(f"s_empty[{g}][{b}]", sw) for b in range(2)] for g in range(G)]
        self.p_full = [Bar(f"p_full[{g}]", sw) for g in range(G)]
        self.p_empty = [[Bar(f"p_empty[{g}]@{r}", 1) for g in range(G)] for r in range(n)]
        self.o_full = [[Bar(f"o_full[{g}]@{r}", 1) for g in range(G)] for r in range(n)]
        # buffer state for the hazard checks
        self.stage_use = [[-1] * nst for _ in range(n)]       # use whose copy has landed, per CTA
        self.stage_readers = [dict() for _ in range(nst)]      # use -> products not yet complete
        self.s_written = {}    # (g, b) -> uses whose product completed
        self.s_readers = {}    # (g, b, use) -> warps still reading
        self.p_written = {}    # (g, j) -> warps that wrote P
        self.pv_done = set()   # (g, j) products complete
        self.pv_issued = {g: 0 for g in range(G)}
        self.events = []       # pending asynchronous completions: (ready_check, action, issuer)
        self.issuer_outstanding = {g: 0 for g in range(G)}

    # ------------------------------------------------------------------ roles
    def producer(self, r):
        n, nst = self.ncta, self.nst
        arms = r == 0
        if arms:
            yield ("do", lambda: self.q_full.arrive(0, tx=n))
        yield ("copy", self.q_full, 0, None)
        fills = [("K", j) for j in range(self.nkt)] + [("K", 0)]
        for j in range(1, self.nkt):
            fills += [("K", j), ("V", j - 1)]
        fills.append(("V", self.nkt - 1))
        for it, _ in enumerate(fills):
            st, use = it % nst, it // nst
            yield ("wait", self.ring_empty[r][st], use - 1)
            # every product that read this stage's previous use has completed
            for u, left in self.stage_readers[st].items():
                if u < use and left:
                    raise ProtocolError(f"stage {st} refilled (use {use}) while use {u} still has readers")
            if arms:
                yield ("do", lambda st=st, use=use: self.ring_full[st].arrive(use, tx=n))
            yield ("copy", self.ring_full[st], use, (r, st, use))

    def issuer(self, g):
        n, nst, G = self.ncta, self.nst, self.NGROUP
        nkt, nkt_g = self.nkt, self.nkt_g[g]
        yield ("wait", self.q_full, 0)
        pos = 0
        uses = [0, 0]

        def ring_wait(p):
            st, use = p % nst, p // nst
            yield ("wait", self.ring_full[st], use)
            for r in range(n):
                if self.stage_use[r][st] != use:
                    raise ProtocolError(f"product reads stage {st} use {use} before CTA {r}'s copy landed")

        def release(p):
            st, use = p % nst, p // nst
            yield ("commit", g, [(self.ring_empty[r][st], use) for r in range(n)])

        def mma_s(p, b):
            use = uses[b]
            yield ("wait", self.s_empty[g][b], use - 1)
            if any(self.s_readers.get((g, b, u), 0) for u in range(use)):
                raise ProtocolError(f"S[{g}][{b}] use {use} written while an earlier use is being read")
            if b == 1 and self.pv_issued[g]:
                raise ProtocolError(f"pass-1 S into O[{g}]'s columns after a P V product")
            st, suse = p % nst, p // nst
            self.stage_readers[st][suse] = self.stage_readers[st].get(suse, 0) + 1
            yield ("mma", g, ("S", b, use, st, suse))
            yield ("commit", g, [(self.s_full[r][g][b], use) for r in range(n)])
            uses[b] += 1

        def mma_pv(j, p):
            yield ("wait", self.p_full[g], j)
            if len(self.p_written.get((g, j), ())) != n * self.WARPS:
                raise ProtocolError(f"P V product {j} issued before every warp wrote P[{g}]")
            if any(self.s_readers.get((g, 1, u), 0) for u in range(uses[1])):
                raise ProtocolError(f"P V product into O[{g}] while pass-1 scores in its columns are read")
            if (g, j) not in self.dead:
                st, suse = p % nst, p // nst
                self.stage_readers[st][suse] = self.stage_readers[st].get(suse, 0) + 1
                self.pv_issued[g] += 1
                yield ("mma", g, ("PV", j, st, suse))
            else:
                yield ("mark_pv", g, j)
            yield ("commit", g, [(self.p_empty[r][g], j) for r in range(n)])

        for j in range(nkt):                                   # pass 1
            if self.mutation == "release_without_fill" and j >= nkt_g:
                yield from release(pos)
                pos += 1
                continue
            yield from ring_wait(pos)
            if j < nkt_g:
                yield from mma_s(pos, j & 1)
            yield from release(pos)
            pos += 1
        yield from ring_wait(pos)                              # pass 2: S(0)
        yield from mma_s(pos, 0)
        yield from release(pos)
        pos += 1
        for j in range(nkt):
            if j + 1 < nkt:
                kpos = pos
                pos += 1
                if self.mutation == "release_without_fill" and j + 1 >= nkt_g:
                    yield from release(kpos)
                else:
                    yield from ring_wait(kpos)
                    if j + 1 < nkt_g:
                        yield from mma_s(kpos, 0)
                    yield from release(kpos)
            vpos = pos
            pos += 1
            if self.mutation == "release_without_fill" and j >= nkt_g:
                yield from release(vpos)
                continue
            yield from ring_wait(vpos)
            if j < nkt_g:
                yield from mma_pv(j, vpos)
            yield from release(vpos)
        yield ("commit", g, [(self.o_full[r][g], 0) for r in range(n)])

    def softmax(self, r, g, w):
        nkt_g = self.nkt_g[g]

        def take(b, use):
            yield ("wait", self.s_full[r][g][b], use)
            if use not in self.s_written.get((g, b), ()):
                raise ProtocolError(f"S[{g}][{b}] use {use} read before its product completed")
            key = (g, b, use)
            self.s_readers[key] = self.s_readers.get(key, 0) + 1
            yield ("yield",)
            self.s_readers[key] -= 1
            yield ("do", lambda: self.s_empty[g][b].arrive(use))

        for j in range(nkt_g):                                 # pass 1
            yield from take(j & 1, j >> 1)
        sidx = (nkt_g + 1) >> 1
        for j in range(nkt_g):                                 # pass 2
            yield from take(0, sidx)
            sidx += 1
            yield ("wait", self.p_empty[r][g], j - 1)
            if j > 0 and (g, j - 1) not in self.pv_done:
                raise ProtocolError(f"P[{g}] rewritten (tile {j}) before P V product {j - 1} completed")
            self.p_written.setdefault((g, j), set()).add((r, w))
            yield ("do", lambda j=j: self.p_full[g].arrive(j))
        yield ("wait", self.o_full[r][g], 0)
        if self.pv_issued[g] and self.issuer_outstanding[g]:
            raise ProtocolError(f"O[{g}] read while products are outstanding")

    # ------------------------------------------------------------------ scheduler
    def run(self):
        roles = [self.producer(r) for r in range(self.ncta)]
        roles += [self.issuer(g) for g in range(self.NGROUP)]
        roles += [self.softmax(r, g, w) for r in range(self.ncta) for g in range(self.NGROUP) for w in range(self.WARPS)]
        state = [None] * len(roles)   # the action a role is blocked on
        alive = set(range(len(roles)))
        commits = {g: [] for g in range(self.NGROUP)}   # per issuer, in issue order: ("mma"|"commit", payload)
        copies = []

        def advance(i):
            try:
                state[i] = next(roles[i])
            except StopIteration:
                alive.discard(i)
                state[i] = None

        for i in range(len(roles)):
            advance(i)
        for _ in range(200000):
            if not alive and not copies and not any(commits.values()):
                return
            choices = []
            for i in list(alive):
                a = state[i]
                if a[0] == "wait":
                    if a[1].test(a[2]):
                        choices.append(("role", i))
                else:
                    choices.append(("role", i))
            if copies:
                choices.append(("copy", None))
            for g, q in commits.items():
                if q:
                    choices.append(("tc", g))
            if not choices:
                raise ProtocolError("deadlock: " + ", ".join(
                    f"{state[i][1].name} phase {state[i][2]}" for i in alive if state[i][0] == "wait"))
            kind, i = self.rng.choice(choices)
            if kind == "copy":
                bar, phase, tag = copies.pop(self.rng.randrange(len(copies)))
                bar.complete_tx(phase, 1)
                if tag is not None:
                    r, st, use = tag
                    self.stage_use[r][st] = use
                continue
            if kind == "tc":                  # the oldest tensor-core operation of issuer i completes
                op, payload = commits[i].pop(0)
                if op == "mma":
                    self.issuer_outstanding[i] -= 1
                    if payload[0] == "S":
                        _, b, use, st, suse = payload
                        self.s_written.setdefault((i, b), set()).add(use)
                    else:
                        _, j, st, suse = payload
                        self.pv_done.add((i, j))
                    self.stage_readers[st][suse] -= 1
                elif op == "mark":
                    self.pv_done.add((i, payload))
                else:
                    for bar, phase in payload:
                        bar.arrive(phase)
                continue
            a = state[i]
            if a[0] == "copy":
                copies.append((a[1], a[2], a[3]))
            elif a[0] == "mma":
                self.issuer_outstanding[a[1]] += 1
                commits[a[1]].append(("mma", a[2]))
            elif a[0] == "mark_pv":
                commits[a[1]].append(("mark", a[2]))
            elif a[0] == "commit":
                commits[a[1]].append(("commit", a[2]))
            elif a[0] == "do":
                a[1]()
            advance(i)
        raise ProtocolError("schedule did not finish")


CONFIGS = [
    # (CTAs, ring stages, key tiles, key tiles of product 0, dead fraction)
    (1, 3, 1, 1, 0.0), (1, 3, 4, 4, 0.0), (1, 3, 5, 4, 0.3), (1, 6, 3, 3, 0.5), (1, 6, 7, 6, 0.0),
    (2, 6, 1, 1, 0.0), (2, 6, 4, 4, 0.0), (2, 6, 5, 3, 0.3), (2, 6, 9, 7, 0.2), (2, 6, 2, 1, 0.0),
]


@pytest.mark.parametrize("ncta,nst,nkt,nkt0,dead_frac", CONFIGS)
def test_forward_protocol_holds_on_random_schedules(ncta, nst, nkt, nkt0, dead_frac):
    for seed in range(60):
        rng = random.Random(seed * 1000 + nkt * 10 + ncta)
        dead = {(g, j) for g in range(2) for j in range(nkt) if rng.random() < dead_frac}
        Model(ncta, nst, nkt, (nkt0, nkt), dead, rng).run()


@pytest.mark.parametrize("mutation,ncta,nkt,nkt0", [("release_without_fill", 1, 6, 3),
                                                    ("release_without_fill", 2, 6, 2),
                                                    ("single_cta_counts", 2, 3, 3)])
def test_planted_protocol_mistakes_are_caught(mutation, ncta, nkt, nkt0):
    """Releasing ring stages without waiting for their fill lets the issuer that skips tiles
    run a phase ahead; counting one CTA's warps on the pair's barriers completes a phase
    early.  Some schedule must expose each."""
    caught = False
    for seed in range(200):
        try:
            Model(ncta, 6 if ncta == 2 else 3, nkt, (nkt0, nkt), set(), random.Random(seed), mutation).run()
        except ProtocolError:
            caught = True
            break
    assert caught
