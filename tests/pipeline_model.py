"""Executable model of the synchronisation protocols of the forward kernel with two Q tiles per
CTA and a dedicated S-issuer warp (`run`): at d = 64 three rotating S buffers in tensor memory that
P aliases (mode "s3"), at d = 128 (bf16 and e4m3) one S buffer both tiles share with P in a
tensor-memory area per tile (mode "s1").

This is test infrastructure: a model of the kernel's warp roles and mbarriers, not the kernel. It
runs the roles as Python generators under random interleavings and checks three things:

* every parity wait sees its barrier at the intended phase or one past it, since a parity wait
  cannot tell phases two apart (hardware semantics: the wait returns once the phase with the
  awaited parity has completed);
* no tensor-memory S buffer is overwritten before the softmax has read it and the PV has read the
  P written over it, and no PV reads a buffer that holds anything but its own P;
* the O accumulator is touched by a rescale only after the tile's previous PV has completed, and
  read by the epilogue only after all of the tile's PVs.

Roles, as in the kernel:
  producer   loads Q once per work tile, then K_j, V_j through a ring of NS stages;
  S issuer   issues S products in the order S0_0, S1_0, S0_1, S1_1, ..., skipping those a Q tile
             does not need. S number k goes to buffer k % 3 once the PV of number k - 3 has
             completed (s_free). It releases each K stage and, after the last S, Q;
  PV issuer  one per Q tile: waits for the two P halves of its tile's S_j, issues PV_j, and commits
             s_free (the buffer), o_done (for rescales), and o_full after the tile's last PV. At
             a step where its tile has no S (past a ragged end, or the shorter causal tile's last
             step) it still waits for the V stage before releasing it;
  softmax    one per Q tile: waits for S_j, maybe rescales O (after waiting for PV_{j-1}), writes
             P_j over S_j, and at the end of the work tile waits for o_full.

Mode "s1" (d = 128): S number k always goes to the one shared buffer, once the softmax that owns S
number k - 1 has loaded it (s_free, arrived by the softmax, not by a PV). The softmax writes P_j
to its tile's own P area after waiting for PV_{j-1}, which read the P before it.

Both modes need an even number of K/V stages (`ns`): then each stage holds only K tiles (waited
for by the S issuer) or only V tiles (waited for by the PV issuers), and every waiter has waited
for the stage's previous load itself. With an odd count a PV issuer whose tile has no keys in a
work tile, paced by nothing, can reach a V stage whose previous load (a K tile it never waits for)
has not landed, and its parity wait then passes two phases early.
  tensor pipe executes MMAs and commits in issue order: one shared in-order queue, or (a weaker
             model) one queue per issuing warp;
  TMA        lands the producer's K/V copies in any order.

Each Q tile has M S-ready, P-ready and PV-done barriers, its g-th S product using index g % M and
phase g // M. The kernel uses M = 3 at d = 64 and M = 1 in mode "s1".
"""
import random

NS = 8   # K/V ring stages of the d = 64 instance (the d = 128 instance has 5)


class ProtocolError(Exception):
    pass


class Bar:
    """An mbarrier: `expected` arrivals complete a phase."""

    def __init__(self, name, expected, pre=0):
        self.name, self.expected, self.done, self.arr = name, expected, 0, 0
        for _ in range(pre):
            self.arrive()

    def arrive(self):
        self.arr += 1
        if self.arr == self.expected:
            self.done += 1
            self.arr = 0


def wait(bar, parity, intended):
    """Poll until the phase with this parity has completed, checking the phase window."""
    while True:
        if bar.done not in (intended, intended + 1):
            raise ProtocolError(f"phase window broken on {bar.name}: done={bar.done} awaited={intended}")
        if (bar.done & 1) != parity:
            return
        yield


def s_number(sbase, qt, j, n0, n1):
    """Position of Q tile qt's S_j among the CTA's S products (n0, n1: KV tiles of the two tiles)."""
    return sbase + min(j, n0) + min(j, n1) + (1 if (qt == 1 and j < n0) else 0)


def run(tiles, seed, shared_pipe=True, rescale_p=0.3, M=3, skip_s_free=False, skip_rescale_wait=False,
        mode="s3", ns=NS):
    """Runs the work tiles [(n0, n1), ...] of one CTA to completion under a random schedule."""
    rnd = random.Random(seed)
    s1 = mode == "s1"
    if s1:
        M = 1
    NS = ns
    q_full, q_empty = Bar("q_full", 1), Bar("q_empty", 2)
    kv_full = [Bar(f"kv_full{i}", 1) for i in range(NS)]
    kv_empty = [Bar(f"kv_empty{i}", 2) for i in range(NS)]
    s_full = [Bar(f"s_full{i}", 1) for i in range(2 * M)]
    p_half = [[Bar(f"p_half{i}.{h}", 1) for h in range(2)] for i in range(2 * M)]
    o_done = [Bar(f"o_done{i}", 1) for i in range(2 * M)]
    s_free = [Bar(f"s_free{i}", 1) for i in range(3)]
    nsb = 1 if s1 else 3          # S buffers
    inflight = []                 # K/V copies issued but not landed: TMA completes them in any order
    s_loaded = set()              # s1: S numbers the softmax has loaded
    p_area = [None, None]         # s1: the P each tile's tensor-memory P area holds
    o_full = [Bar(f"o_full{i}", 1) for i in range(2)]
    tmem = [None, None, None]                 # ("S", k) or ("P", k)
    pv_done = set()                           # S numbers whose PV has completed
    pv_complete = {0: set(), 1: set()}        # (work tile, j) per Q tile
    queues = {0: [], 1: [], 2: []}            # per issuing warp (2: the S issuer)
    shared = []

    def enqueue(iss, op):
        (shared if shared_pipe else queues[iss]).append((iss, op))

    def commit(iss, bar):
        enqueue(iss, ("commit", bar))

    def producer():
        ring, nq = 0, 0
        for (n0, n1) in tiles:
            nmax = max(n0, n1)
            if nmax == 0:
                continue
            if nq > 0:
                yield from wait(q_empty, (nq - 1) & 1, nq - 1)
            nq += 1
            yield
            q_full.arrive()
            for _ in range(2 * nmax):
                slot = ring % NS
                if ring >= NS:
                    yield from wait(kv_empty[slot], (ring // NS - 1) & 1, ring // NS - 1)
                yield
                inflight.append(slot)
                ring += 1

    def s_issuer():
        ring, nq, sbase, g = 0, 0, 0, [0, 0]
        for (n0, n1) in tiles:
            nmax = max(n0, n1)
            if nmax == 0:
                continue
            sb, gb = sbase, list(g)
            sbase += n0 + n1
            g[0] += n0
            g[1] += n1
            yield from wait(q_full, nq & 1, nq)
            nq += 1
            base = ring
            for j in range(nmax):
                pos_k = base + 2 * j
                yield from wait(kv_full[pos_k % NS], (pos_k // NS) & 1, pos_k // NS)
                for qt in range(2):
                    if j < (n1 if qt else n0):
                        k = s_number(sb, qt, j, n0, n1)
                        if k >= nsb and not skip_s_free:
                            yield from wait(s_free[k % nsb], (k // nsb - 1) & 1, k // nsb - 1)
                        enqueue(2, ("S", k, k % nsb))
                        commit(2, s_full[M * qt + (gb[qt] + j) % M])
                commit(2, kv_empty[pos_k % NS])
                commit(2, kv_empty[pos_k % NS])
                if j + 1 == nmax:
                    commit(2, q_empty)
                    commit(2, q_empty)
                yield
            ring = base + 2 * nmax

    def pv_issuer(myq):
        ring, sbase, g = 0, 0, 0
        for ti, (n0, n1) in enumerate(tiles):
            n, nmax = (n1 if myq else n0), max(n0, n1)
            if nmax == 0:
                continue
            sb, gb = sbase, g
            sbase += n0 + n1
            g += n
            base = ring
            for j in range(nmax):
                pos_v = base + 2 * j + 1
                yield from wait(kv_full[pos_v % NS], (pos_v // NS) & 1, pos_v // NS)
                if j < n:
                    gj = gb + j
                    k = s_number(sb, myq, j, n0, n1)
                    for h in range(2):
                        yield from wait(p_half[M * myq + gj % M][h], (gj // M) & 1, gj // M)
                    enqueue(myq, ("PV", k, k % 3, myq, ti, j))
                    if not s1:
                        commit(myq, s_free[k % 3])
                    commit(myq, o_done[M * myq + gj % M])
                    if j + 1 == n:
                        commit(myq, o_full[myq])
                    commit(myq, kv_empty[pos_v % NS])
                else:
                    kv_empty[pos_v % NS].arrive()
                yield
            ring = base + 2 * nmax

    def softmax(qt):
        sbase, g, tiles_done = 0, 0, 0
        for ti, (n0, n1) in enumerate(tiles):
            n = n1 if qt else n0
            sb, gb = sbase, g
            sbase += n0 + n1
            g += n
            if n == 0:
                continue
            for j in range(n):
                gj = gb + j
                k = s_number(sb, qt, j, n0, n1)
                yield from wait(s_full[M * qt + gj % M], (gj // M) & 1, gj // M)
                if tmem[k % nsb] != ("S", k):
                    raise ProtocolError(f"softmax {qt} expected S{k} in buffer {k % nsb}, found {tmem[k % nsb]}")
                yield
                if s1:
                    # S is in registers: the shared buffer may take the next S. P_j then waits for
                    # PV_{j-1}, which read this tile's P area (and that wait also covers rescales).
                    s_loaded.add(k)
                    s_free[0].arrive()
                    yield
                    if j > 0:
                        if not skip_rescale_wait:
                            gp = gj - 1
                            yield from wait(o_done[qt], gp & 1, gp)
                        if (ti, j - 1) not in pv_complete[qt]:
                            raise ProtocolError(f"P{k} written before the PV before it read P or O settled")
                    p_area[qt] = ("P", k)
                else:
                    if j > 0 and rnd.random() < rescale_p:
                        if not skip_rescale_wait:
                            gp = gj - 1
                            yield from wait(o_done[M * qt + gp % M], (gp // M) & 1, gp // M)
                        if (ti, j - 1) not in pv_complete[qt]:
                            raise ProtocolError("O rescaled while PV_{j-1} may still accumulate into it")
                    if tmem[k % 3] != ("S", k):
                        raise ProtocolError(f"S{k} overwritten before its P was written")
                    tmem[k % 3] = ("P", k)
                p_half[M * qt + gj % M][0].arrive()
                yield
                p_half[M * qt + gj % M][1].arrive()
            yield from wait(o_full[qt], tiles_done & 1, tiles_done)
            if any((ti, j) not in pv_complete[qt] for j in range(n)):
                raise ProtocolError("epilogue read O before the tile's last PV completed")
            tiles_done += 1

    def execute(op):
        if op[0] == "S":
            _, k, b = op
            prev = tmem[b]
            if s1:
                if prev is not None and (prev != ("S", k - 1) or (k - 1) not in s_loaded):
                    raise ProtocolError(f"S{k} overwrites buffer {b} holding {prev} before the softmax loaded it")
            elif prev is not None and (prev != ("P", k - 3) or (k - 3) not in pv_done):
                raise ProtocolError(f"S{k} overwrites buffer {b} holding {prev}")
            tmem[b] = ("S", k)
        elif op[0] == "PV":
            _, k, b, qt, ti, j = op
            held = p_area[qt] if s1 else tmem[b]
            if held != ("P", k):
                raise ProtocolError(f"PV{k} reads P holding {held}")
            pv_done.add(k)
            pv_complete[qt].add((ti, j))
        else:
            op[1].arrive()

    def pipe(q):
        while True:
            if q:
                execute(q.pop(0)[1])
            yield

    def tma():
        while True:
            if inflight:
                kv_full[inflight.pop(rnd.randrange(len(inflight)))].arrive()
            yield

    procs = {"producer": producer(), "s_issuer": s_issuer(), "pv0": pv_issuer(0), "pv1": pv_issuer(1),
             "softmax0": softmax(0), "softmax1": softmax(1)}
    finite = set(procs)
    procs["tma"] = tma()
    if shared_pipe:
        procs["pipe"] = pipe(shared)
    else:
        for i in range(3):
            procs[f"pipe{i}"] = pipe(queues[i])
    steps = 0
    while finite:
        name = rnd.choice(list(procs))
        try:
            next(procs[name])
        except StopIteration:
            del procs[name]
            finite.discard(name)
        steps += 1
        if steps > 1_000_000:
            raise ProtocolError("no progress: " + ", ".join(sorted(finite)))


def random_tiles(rnd, kind):
    """Work tiles (n0, n1) of one CTA: equal counts (non-causal), one more KV tile for the second
    Q tile (causal), or any pair including empty Q tiles (ragged batches)."""
    out = []
    for _ in range(rnd.randint(1, 10)):
        if kind == "noncausal":
            n = rnd.randint(1, 9)
            out.append((n, n))
        elif kind == "causal":
            n0 = rnd.randint(1, 8)
            out.append((n0, n0 + 1))
        else:
            out.append((rnd.randint(0, 6), rnd.randint(0, 6)))
    return out


def random_tiles_causal_ragged(rnd):
    """Causal ragged batches as the varlen plan yields them: one more KV tile for the second Q
    tile, or none at all where the second tile lies past the sequence's end."""
    out = []
    for _ in range(rnd.randint(1, 10)):
        n0 = rnd.randint(1, 8)
        out.append((n0, 0 if rnd.random() < 0.5 else n0 + 1))
    return out


SCHEDULES = ((True, 0.3), (False, 0.3), (True, 1.0), (False, 1.0))


def sweep(n_cases, case_seed, **kw):
    """Runs n_cases random tile lists under every schedule; returns the first failure or None."""
    rnd = random.Random(case_seed)
    for i in range(n_cases):
        kind = ("noncausal", "causal", "ragged", "causal-ragged")[i % 4]
        tiles = random_tiles_causal_ragged(rnd) if kind == "causal-ragged" else random_tiles(rnd, kind)
        for shared, rp in SCHEDULES:
            try:
                run(tiles, seed=i * 7 + shared + int(rp * 10), shared_pipe=shared, rescale_p=rp, **kw)
            except ProtocolError as e:
                return f"{kind} {tiles}: {e}"
    return None
