"""A randomized model of the tensor-core kernels' mbarrier protocols (test
infrastructure; it models the protocols, it shares no code with the kernels).

Each warp role is a generator that yields the operations it performs on
mbarriers: wait for a phase (by parity, as mbarrier.try_wait.parity does),
arrive with a tag naming the block it signals, or issue work to the tensor
core.  The tensor core is a FIFO: issued MMAs and commits retire in order at
random times, and a commit arrives on its barrier when it retires (as
tcgen05.commit does).  A scheduler runs the roles in a random interleaving
with random per-role speeds (so one warp can fall far behind the others).

Checked per run: every completed phase of a tagged barrier collected arrivals
that all carry the same tag (a fast warp's arrival for the next block must not
complete the phase of this one), and the run ends with every role finished
(no deadlock).  Where a protocol names the tensor-memory buffers its MMAs and
warps use, the model also tracks which block each buffer holds: an MMA writes
its result when it retires and checks the operands it reads then, a warp checks
the buffer it reads (or sets the one it writes) at that step, so a buffer
overwritten before every reader is done, or read before it is written, is
reported.
"""
from __future__ import annotations

import random


class Barrier:
    """Arrival count and transaction bytes (expect-tx / complete-tx, as TMA
    loads use them): a phase completes when every arrival is in and the
    outstanding byte count is back to zero."""

    def __init__(self, name, count, tagged=True):
        self.name, self.count, self.tagged = name, count, tagged
        self.phase = 0
        self.pending = count
        self.tx = 0
        self.tags = []

    def _maybe_complete(self, violations):
        if self.pending == 0 and self.tx == 0:
            if self.tagged and len(set(self.tags)) > 1:
                violations.append(f"{self.name} phase {self.phase} completed with arrivals for {sorted(set(self.tags))}")
            self.phase += 1
            self.pending = self.count
            self.tags = []

    def arrive(self, tag, violations, expect_tx=0):
        self.tags.append(tag)
        self.tx += expect_tx
        self.pending -= 1
        self._maybe_complete(violations)

    def complete_tx(self, nbytes, violations):
        self.tx -= nbytes
        self._maybe_complete(violations)

    def done(self, parity):
        """try_wait.parity(parity): the phase with that parity has completed."""
        return (self.phase & 1) != parity


class TensorCore:
    """In-order queue of ("mma", reads, writes) and ("commit", barrier, tag)
    items; `mem` maps a tensor-memory buffer to the block it holds."""

    def __init__(self):
        self.queue = []
        self.mem = {}

    def check(self, who, buf, tag, violations):
        if self.mem.get(buf) != tag:
            violations.append(f"{who} read {buf} holding {self.mem.get(buf)}, expected {tag}")

    def retire_one(self, violations):
        kind, x, y = self.queue.pop(0)
        if kind == "commit":
            x.arrive(y, violations)
            return
        for buf, tag in x or ():
            self.check("mma", buf, tag, violations)
        for buf, tag in y or ():
            self.mem[buf] = tag


def run(roles, tc, rng, max_steps=200000):
    """Interleave the role generators randomly.  Each role yields
    ("wait", bar, parity), ("arrive", bar, tag), ("arrive_tx", bar, tag, loads)
    (arrive with expect-tx for `loads` one-unit TMA loads, which then land in
    any order), ("mma",) or ("mma", reads, writes) (lists of (buffer, tag)),
    ("commit", bar, tag), ("read", buffer, tag), ("write", buffer, tag),
    ("poll", bar, parity) (mbarrier.test_wait: never blocks; the generator
    receives whether the phase has completed) or ("work",) (local computation,
    no synchronisation).  Returns (violations, deadlocked)."""
    violations = []
    tma = []  # barriers with one load in flight each
    speed = {name: rng.choice([0.05, 0.3, 1.0, 1.0, 1.0]) for name in roles}
    pending = {}
    for name, gen in roles.items():
        pending[name] = next(gen, None)
    for _ in range(max_steps):
        ready = [n for n, op in pending.items()
                 if op is not None and not (op[0] == "wait" and not op[1].done(op[2]))]
        choices = ready + (["__tc__"] if tc.queue else []) + (["__tma__"] if tma else [])
        if not choices:
            stuck = [n for n, op in pending.items() if op is not None]
            return violations, bool(stuck)
        weights = [speed.get(c, 1.0) for c in choices]
        who = rng.choices(choices, weights)[0]
        if who == "__tc__":
            tc.retire_one(violations)
            continue
        if who == "__tma__":
            tma.pop(rng.randrange(len(tma))).complete_tx(1, violations)
            continue
        op = pending[who]
        if op[0] == "arrive":
            op[1].arrive(op[2], violations)
        elif op[0] == "arrive_tx":
            op[1].arrive(op[2], violations, expect_tx=op[3])
            tma.extend([op[1]] * op[3])
        elif op[0] == "mma":
            tc.queue.append(("mma", op[1], op[2]) if len(op) > 1 else ("mma", None, None))
        elif op[0] == "read":
            tc.check(who, op[1], op[2], violations)
        elif op[0] == "write":
            tc.mem[op[1]] = op[2]
        elif op[0] == "commit":
            tc.queue.append(("commit", op[1], op[2]))
        elif op[0] == "poll":
            try:
                pending[who] = roles[who].send(op[1].done(op[2]))
            except StopIteration:
                pending[who] = None
            continue
        pending[who] = next(roles[who], None)
    return violations + ["step limit"], True


# ---- the kernels' protocols ---------------------------------------------------------
# Only the synchronisation is modelled; "work" stands for computation and
# tensor-memory loads / stores.  Tags: the global block (or item) index the
# arrival belongs to.

def _dq_issue_s(g, bars):
    yield ("mma", [], [("S", g)])
    yield ("commit", bars["s_full"], g)


def _dq_issue_dp(g, bars, vstages):
    yield ("mma", [], [("dP", g)])
    yield ("commit", bars["dp_full"], g)
    if bars["v_empty"] is not None:
        yield ("commit", bars["v_empty"][g % vstages], g)


def _dq_issuer_item(it, g0, nk, st, bars, kstages, vstages, ds_buffers=2, test_s_free=True):
    """The dq issuer's work item: S_0 and dP_0, then per key block j (global
    index g) three steps, each behind its barriers: S_{j+1} once every warp has
    read S_j (and block j + 1's K / V landed), dP_{j+1} once dP_j has been read,
    dQ_j once dS_j is in TMEM (and, at j = 0, the previous item's dQ was read
    out).  The kernel's issuing lane tests these barriers with short polls and
    the warp falls back to a bounded wait; either way a step starts only once
    its barriers are complete, which is what is modelled.
    ds_buffers, test_s_free: planted mistakes for the model's own tests."""
    k_full = bars["k_full"]
    if k_full is not None:
        yield ("wait", k_full[g0 % kstages], (g0 // kstages) & 1)
    yield from _dq_issue_s(g0, bars)
    yield from _dq_issue_dp(g0, bars, vstages)
    ds = bars["ds"]
    for j in range(nk):
        g, more = g0 + j, j + 1 < nk
        if test_s_free:
            yield ("wait", bars["s_free"], g & 1)
        if more:
            if k_full is not None:
                yield ("wait", k_full[(g + 1) % kstages], ((g + 1) // kstages) & 1)
            yield from _dq_issue_s(g + 1, bars)
        yield ("wait", bars["dp_free"], g & 1)
        if more:
            yield from _dq_issue_dp(g + 1, bars, vstages)
        if len(ds) == 2:
            yield ("wait", ds[g & 1], (g >> 1) & 1)
        else:
            yield ("wait", ds[0], st["ds"] & 1)
        st["ds"] += 1
        if j == 0:
            yield ("wait", bars["acc_free"], (st["af"] & 1) ^ 1)
            st["af"] += 1
        yield ("mma", [(("dS", j % ds_buffers), g)], [])  # dQ += dS_j K_j
        if bars["k_empty"] is not None:
            yield ("commit", bars["k_empty"][g % kstages], g)
    yield ("commit", bars["acc_done"], it)


def _dq_warp(items, rng, bars, ds_buffers=2):
    c = {"s": 0, "dp": 0, "ad": 0}
    ds = bars["ds"]
    step = 0
    for it, nk in enumerate(items):
        for j in range(nk):
            yield ("wait", bars["s_full"], c["s"] & 1)
            c["s"] += 1
            yield ("read", "S", step)
            yield ("arrive", bars["s_free"], step)
            yield ("work",)  # the exponentials
            yield ("wait", bars["dp_full"], c["dp"] & 1)
            c["dp"] += 1
            yield ("read", "dP", step)
            yield ("arrive", bars["dp_free"], step)
            for _ in range(rng.randint(1, 6)):
                yield ("work",)
            yield ("write", ("dS", j % ds_buffers), step)
            yield ("arrive", ds[step & 1] if len(ds) == 2 else ds[0], step)
            step += 1
        yield ("wait", bars["acc_done"], c["ad"] & 1)
        c["ad"] += 1
        yield ("work",)
        yield ("arrive", bars["acc_free"], it)


def _dq_bars(n_warps, split_ds=True):
    return {
        "s_full": Barrier("s_full", 1), "s_free": Barrier("s_free", n_warps),
        "dp_full": Barrier("dp_full", 1), "dp_free": Barrier("dp_free", n_warps),
        "ds": [Barrier("ds_ready[0]", n_warps), Barrier("ds_ready[1]", n_warps)] if split_ds
        else [Barrier("ds_ready", n_warps)],
        "acc_done": Barrier("acc_done", 1), "acc_free": Barrier("acc_free", n_warps),
        "k_full": None, "k_empty": None, "v_empty": None,
    }


def dq_protocol(items, rng, n_warps=8, split_ds=True, ds_buffers=2, test_s_free=True):
    """dq kernel: per key block S and dP into TMEM, each committed on its own
    barrier (s_full, dp_full); the elementwise warps read S (s_free), then dP
    (dp_free), form dS into one of two TMEM buffers (ds_ready); the issuer's
    order is S_{j+1}, dP_{j+1}, dQ_j (see _dq_issuer_item).  split_ds False
    models the earlier single dS-ready barrier, whose lapping race the model
    must find; ds_buffers=1 and test_s_free=False (S_{j+1} issued without
    waiting for every warp's read of S_j) plant mistakes the TMEM checks must
    catch."""
    tc = TensorCore()
    bars = _dq_bars(n_warps, split_ds)
    st = {"ds": 0, "af": 0}

    def issuer():
        g = 0
        for it, nk in enumerate(items):
            yield from _dq_issuer_item(it, g, nk, st, bars, 1, 1, ds_buffers, test_s_free)
            g += nk

    roles = {"issuer": issuer()}
    roles.update({f"warp{w}": _dq_warp(items, rng, bars, ds_buffers) for w in range(n_warps)})
    return roles, tc


def fwd_protocol(items, rng, warps_per_tile=4):
    """Forward kernel: two query tiles ping-pong; per key tile the issuer waits
    for P_j(t) (p_full, one arrival per softmax warp), issues PV_j(t) and
    S_{j+1}(t) (commit s_full); after the last PV it commits o_done, and before
    the next item's first PV it waits for the epilogue's o_free."""
    tc = TensorCore()
    s_full = [Barrier(f"s_full[{t}]", 1) for t in (0, 1)]
    p_full = [Barrier(f"p_full[{t}]", warps_per_tile) for t in (0, 1)]
    o_done = [Barrier(f"o_done[{t}]", 1) for t in (0, 1)]
    o_free = [Barrier(f"o_free[{t}]", warps_per_tile) for t in (0, 1)]

    def issuer():
        pc = [0, 0]
        of = [0, 0]
        blk = 0
        for it, n in enumerate(items):
            for t in (0, 1):
                yield ("mma",)
                yield ("commit", s_full[t], blk)
            for j in range(n):
                for t in (0, 1):
                    yield ("wait", p_full[t], pc[t] & 1)
                    pc[t] += 1
                    if j == 0:
                        yield ("wait", o_free[t], (of[t] & 1) ^ 1)
                        of[t] += 1
                    yield ("mma",)  # PV_j(t)
                    if j == n - 1:
                        yield ("commit", o_done[t], it)
                    else:
                        yield ("mma",)  # S_{j+1}(t)
                        yield ("commit", s_full[t], blk + j + 1)
            blk += n

    def softmax(t):
        sc = oc = 0
        blk = 0
        for it, n in enumerate(items):
            for j in range(n):
                yield ("wait", s_full[t], sc & 1)
                sc += 1
                for _ in range(rng.randint(1, 6)):
                    yield ("work",)
                yield ("arrive", p_full[t], blk + j)
            blk += n
            yield ("wait", o_done[t], oc & 1)
            oc += 1
            yield ("work",)
            yield ("arrive", o_free[t], it)

    roles = {"issuer": issuer()}
    for t in (0, 1):
        roles.update({f"sm{t}.{w}": softmax(t) for w in range(warps_per_tile)})
    return roles, tc


def _dkdv_regions(n_warps, what, blk):
    """Each elementwise warp's part of the S^T (or dP^T) TMEM columns, holding
    `what` of block blk."""
    region = "S" if what in ("S", "P") else "D"
    return [((region, w), (what, blk)) for w in range(n_warps)]


def _dkdv_issuer_item(it, n, nq, st, bars, n_warps, stages=None, s_before_dv=False):
    """The dK/dV issuer's work item (query blocks n .. n + nq - 1 in ring
    order): S^T_0, dP^T_0, then per block qb the steps dV_qb (after P^T_qb is
    in TMEM), S^T_{qb+1} (after its Q / dO tiles landed), dK_qb and dP^T_{qb+1}
    (after dS^T_qb is in TMEM).  S^T_{qb+1} overwrites the P^T that dV_qb reads
    and dP^T_{qb+1} the dS^T that dK_qb reads, so they follow those MMAs on the
    in-order tensor pipe.  s_before_dv plants the mistake of issuing S^T_{qb+1}
    ahead of dV_qb (once P^T_qb is complete)."""
    q_full = bars["q_full"]
    if q_full is not None:
        yield ("wait", q_full[n % stages], (n // stages) & 1)
    yield ("mma", [], _dkdv_regions(n_warps, "S", n))
    yield ("commit", bars["st_full"], n)
    yield ("mma", [], _dkdv_regions(n_warps, "dP", n))
    yield ("commit", bars["dp_full"], n)
    for qb in range(nq):
        cur, nxt = n + qb, qb + 1 < nq

        def next_s():
            if q_full is not None:
                yield ("wait", q_full[(cur + 1) % stages], ((cur + 1) // stages) & 1)
            yield ("mma", [], _dkdv_regions(n_warps, "S", cur + 1))
            yield ("commit", bars["st_full"], cur + 1)

        yield ("wait", bars["p_ready"], st["pr"] & 1)
        st["pr"] += 1
        if qb == 0:
            yield ("wait", bars["acc_free"], (st["af"] & 1) ^ 1)
            st["af"] += 1
        if s_before_dv and nxt:
            yield from next_s()
        yield ("mma", _dkdv_regions(n_warps, "P", cur), [])  # dV += P^T dO
        if bars["do_empty"] is not None:
            yield ("commit", bars["do_empty"][cur % stages], cur)
        if nxt and not s_before_dv:
            yield from next_s()
        yield ("wait", bars["ds_ready"], st["dsr"] & 1)
        st["dsr"] += 1
        yield ("mma", _dkdv_regions(n_warps, "dS", cur), [])  # dK += dS^T Q
        if bars["q_empty"] is not None:
            yield ("commit", bars["q_empty"][cur % stages], cur)
        if nxt:
            yield ("mma", [], _dkdv_regions(n_warps, "dP", cur + 1))
            yield ("commit", bars["dp_full"], cur + 1)
    yield ("commit", bars["acc_done"], it)


def _dkdv_elementwise(items, rng, w, bars, stats):
    st = dp = ad = si = 0
    blk = 0
    for it, nq in enumerate(items):
        for qb in range(nq):
            yield ("arrive", stats[si & 1], si)
            yield ("wait", stats[si & 1], (si >> 1) & 1)
            si += 1
            yield ("wait", bars["st_full"], st & 1)
            st += 1
            yield ("read", ("S", w), ("S", blk + qb))
            for _ in range(rng.randint(1, 6)):
                yield ("work",)
            yield ("write", ("S", w), ("P", blk + qb))  # P^T over S^T
            yield ("arrive", bars["p_ready"], blk + qb)
            yield ("wait", bars["dp_full"], dp & 1)
            dp += 1
            yield ("read", ("D", w), ("dP", blk + qb))
            for _ in range(rng.randint(1, 3)):
                yield ("work",)
            yield ("write", ("D", w), ("dS", blk + qb))  # dS^T over dP^T
            yield ("arrive", bars["ds_ready"], blk + qb)
        blk += nq
        yield ("wait", bars["acc_done"], ad & 1)
        ad += 1
        yield ("work",)
        yield ("arrive", bars["acc_free"], it)


def _dkdv_bars(n_warps):
    return {
        "st_full": Barrier("st_full", 1), "dp_full": Barrier("dp_full", 1),
        "p_ready": Barrier("p_ready", n_warps), "ds_ready": Barrier("ds_ready", n_warps),
        "acc_done": Barrier("acc_done", 1), "acc_free": Barrier("acc_free", n_warps),
        "q_full": None, "q_empty": None, "do_empty": None,
    }


def dkdv_protocol(items, rng, n_warps=8, s_before_dv=False):
    """dK/dV kernel: issue order dV_i, S^T_{i+1}, dK_i, dP^T_{i+1}; the
    elementwise warps stage each query block's statistics (double-buffered
    stats_ready), write P^T over S^T (p_ready) and dS^T over dP^T (ds_ready)."""
    tc = TensorCore()
    bars = _dkdv_bars(n_warps)
    stats = [Barrier("stats_ready[0]", n_warps), Barrier("stats_ready[1]", n_warps)]
    st = {"pr": 0, "dsr": 0, "af": 0}

    def issuer():
        blk = 0
        for it, nq in enumerate(items):
            yield from _dkdv_issuer_item(it, blk, nq, st, bars, n_warps, s_before_dv=s_before_dv)
            blk += nq

    roles = {"issuer": issuer()}
    roles.update({f"warp{w}": _dkdv_elementwise(items, rng, w, bars, stats) for w in range(n_warps)})
    return roles, tc


def explore(protocol, trials, seed, **kw):
    """Run `trials` random interleavings of random items; returns the first
    violation or deadlock found (or None)."""
    rng = random.Random(seed)
    for trial in range(trials):
        items = [rng.choice([1, 1, 2, 3, 5]) for _ in range(rng.randint(1, 4))]
        roles, tc = protocol(items, rng, **kw)
        violations, deadlocked = run(roles, tc, rng)
        if violations or deadlocked:
            return {"trial": trial, "items": items, "violations": violations, "deadlock": deadlocked}
    return None


# ---- protocols with their TMA producers -------------------------------------------

def dkdv_loads_protocol(items, rng, n_warps=8, stages=2, q_full_arrivals=2):
    """The dK/dV kernel with its producers: warp 0 loads K, V (kv_full) and
    the Q ring, warp 2 the dO ring, and a block's Q and dO land on one full
    barrier (q_full, one arrival with expect-tx from each producer).
    q_full_arrivals = 1 models forgetting the second producer's arrival."""
    tc = TensorCore()
    kv_full, kv_empty = Barrier("kv_full", 1), Barrier("kv_empty", 1)
    bars = _dkdv_bars(n_warps)
    bars["q_full"] = [Barrier(f"q_full[{s}]", q_full_arrivals) for s in range(stages)]
    bars["q_empty"] = [Barrier(f"q_empty[{s}]", 1) for s in range(stages)]
    bars["do_empty"] = [Barrier(f"do_empty[{s}]", 1) for s in range(stages)]
    stats = [Barrier("stats_ready[0]", n_warps), Barrier("stats_ready[1]", n_warps)]
    st = {"pr": 0, "dsr": 0, "af": 0}

    def q_producer():
        kvu = n = 0
        for it, nq in enumerate(items):
            yield ("wait", kv_empty, (kvu & 1) ^ 1)
            kvu += 1
            yield ("arrive_tx", kv_full, it, 2)
            for _ in range(nq):
                yield ("wait", bars["q_empty"][n % stages], ((n // stages) & 1) ^ 1)
                yield ("arrive_tx", bars["q_full"][n % stages], n, 1)
                n += 1

    def do_producer():
        n = 0
        for it, nq in enumerate(items):
            for _ in range(nq):
                yield ("wait", bars["do_empty"][n % stages], ((n // stages) & 1) ^ 1)
                yield ("arrive_tx", bars["q_full"][n % stages], n, 1)
                n += 1

    def issuer():
        kvc = n = 0
        for it, nq in enumerate(items):
            yield ("wait", kv_full, kvc & 1)
            kvc += 1
            yield from _dkdv_issuer_item(it, n, nq, st, bars, n_warps, stages)
            yield ("commit", kv_empty, it)
            n += nq

    roles = {"q_producer": q_producer(), "do_producer": do_producer(), "issuer": issuer()}
    roles.update({f"warp{w}": _dkdv_elementwise(items, rng, w, bars, stats) for w in range(n_warps)})
    return roles, tc


def fwd_loads_protocol(items, rng, warps_per_tile=4, kstages=2, vstages=3, s_before_pv=False):
    """The forward kernel with its producer: Q per tile (q_full / q_empty),
    and each key tile's K and V landing on the K slot's full barrier (two
    loads); the issuer waits once per key tile and releases K after the score
    MMAs and V after the value MMAs.  items: (key tiles of tile 0, of tile 1).
    TMEM per softmax warp w of tile t: ("S", t, w) holds S_j, then the P_j the
    warp writes over it, which PV_j reads; ("U", t, w) holds the value
    accumulator after PV_j (tag j), which the warp may rescale after seeing
    S_{j+1} and reads out after o_done.  (The issuer's o_free wait before an
    item's first PV is implied by that PV's p_full: each softmax warp writes the
    item's first P only after its epilogue has read U.)  s_before_pv plants the
    mistake of issuing S_{j+1} ahead of the PV_j that reads P_j."""
    W = range(warps_per_tile)
    tc = TensorCore()
    q_full = [Barrier(f"q_full[{t}]", 1) for t in (0, 1)]
    q_empty = [Barrier(f"q_empty[{t}]", 1) for t in (0, 1)]
    k_full = [Barrier(f"k_full[{s}]", 1) for s in range(kstages)]
    k_empty = [Barrier(f"k_empty[{s}]", 1) for s in range(kstages)]
    v_empty = [Barrier(f"v_empty[{s}]", 1) for s in range(vstages)]
    s_full = [Barrier(f"s_full[{t}]", 1) for t in (0, 1)]
    p_full = [Barrier(f"p_full[{t}]", warps_per_tile) for t in (0, 1)]
    o_done = [Barrier(f"o_done[{t}]", 1) for t in (0, 1)]
    o_free = [Barrier(f"o_free[{t}]", warps_per_tile) for t in (0, 1)]

    def producer():
        qu = [0, 0]
        kn = 0
        for it, ns in enumerate(items):
            for t in (0, 1):
                if ns[t] == 0:
                    continue
                yield ("wait", q_empty[t], (qu[t] & 1) ^ 1)
                qu[t] += 1
                yield ("arrive_tx", q_full[t], it, 1)
            for _ in range(max(ns)):
                yield ("wait", k_empty[kn % kstages], ((kn // kstages) & 1) ^ 1)
                yield ("wait", v_empty[kn % vstages], ((kn // vstages) & 1) ^ 1)
                yield ("arrive_tx", k_full[kn % kstages], kn, 2)
                kn += 1

    def issuer():
        qc, pc, of = [0, 0], [0, 0], [0, 0]
        kn = 0  # global number of the next key tile to take
        for it, ns in enumerate(items):
            nkv = max(ns)
            if nkv == 0:
                continue
            for t in (0, 1):
                if ns[t]:
                    yield ("wait", q_full[t], qc[t] & 1)
                    qc[t] += 1
            g = kn  # key tile 0 of this item
            yield ("wait", k_full[g % kstages], (g // kstages) & 1)
            kn += 1
            for t in (0, 1):
                if ns[t]:
                    yield ("mma", [], [(("S", t, w), ("S", it, 0)) for w in W])
                    yield ("commit", s_full[t], (it, 0))
                    if ns[t] == 1:
                        yield ("commit", q_empty[t], it)
            yield ("commit", k_empty[g % kstages], g)
            for j in range(nkv):
                gj = g + j  # V_j landed with K_j
                have_next = False
                for t in (0, 1):
                    if j >= ns[t]:
                        continue
                    yield ("wait", p_full[t], pc[t] & 1)
                    pc[t] += 1
                    if j == 0:
                        yield ("wait", o_free[t], (of[t] & 1) ^ 1)
                        of[t] += 1

                    def next_s():
                        nonlocal have_next, kn
                        if not have_next:
                            yield ("wait", k_full[(gj + 1) % kstages], ((gj + 1) // kstages) & 1)
                            kn += 1
                            have_next = True
                        yield ("mma", [], [(("S", t, w), ("S", it, j + 1)) for w in W])  # S_{j+1}(t)
                        yield ("commit", s_full[t], (it, j + 1))
                        if j + 1 == ns[t] - 1:
                            yield ("commit", q_empty[t], it)

                    if s_before_pv and j + 1 < ns[t]:
                        yield from next_s()
                    # PV_j(t) reads V_j and P_j, and adds to U (which must hold j - 1)
                    yield ("mma", [(("S", t, w), ("P", it, j)) for w in W] +
                           ([(("U", t, w), ("U", it, j - 1)) for w in W] if j else []),
                           [(("U", t, w), ("U", it, j)) for w in W])
                    if j == ns[t] - 1:
                        yield ("commit", o_done[t], it)
                    if j + 1 < ns[t] and not s_before_pv:
                        yield from next_s()
                yield ("commit", v_empty[gj % vstages], gj)
                if have_next:
                    yield ("commit", k_empty[(gj + 1) % kstages], gj + 1)

    def softmax(t, w):
        sc = oc = 0
        for it, ns in enumerate(items):
            n = ns[t]
            if n == 0:
                continue
            for j in range(n):
                yield ("wait", s_full[t], sc & 1)
                sc += 1
                yield ("read", ("S", t, w), ("S", it, j))
                if j and rng.random() < 0.3:  # the row max grew: rescale U (PV_{j-1} is done)
                    yield ("read", ("U", t, w), ("U", it, j - 1))
                    yield ("write", ("U", t, w), ("U", it, j - 1))
                for _ in range(rng.randint(1, 6)):
                    yield ("work",)
                yield ("write", ("S", t, w), ("P", it, j))
                yield ("arrive", p_full[t], (it, j))
            yield ("wait", o_done[t], oc & 1)
            oc += 1
            yield ("read", ("U", t, w), ("U", it, n - 1))  # the epilogue reads U
            yield ("work",)
            yield ("arrive", o_free[t], it)

    roles = {"producer": producer(), "issuer": issuer()}
    for t in (0, 1):
        roles.update({f"sm{t}.{w}": softmax(t, w) for w in W})
    return roles, tc


def dq_loads_protocol(items, rng, n_warps=8, kstages=3, vstages=2):
    """The dq kernel with its producer: Q and dO per item (q_full / q_empty),
    each key block's K and V on the K slot's full barrier; V is released after
    dP, K after dQ; the issuer as in dq_protocol."""
    tc = TensorCore()
    q_full, q_empty = Barrier("q_full", 1), Barrier("q_empty", 1)
    bars = _dq_bars(n_warps)
    bars["k_full"] = [Barrier(f"k_full[{s}]", 1) for s in range(kstages)]
    bars["k_empty"] = [Barrier(f"k_empty[{s}]", 1) for s in range(kstages)]
    bars["v_empty"] = [Barrier(f"v_empty[{s}]", 1) for s in range(vstages)]
    st = {"ds": 0, "af": 0}

    def producer():
        qu = kn = 0
        for it, nk in enumerate(items):
            yield ("wait", q_empty, (qu & 1) ^ 1)
            qu += 1
            yield ("arrive_tx", q_full, it, 2)
            for _ in range(nk):
                yield ("wait", bars["k_empty"][kn % kstages], ((kn // kstages) & 1) ^ 1)
                yield ("wait", bars["v_empty"][kn % vstages], ((kn // vstages) & 1) ^ 1)
                yield ("arrive_tx", bars["k_full"][kn % kstages], kn, 2)
                kn += 1

    def issuer():
        qc = g = 0
        for it, nk in enumerate(items):
            yield ("wait", q_full, qc & 1)
            qc += 1
            yield from _dq_issuer_item(it, g, nk, st, bars, kstages, vstages)
            yield ("commit", q_empty, it)
            g += nk

    roles = {"producer": producer(), "issuer": issuer()}
    roles.update({f"warp{w}": _dq_warp(items, rng, bars) for w in range(n_warps)})
    return roles, tc


def dkdv_fused_protocol(items, rng, n_warps=8, stages=2, ds_in_do_slot=True):
    """The dK/dV kernel with dq folded in (opt-in fused mode): per block also
    dQ_qb = dS K into TMEM (dq_full), read out by the elementwise warps in the
    next block (dq_free); at D = 128 dS lives in the block's dO slot, so its
    store waits for dV (dv_done) and the next dP^T waits for the dQ read-out
    (dq_region_free); at D = 64 (ds_in_do_slot False) dQ has TMEM of its own
    and only the dQ MMA waits for the previous read-out."""
    tc = TensorCore()
    kv_full, kv_empty = Barrier("kv_full", 1), Barrier("kv_empty", 1)
    q_full = [Barrier(f"q_full[{s}]", 2) for s in range(stages)]
    q_empty = [Barrier(f"q_empty[{s}]", 1) for s in range(stages)]
    do_empty = [Barrier(f"do_empty[{s}]", 1) for s in range(stages)]
    st_full, dp_full = Barrier("st_full", 1), Barrier("dp_full", 1)
    p_ready, ds_ready = Barrier("p_ready", n_warps), Barrier("ds_ready", n_warps)
    acc_done, acc_free = Barrier("acc_done", 1), Barrier("acc_free", n_warps)
    dq_full, dq_free = Barrier("dq_full", 1), Barrier("dq_free", n_warps)
    dv_done = Barrier("dv_done", 1)
    stats = [Barrier("stats_ready[0]", n_warps), Barrier("stats_ready[1]", n_warps)]

    def q_producer():
        kvu = n = 0
        for it, nq in enumerate(items):
            yield ("wait", kv_empty, (kvu & 1) ^ 1)
            kvu += 1
            yield ("arrive_tx", kv_full, it, 2)
            for _ in range(nq):
                yield ("wait", q_empty[n % stages], ((n // stages) & 1) ^ 1)
                yield ("arrive_tx", q_full[n % stages], n, 1)
                n += 1

    def do_producer():
        n = 0
        for it, nq in enumerate(items):
            for _ in range(nq):
                yield ("wait", do_empty[n % stages], ((n // stages) & 1) ^ 1)
                yield ("arrive_tx", q_full[n % stages], n, 1)
                n += 1

    def issuer():
        st = {"kv": 0, "p": 0, "ds": 0, "af": 0, "dqf": 0, "issued": 0}

        def region_free():
            while st["dqf"] < st["issued"]:
                yield ("wait", dq_free, st["dqf"] & 1)
                st["dqf"] += 1

        n = 0
        for it, nq in enumerate(items):
            yield ("wait", kv_full, st["kv"] & 1)
            st["kv"] += 1
            yield ("wait", q_full[n % stages], (n // stages) & 1)
            yield ("mma",)
            yield ("commit", st_full, n)
            if ds_in_do_slot:
                yield from region_free()
            yield ("mma",)
            yield ("commit", dp_full, n)
            for qb in range(nq):
                cur = n + qb
                yield ("wait", p_ready, st["p"] & 1)
                st["p"] += 1
                if qb == 0:
                    yield ("wait", acc_free, (st["af"] & 1) ^ 1)
                    st["af"] += 1
                yield ("mma",)  # dV reads dO
                if ds_in_do_slot:
                    yield ("commit", dv_done, cur)
                if qb > 0:
                    if ds_in_do_slot:
                        yield from region_free()
                    yield ("mma",)  # dP^T of this block
                    yield ("commit", dp_full, cur)
                if qb + 1 < nq:
                    yield ("wait", q_full[(cur + 1) % stages], ((cur + 1) // stages) & 1)
                    yield ("mma",)
                    yield ("commit", st_full, cur + 1)
                yield ("wait", ds_ready, st["ds"] & 1)
                st["ds"] += 1
                yield ("mma",)  # dK reads Q
                yield ("commit", q_empty[cur % stages], cur)
                if not ds_in_do_slot:
                    yield from region_free()
                yield ("mma",)  # dQ reads dS (in the dO slot at D = 128)
                st["issued"] += 1
                yield ("commit", dq_full, cur)
                yield ("commit", do_empty[cur % stages], cur)
            yield ("commit", acc_done, it)
            yield ("commit", kv_empty, it)
            n += nq

    def warp():
        c = {"st": 0, "dp": 0, "ad": 0, "si": 0, "dqf": 0}
        blk = 0

        def drain(tag):
            yield ("wait", dq_full, c["dqf"] & 1)
            c["dqf"] += 1
            yield ("work",)
            yield ("arrive", dq_free, tag)

        for it, nq in enumerate(items):
            for qb in range(nq):
                yield ("arrive", stats[c["si"] & 1], c["si"])
                yield ("wait", stats[c["si"] & 1], (c["si"] >> 1) & 1)
                c["si"] += 1
                yield ("wait", st_full, c["st"] & 1)
                c["st"] += 1
                for _ in range(rng.randint(1, 6)):
                    yield ("work",)
                yield ("arrive", p_ready, blk)
                if qb > 0:
                    yield from drain(blk - 1)
                yield ("wait", dp_full, c["dp"] & 1)
                c["dp"] += 1
                yield ("work",)
                if ds_in_do_slot:
                    yield ("wait", dv_done, blk & 1)
                yield ("work",)
                yield ("arrive", ds_ready, blk)
                blk += 1
            yield from drain(blk - 1)
            yield ("wait", acc_done, c["ad"] & 1)
            c["ad"] += 1
            yield ("work",)
            yield ("arrive", acc_free, it)

    roles = {"q_producer": q_producer(), "do_producer": do_producer(), "issuer": issuer()}
    roles.update({f"warp{w}": warp() for w in range(n_warps)})
    return roles, tc


def sched_ring_protocol(n_items, rng, n_consumers=10, counted_consumers=None, record=None):
    """The two-slot ring through which a CTA's producer warp hands its work
    items to the other roles (sched_full: one arrival; sched_empty: one per
    consumer).  Each consumer must read the items in order: `record` collects
    what every consumer read.  counted_consumers < n_consumers models a
    consumer left out of sched_empty's count."""
    tc = TensorCore()
    counted = n_consumers if counted_consumers is None else counted_consumers
    full = [Barrier(f"sched_full[{s}]", 1) for s in (0, 1)]
    empty = [Barrier(f"sched_empty[{s}]", counted) for s in (0, 1)]
    slot_value = [None, None]
    seen = record if record is not None else {}

    def producer():
        for i in range(n_items + 1):  # the last item is the end marker
            s = i & 1
            yield ("wait", empty[s], ((i >> 1) & 1) ^ 1)
            slot_value[s] = i
            yield ("arrive", full[s], i)

    def consumer(c):
        got = seen.setdefault(c, [])
        for i in range(n_items + 1):
            s = i & 1
            yield ("wait", full[s], (i >> 1) & 1)
            got.append(slot_value[s])
            yield ("arrive", empty[s], i)

    roles = {"producer": producer()}
    roles.update({f"c{c}": consumer(c) for c in range(n_consumers)})
    return roles, tc
