"""CPU model of the mbarrier pipelines of the SWA and GA prefill kernels, the
general prefill kernel, the decode kernel and the backward kernels (dq and
dk/dv).

Each kernel role (the copy thread, the MMA thread, the row threads of the two
column halves) is a generator that yields the operations it performs, in the
order the kernel performs them:

  ("wait", bar, n)         block until `bar` has completed n phases.  The kernel
                           waits on the parity of phase n-1, which is only
                           unambiguous while the barrier has completed n-1 or n
                           phases: with n+1 the wait would miss its phase, with
                           n-2 or fewer it would pass at once on an older one.
                           The model fails on either.
  ("arrive", bar)          one arrival; a barrier completes a phase after
                           `counts[bar]` arrivals (1 unless the roles say).
  ("tma", res, tag, bar)   an asynchronous copy: later, in any order, `res` gets
                           `tag` (res and tag may be lists: one copy of several
                           boxes) and `bar` completes a phase.
  ("mma", reads, writes)   an MMA joins the tensor pipe, which executes in issue
                           order; on execution every (res, tag) it reads must hold
                           that tag, then every (res, tag) it writes is set.
  ("commit", bar)          joins the tensor pipe behind the MMAs issued so far;
                           `bar` completes a phase when it is reached.
  ("read", res, tag)       a thread reads `res` (TMEM or shared memory): it must
                           hold `tag` (written and complete, not overwritten yet).
  ("write", res, tag)      a thread writes `res`.
  ("sync",)                the CTA barrier: every role must arrive.
  ("await", bar, n)        a bounded wait (the kernels' wait_bar): like "wait",
                           but once the CTA is aborting it may return False (the
                           value the generator receives) instead of blocking.
  ("drain", bar, n)        the wait of the drain after an abort: blocks until
                           `bar` has completed n phases, whatever the abort flag.

With `aborts=True` a blocked "await" may time out at any moment (rarely, at
random): the CTA's abort flag is set, that await returns False, and so may
every later await that is not already satisfied.  Roles then run their drain
code.  When every role has finished, no copy may still be in flight and the
tensor pipe must be empty: the kernel frees shared memory and TMEM there.

A scheduler picks at random among the runnable roles, the copies in flight and
the head of the tensor pipe, so one run is one interleaving; many runs with
different seeds explore many.  A run fails on a deadlock, an ambiguous parity
wait, or a read of a resource that does not hold what the reader expects (a
read before the write landed, or after the next write replaced it).
"""
import random


class ModelError(AssertionError):
    pass


# A roles factory that models its kernel's drain puts this key in its counts:
# then, also without aborts, nothing may be in flight when every role is done.
EXIT_CHECK = "__exit_check__"


class Sim:
    def __init__(self, roles, rng, counts=None, aborts=False):
        self.rng = rng
        self.aborts = aborts                  # random timeouts enabled
        self.aborted = False                  # the CTA's abort flag
        self.counts = dict(counts or {})      # barrier -> arrivals per phase
        self.exit_checked = aborts or bool(self.counts.pop(EXIT_CHECK, False))
        self.arrivals = {}
        self.roles = dict(roles)              # name -> generator
        self.pending = {n: None for n in self.roles}  # the op a role is blocked on
        self.done = set()
        self.phases = {}                      # barrier -> completed phases
        self.res = {}                         # resource -> tag
        self.tma = []                         # copies in flight: (res, tag, bar)
        self.pipe = []                        # tensor pipe: ("mma", reads, writes) | ("commit", bar)
        self.sync_waiting = set()

    def _complete(self, bar):
        self.phases[bar] = self.phases.get(bar, 0) + 1

    def _arrive(self, bar):
        self.arrivals[bar] = self.arrivals.get(bar, 0) + 1
        if self.arrivals[bar] == self.counts.get(bar, 1):
            self.arrivals[bar] = 0
            self._complete(bar)

    def _check_waits(self):
        for name, op in self.pending.items():
            if op is not None and op[0] in ("wait", "await", "drain"):
                _, bar, n = op
                c = self.phases.get(bar, 0)
                if c > n or c < n - 1:
                    raise ModelError(f"{name}: waits for {n} phases of {bar}, which has "
                                     f"completed {c} (parity wait ambiguous)")

    def _satisfied(self, op):
        return self.phases.get(op[1], 0) >= op[2]

    def _runnable(self, name):
        op = self.pending[name]
        if op is None:
            return True
        if op[0] in ("wait", "drain"):
            return self._satisfied(op)
        if op[0] == "await":
            return self._satisfied(op) or self.aborted
        if op[0] == "sync":
            return False
        return True

    def _step_role(self, name):
        op = self.pending[name]
        result = None
        if op is not None:
            kind = op[0]
            if kind in ("wait", "drain"):
                pass  # satisfied (checked by _runnable)
            elif kind == "await":
                result = self._satisfied(op)  # False: the CTA is aborting
            elif kind == "arrive":
                self._arrive(op[1])
            elif kind == "tma":
                self.tma.append(op[1:])
            elif kind == "mma":
                self.pipe.append(op)
            elif kind == "commit":
                self.pipe.append(op)
            elif kind == "read":
                _, r, tag = op
                if self.res.get(r) != tag:
                    raise ModelError(f"{name}: reads {r} expecting {tag}, holds {self.res.get(r)}")
            elif kind == "write":
                self.res[op[1]] = op[2]
            else:
                raise ValueError(op)
        try:
            self.pending[name] = self.roles[name].send(result)
        except StopIteration:
            self.pending[name] = None
            self.done.add(name)
            return
        if self.pending[name][0] == "sync":
            self.sync_waiting.add(name)

    def run(self, max_steps=2_000_000):
        for name in self.roles:
            self._step_role_first(name)
        for _ in range(max_steps):
            self._check_waits()
            live = [n for n in self.roles if n not in self.done]
            if not live and self.exit_checked and (self.tma or self.pipe):
                raise ModelError(f"every role finished with copies {self.tma} or tensor-pipe "
                                 f"work {self.pipe} still in flight")
            if not live and not self.tma and not self.pipe:
                return
            # the CTA barrier releases once every live role has reached it
            if live and self.sync_waiting == set(live):
                self.sync_waiting.clear()
                for n in live:
                    self.pending[n] = ("wait", "__none__", 0)  # released: no-op
                    self.phases.setdefault("__none__", 0)
            choices = [("role", n) for n in live if self._runnable(n)]
            if self.aborts and not self.aborted and self.rng.random() < 0.01:
                blocked = [n for n in live if self.pending[n] is not None
                           and self.pending[n][0] == "await" and not self._satisfied(self.pending[n])]
                if blocked:
                    self.aborted = True  # a wait ran out: the CTA aborts
                    choices = [("role", self.rng.choice(blocked))]
            choices += [("tma", i) for i in range(len(self.tma))]
            if self.pipe:
                choices.append(("pipe", 0))
            if not choices and self.aborts and not self.aborted:
                # nothing can move: a bounded wait is the next thing to run out
                blocked = [n for n in live if self.pending[n] is not None
                           and self.pending[n][0] == "await"]
                if blocked:
                    self.aborted = True
                    choices = [("role", self.rng.choice(blocked))]
            if not choices:
                state = {n: self.pending[n] for n in live}
                raise ModelError(f"deadlock: {state}")
            kind, i = self.rng.choice(choices)
            if kind == "role":
                self._step_role(i)
            elif kind == "tma":
                r, tag, bar = self.tma.pop(i)
                if isinstance(r, list):
                    for rr, tt in zip(r, tag):
                        self.res[rr] = tt
                else:
                    self.res[r] = tag
                self._complete(bar)
            else:
                op = self.pipe.pop(0)
                if op[0] == "commit":
                    self._complete(op[1])
                else:
                    _, reads, writes = op
                    for r, tag in reads:
                        if self.res.get(r) != tag:
                            raise ModelError(f"MMA reads {r} expecting {tag}, holds {self.res.get(r)}")
                    for r, tag in writes:
                        self.res[r] = tag
        raise ModelError("step limit")

    def _step_role_first(self, name):
        try:
            self.pending[name] = next(self.roles[name])
        except StopIteration:
            self.pending[name] = None
            self.done.add(name)
            return
        if self.pending[name][0] == "sync":
            self.sync_waiting.add(name)


NS = 3  # K/V (dq) or Q/dO (dk/dv) stages


def dq_roles(nblk, skip=()):
    """The dq kernel for one CTA whose items have nblk[i] key blocks each.  The
    roles meet only on mbarriers: the rows tell the MMA thread that dS(g) is in
    TMEM (DSR, per S/dP buffer); the same threads ran the previous item's
    epilogue before, so the first dQ of an item cannot overwrite what the
    epilogue still reads.  The MMA thread frees a K/V stage with a commit after
    the dQ that read it (KVE), the Q/dO tile with a commit after the item's last
    S/dP (QE) and hands the finished dQ to the rows with a commit after the
    item's last dQ (ACCF): one phase per item, so neither of the last two waits
    can find its barrier two phases behind.  Every wait is bounded ("await"):
    a role whose wait returns False (the CTA is aborting) leaves its loop; the
    copy thread then waits for the last copy into the Q/dO tile and into each
    K/V stage and the MMA thread for a commit behind its last MMA, as the
    kernel does before shared memory and TMEM go back.
    `skip` names waits to leave out (to show that the model notices)."""
    items = list(nblk)
    seq = [(it, j) for it, n in enumerate(items) for j in range(n)]  # loader order
    first = [sum(items[:i]) for i in range(len(items))]

    def producer():
        yield ("tma", "QO", ("QO", 0), "QF")
        n_q, ld_g = 1, 0
        for ld in range(len(seq)):
            st = ld % NS
            if ld >= NS and "producer_kve" not in skip:
                if not (yield ("await", f"KVE{st}", ld // NS)):  # dQ(ld - NS) read the stage
                    break
            yield ("tma", f"KV{st}", ("KV", ld), f"KV{st}")
            ld_g += 1
            it, j = seq[ld]
            # once block ld is queued, the next item's Q/dO follows the item's
            # last S/dP (interleaved with the K/V loads as the kernel does)
            if j == items[it] - 1 and it + 1 < len(items):
                if "producer_qe" not in skip:
                    if not (yield ("await", "QE", it + 1)):
                        break
                yield ("tma", "QO", ("QO", it + 1), "QF")
                n_q += 1
        # drain: no copy may still be landing when shared memory goes back
        if "producer_drain" not in skip:
            yield ("drain", "QF", n_q)
            for st in range(NS):
                if ld_g > st:
                    yield ("drain", f"KV{st}", (ld_g - 1 - st) // NS + 1)

    def issuer():
        def issue_sdp(it, g):
            if not (yield ("await", f"KV{g % NS}", g // NS + 1)):
                return False
            b = g & 1
            yield ("mma", [("QO", ("QO", it)), (f"KV{g % NS}", ("KV", g))],
                   [(f"S{b}h0", ("S", g)), (f"S{b}h1", ("S", g))])
            yield ("commit", f"MM1{b}")
            return True

        issued = False
        ok = True
        for it, n in enumerate(items):
            g0 = first[it]
            ok = yield ("await", "QF", it + 1)
            if ok:
                ok = yield from issue_sdp(it, g0)
            if not ok:
                break
            issued = True
            if n == 1:
                yield ("commit", "QE")
            for j in range(n):
                g = g0 + j
                if j + 1 < n:
                    ok = yield from issue_sdp(it, g + 1)
                    if not ok:
                        break
                    if j + 2 == n:
                        yield ("commit", "QE")  # the item's last S/dP
                b = g & 1
                if "issuer_dsr" not in skip:
                    ok = yield ("await", f"DSR{b}", (g >> 1) + 1)  # both row halves wrote dS(g)
                    if not ok:
                        break
                reads = [(f"S{b}h0", ("dS", g)), (f"S{b}h1", ("dS", g)), (f"KV{g % NS}", ("KV", g))]
                if j > 0:
                    reads.append(("dQ", ("dQ", it, j - 1)))
                yield ("mma", reads, [("dQ", ("dQ", it, j))])
                yield ("commit", f"KVE{g % NS}")
                if j == n - 1:
                    yield ("commit", "ACCF")
            if not ok:
                break
        # drain: every MMA done before TMEM goes back
        if issued and "mma_drain" not in skip:
            yield ("commit", "DRAIN")
            yield ("drain", "DRAIN", 1)

    def rows(h):
        def role():
            for it, n in enumerate(items):
                g0 = first[it]
                for j in range(n):
                    g = g0 + j
                    b = g & 1
                    if not (yield ("await", f"MM1{b}", (g >> 1) + 1)):
                        return
                    yield ("read", f"S{b}h{h}", ("S", g))
                    yield ("write", f"S{b}h{h}", ("dS", g))  # dS over this half's S columns
                    yield ("arrive", f"DSR{b}")
                if "rows_accf" not in skip:
                    if not (yield ("await", "ACCF", it + 1)):  # the item's last dQ
                        return
                yield ("read", "dQ", ("dQ", it, n - 1))
        return role()

    roles = {"producer": producer(), "issuer": issuer(), "rows0": rows(0), "rows1": rows(1)}
    return roles, {"DSR0": 2, "DSR1": 2, EXIT_CHECK: True}


def dkdv_roles(nsub, skip=()):
    """The dk/dv kernel for one CTA whose items (key blocks) have nsub[i] query
    sub-tiles each.  The roles meet only on mbarriers: the rows tell the MMA
    thread that they have read S^T/dP^T(g) into registers (SR, 256 arrivals;
    S^T/dP^T(g+1) follow into the same columns) and that P^T/dS^T(g) are in
    TMEM (PR, 256 arrivals; dV/dK(g) follow); rows 0..63 stage lse and D of the next sub-tile in one of
    two shared-memory slots (LF: written).  They write slot (g+1) & 1 after
    waiting for dV/dK(g-1), which needed every row's PR for sub-tile g-1, so
    every read of that slot's previous contents is done.  The MMA thread
    frees a Q/dO stage after the dV/dK that read it (QSE), the K/V block after
    the item's last S^T/dP^T (KVE) and hands the finished accumulators to the
    rows after the item's last dV/dK (ACCF).  Every wait is bounded, with the
    copy and MMA threads' drains of the dq kernel.  `skip` names waits to
    leave out."""
    items = list(nsub)
    seq = [(it, j) for it, n in enumerate(items) for j in range(n)]
    first = [sum(items[:i]) for i in range(len(items))]
    total = len(seq)

    def producer():
        yield ("tma", "KVB", ("KVB", 0), "KF")
        n_kv, ld_g = 1, 0
        for ld in range(total):
            it, j = seq[ld]
            if j == 0 and it > 0:
                if "producer_kve" not in skip:
                    if not (yield ("await", "KVE", it)):  # the previous item's last S^T/dP^T
                        break
                yield ("tma", "KVB", ("KVB", it), "KF")
                n_kv += 1
            if ld >= NS and "producer_qse" not in skip:
                # dV/dK(ld - NS) read the stage
                if not (yield ("await", f"QSE{ld % NS}", ld // NS)):
                    break
            yield ("tma", f"QO{ld % NS}", ("QO", ld), f"QS{ld % NS}")
            ld_g += 1
        if "producer_drain" not in skip:
            yield ("drain", "KF", n_kv)
            for st in range(NS):
                if ld_g > st:
                    yield ("drain", f"QS{st}", (ld_g - 1 - st) // NS + 1)

    def issuer():
        def issue_sdp(it, g):
            if not (yield ("await", f"QS{g % NS}", g // NS + 1)):
                return False
            yield ("mma", [("KVB", ("KVB", it)), (f"QO{g % NS}", ("QO", g))],
                   [("STh0", ("ST", g)), ("STh1", ("ST", g))])
            yield ("commit", "MM1")
            return True

        issued = False
        ok = True
        for it, n in enumerate(items):
            g0 = first[it]
            ok = yield ("await", "KF", it + 1)
            if ok:
                ok = yield from issue_sdp(it, g0)
            if not ok:
                break
            issued = True
            if n == 1:
                yield ("commit", "KVE")
            for s in range(n):
                g = g0 + s
                if s + 1 < n:
                    if "issuer_sr" not in skip:
                        ok = yield ("await", "SR", g + 1)  # S^T/dP^T(g) read by every row
                        if not ok:
                            break
                    ok = yield from issue_sdp(it, g + 1)
                    if not ok:
                        break
                    if s + 2 == n:
                        yield ("commit", "KVE")
                if "issuer_pr" not in skip:
                    ok = yield ("await", "PR", g + 1)  # P^T/dS^T(g) written
                    if not ok:
                        break
                reads = [("Ph0", ("P", g)), ("Ph1", ("P", g)), (f"QO{g % NS}", ("QO", g))]
                if s > 0:
                    reads.append(("acc", ("acc", it, s - 1)))
                yield ("mma", reads, [("acc", ("acc", it, s))])
                yield ("commit", "MM2")
                yield ("commit", f"QSE{g % NS}")
                if s + 1 == n:
                    yield ("commit", "ACCF")
            if not ok:
                break
        if issued and "mma_drain" not in skip:
            yield ("commit", "DRAIN")
            yield ("drain", "DRAIN", 1)

    def rows(h, writer):
        def role():
            if writer:  # the first sub-tile's lse / D
                yield ("write", "L0", ("L", 0))
                yield ("arrive", "LF0")
            for it, n in enumerate(items):
                g0 = first[it]
                for s in range(n):
                    g = g0 + s
                    if not (yield ("await", "MM1", g + 1)):
                        return
                    yield ("read", f"STh{h}", ("ST", g))
                    yield ("arrive", "SR")
                    if "rows_lf" not in skip:
                        if not (yield ("await", f"LF{g & 1}", (g >> 1) + 1)):
                            return
                    yield ("read", f"L{g & 1}", ("L", g))
                    if g > 0 and "rows_mm2" not in skip:
                        if not (yield ("await", "MM2", g)):  # dV/dK(g-1) read P^T/dS^T
                            return
                    yield ("write", f"Ph{h}", ("P", g))
                    yield ("arrive", "PR")
                    if writer and g + 1 < total:
                        yield ("write", f"L{(g + 1) & 1}", ("L", g + 1))
                        yield ("arrive", f"LF{(g + 1) & 1}")
                if not (yield ("await", "ACCF", it + 1)):
                    return
                yield ("read", "acc", ("acc", it, n - 1))
        return role()

    roles = {"producer": producer(), "issuer": issuer(), "rows0": rows(0, True),
             "rows1": rows(1, False)}
    # PR, SR: both row roles arrive; LF: only the writer
    return roles, {"PR": 2, "SR": 2, EXIT_CHECK: True}


def run(make_roles, sizes, seed, skip=(), aborts=False):
    roles, counts = make_roles(sizes, skip)
    sim = Sim(roles, random.Random(seed), counts, aborts=aborts)
    sim.run()
    return sim


def decode_roles(nblk, f8=False, skip=()):
    """sinkattn_decode_kernel for one CTA whose segments (the cache blocks of a
    unit in this CTA's range) have nblk[i] 64-key blocks each: the copy thread,
    the MMA thread, the softmax rows and the RoPE / conversion warps.  bf16
    cache: four K/V stages the copies fill.  FP8 cache: two staging slots the
    copies fill and three fp16 stages the conversion warps fill.  QK^T(j) is
    issued before PV(j-1), which waits for the softmax of block j-1.  The
    conversion warps rotate each unit's Q tile in shared memory, copy it into
    one of two TMEM buffers (QK^T reads it there) once the last QK^T of the
    unit two back has freed that buffer (QTFREE, a commit), and then free the
    shared-memory tile.  Every wait is bounded ("await"); after leaving its loop
    the copy thread waits for the last copy into the Q tile and into each
    stage or slot, and the MMA thread for a commit behind its last MMA."""
    segs = list(nblk)
    S = 3 if f8 else 4
    S8 = 2

    def producer():
        gk = gq = 0
        ok = True
        for q, n in enumerate(segs):
            ok = yield ("await", "QEMPTY", q)  # the rows copied the previous tile to TMEM
            if not ok:
                break
            yield ("tma", "Q", ("Qraw", q), "QFULL")
            gq += 1
            for _ in range(n):
                if f8:
                    s8 = gk % S8
                    ok = yield ("await", f"STGEMPTY{s8}", gk // S8)
                    if not ok:
                        break
                    yield ("tma", f"STG{s8}", ("stg", gk), f"STGFULL{s8}")
                else:
                    st = gk % S
                    if "producer_kvempty" not in skip:
                        ok = yield ("await", f"KVEMPTY{st}", gk // S)
                        if not ok:
                            break
                    yield ("tma", [f"K{st}", f"V{st}"], [("Kraw", gk), ("V", gk)], f"KVFULL{st}")
                gk += 1
            if not ok:
                break
        if "producer_drain" not in skip:
            if gq > 0:
                yield ("drain", "QFULL", gq)
            slots, name = (S8, "STGFULL") if f8 else (S, "KVFULL")
            for st in range(slots):
                if gk > st:
                    yield ("drain", f"{name}{st}", (gk - 1 - st) // slots + 1)

    def mma():
        gk = 0
        issued = False

        def issue_pv(q, j, b, first):
            if not (yield ("await", f"PFULL{b & 1}", (b >> 1) + 1)):
                return False
            if first:
                if not (yield ("await", "OEMPTY", q)):
                    return False
            reads = [(f"P{b & 1}", ("P", b)), (f"V{b % S}", ("V", b))]
            if not first:
                reads.append(("O", ("Ors", q, j - 1)))
            yield ("mma", reads, [("O", ("O", q, j))])
            yield ("commit", f"KVEMPTY{b % S}")
            yield ("commit", "PVDONE")
            return True

        def body():
            nonlocal gk, issued
            for q, n in enumerate(segs):
                qb = q & 1
                if not (yield ("await", f"QTMEM{qb}", q // 2 + 1)):
                    return
                for j in range(n):
                    b = gk + j
                    if not (yield ("await", f"KREADY{b % S}", b // S + 1)):
                        return
                    yield ("mma", [(f"QT{qb}", ("Q", q)), (f"K{b % S}", ("K", b))],
                           [(f"P{b & 1}", ("S", b))])
                    issued = True
                    yield ("commit", f"SFULL{b & 1}")
                    if j == n - 1:
                        yield ("commit", f"QTFREE{qb}")
                    if j > 0:
                        if not (yield from issue_pv(q, j - 1, b - 1, j == 1)):
                            return
                if not (yield from issue_pv(q, n - 1, gk + n - 1, n == 1)):
                    return
                gk += n

        yield from body()
        if issued and "mma_drain" not in skip:
            yield ("commit", "DRAIN")
            yield ("drain", "DRAIN", 1)

    def softmax():
        gs = 0
        for q, n in enumerate(segs):
            for j in range(n):
                b = gs + j
                if not (yield ("await", f"SFULL{b & 1}", (b >> 1) + 1)):
                    return
                yield ("read", f"P{b & 1}", ("S", b))
                yield ("write", f"P{b & 1}", ("P", b))  # P over the S columns
                if j > 0:
                    if "softmax_pvdone" not in skip:
                        if not (yield ("await", "PVDONE", b)):  # PV(j-1) complete
                            return
                    yield ("read", "O", ("O", q, j - 1))
                    yield ("write", "O", ("Ors", q, j - 1))  # rescale before PV(j)
                yield ("arrive", f"PFULL{b & 1}")
            if not (yield ("await", "PVDONE", gs + n)):
                return
            yield ("read", "O", ("O", q, n - 1))
            yield ("arrive", "OEMPTY")
            gs += n

    def convert():
        gk = 0
        for q, n in enumerate(segs):
            if not (yield ("await", "QFULL", q + 1)):
                return
            yield ("read", "Q", ("Qraw", q))
            yield ("write", "Q", ("Q", q))  # RoPE (and fp16) in place
            qb = q & 1
            if q >= 2 and "convert_qtfree" not in skip:
                # the unit two back read the buffer
                if not (yield ("await", f"QTFREE{qb}", q // 2)):
                    return
            yield ("read", "Q", ("Q", q))
            yield ("write", f"QT{qb}", ("Q", q))  # into TMEM buffer qb
            yield ("arrive", f"QTMEM{qb}")
            yield ("arrive", "QEMPTY")
            for _ in range(n):
                st = gk % S
                if f8:
                    # the staging slot's bytes go to registers and the slot back
                    # to the copies before the wait for the fp16 stage
                    s8 = gk % S8
                    if not (yield ("await", f"STGFULL{s8}", gk // S8 + 1)):
                        return
                    yield ("read", f"STG{s8}", ("stg", gk))
                    yield ("arrive", f"STGEMPTY{s8}")
                    if "convert_kvempty" not in skip:
                        if not (yield ("await", f"KVEMPTY{st}", gk // S)):  # PV(gk-S) read the stage
                            return
                    yield ("write", f"K{st}", ("K", gk))
                    yield ("write", f"V{st}", ("V", gk))
                else:
                    if not (yield ("await", f"KVFULL{st}", gk // S + 1)):  # K and V copies landed
                        return
                    yield ("read", f"K{st}", ("Kraw", gk))
                    yield ("write", f"K{st}", ("K", gk))  # RoPE in place
                yield ("arrive", f"KREADY{st}")
                gk += 1

    return ({"producer": producer(), "mma": mma(), "softmax": softmax(), "convert": convert()},
            {EXIT_CHECK: True})


def general_roles(nblk, skip=(), NQ=1, NKV=2):
    """sinkattn_fwd_kernel (the general prefill kernel) for one CTA whose items
    (one query tile each) run over nblk[i] key blocks: the copy thread (Q into
    NQ stages, K/V into NKV stages), the RoPE warps, the MMA thread and the
    softmax rows.  With one K/V stage (NQ = 2, NKV = 1: a window that fits one
    block per tile) PV(j-1) goes out before QK^T(j), which needs the stage back;
    with two, after it.  S and P share one of two buffers per block.  Every
    wait is bounded, with the copy and MMA threads' drains."""
    items = list(nblk)

    def producer():
        gq = gk = 0
        ok = True
        for n in items:
            qs = gq % NQ
            ok = yield ("await", f"QEMPTY{qs}", gq // NQ)
            if not ok:
                break
            yield ("tma", f"Q{qs}", ("Qraw", gq), f"QFULL{qs}")
            gq += 1
            for _ in range(n):
                ks = gk % NKV
                if "producer_kvempty" not in skip:
                    ok = yield ("await", f"KVEMPTY{ks}", gk // NKV)
                    if not ok:
                        break
                yield ("tma", f"KV{ks}", ("KVraw", gk), f"KVFULL{ks}")
                gk += 1
            if not ok:
                break
        if "producer_drain" not in skip:
            for st in range(NQ):
                if gq > st:
                    yield ("drain", f"QFULL{st}", (gq - 1 - st) // NQ + 1)
            for st in range(NKV):
                if gk > st:
                    yield ("drain", f"KVFULL{st}", (gk - 1 - st) // NKV + 1)

    def rope():
        gq = gk = 0
        for n in items:
            qs = gq % NQ
            if not (yield ("await", f"QFULL{qs}", gq // NQ + 1)):
                return
            yield ("read", f"Q{qs}", ("Qraw", gq))
            yield ("write", f"Q{qs}", ("Q", gq))
            yield ("arrive", f"QREADY{qs}")
            gq += 1
            for _ in range(n):
                ks = gk % NKV
                if "rope_kvfull" not in skip:
                    if not (yield ("await", f"KVFULL{ks}", gk // NKV + 1)):
                        return
                yield ("read", f"KV{ks}", ("KVraw", gk))
                yield ("write", f"KV{ks}", ("KV", gk))
                yield ("arrive", f"KREADY{ks}")
                gk += 1

    def mma():
        gq = gk = gs = gt = 0
        issued = False

        def issue_pv(i, jj):
            g = gs + jj
            buf = g & 1
            if not (yield ("await", f"PFULL{buf}", (g >> 1) + 1)):
                return False
            # (the O_EMPTY wait is implied by P_FULL: the softmax rows finish the
            # previous item's epilogue before they store this item's first P)
            if jj == 0 and "mma_oempty" not in skip:
                if not (yield ("await", "OEMPTY", gt)):
                    return False
            ks = (gk + jj) % NKV
            reads = [(f"S{buf}", ("P", g)), (f"KV{ks}", ("KV", gk + jj))]
            if jj > 0:
                reads.append(("O", ("Ors", i, jj - 1)))
            yield ("mma", reads, [("O", ("O", i, jj))])
            yield ("commit", f"KVEMPTY{ks}")
            yield ("commit", "PVDONE")
            return True

        def body():
            nonlocal gq, gk, gs, gt, issued
            for i, n in enumerate(items):
                qs = gq % NQ
                if not (yield ("await", f"QREADY{qs}", gq // NQ + 1)):
                    return
                for j in range(n):
                    if NKV == 1 and j > 0:
                        if not (yield from issue_pv(i, j - 1)):
                            return
                    gkj = gk + j
                    ks = gkj % NKV
                    if not (yield ("await", f"KREADY{ks}", gkj // NKV + 1)):
                        return
                    buf = (gs + j) & 1
                    yield ("mma", [(f"Q{qs}", ("Q", gq)), (f"KV{ks}", ("KV", gkj))],
                           [(f"S{buf}", ("S", gs + j))])
                    issued = True
                    yield ("commit", f"SFULL{buf}")
                    if j == n - 1:
                        yield ("commit", f"QEMPTY{qs}")
                    if NKV > 1 and j > 0:
                        if not (yield from issue_pv(i, j - 1)):
                            return
                if not (yield from issue_pv(i, n - 1)):
                    return
                gq += 1
                gk += n
                gs += n
                gt += 1

        yield from body()
        if issued and "mma_drain" not in skip:
            yield ("commit", "DRAIN")
            yield ("drain", "DRAIN", 1)

    def softmax():
        gs = gp = 0
        for i, n in enumerate(items):
            for j in range(n):
                buf = gs & 1
                if not (yield ("await", f"SFULL{buf}", (gs >> 1) + 1)):
                    return
                yield ("read", f"S{buf}", ("S", gs))
                yield ("write", f"S{buf}", ("P", gs))  # P over the S columns
                if j > 0:
                    if "softmax_pvdone" not in skip:
                        if not (yield ("await", "PVDONE", gp + 1)):  # PV(j-1) complete
                            return
                    yield ("read", "O", ("O", i, j - 1))
                    yield ("write", "O", ("Ors", i, j - 1))  # lazy rescale before PV(j)
                    gp += 1
                yield ("arrive", f"PFULL{buf}")
                gs += 1
            if not (yield ("await", "PVDONE", gp + 1)):
                return
            yield ("read", "O", ("O", i, n - 1))
            yield ("arrive", "OEMPTY")
            gp += 1

    roles = {"producer": producer(), "rope": rope(), "mma": mma(), "softmax": softmax()}
    return roles, {EXIT_CHECK: True}


def causal_roles(nblk, skip=()):
    """sinkattn_causal_kernel (GA prefill) for one CTA whose items (two query
    tiles A and B of one KV head) run over nblk[i] 128-key blocks: the Q/K copy
    warp, the V copy warp, the RoPE warps, the MMA thread and the softmax warps
    of each tile.  Per block the MMA thread issues PV_A(j), QK_A(j+1), PV_B(j),
    QK_B(j+1), so each tile's softmax overlaps the other tile's products.
    Every wait is bounded ("await"); after leaving its loop each copy thread
    waits for the last copy into each of its buffers and the MMA thread for a
    commit behind its last MMA, as the kernel does."""
    items = list(nblk)

    def producer():
        gk = gi = 0
        ok = True
        for i, n in enumerate(items):
            ok = yield ("await", "QEMPTY", i)  # the previous item's last QK^T read Q
            if not ok:
                break
            for x in range(2):
                yield ("tma", f"Q{x}", ("Qraw", i, x), f"QFULL{x}")
            gi += 1
            for _ in range(n):
                st = gk & 1
                if "producer_kempty" not in skip:
                    ok = yield ("await", f"KEMPTY{st}", gk >> 1)
                    if not ok:
                        break
                yield ("tma", f"K{st}", ("Kraw", gk), f"KFULL{st}")
                gk += 1
            if not ok:
                break
        if "producer_drain" not in skip:
            for x in range(2):
                if gi > 0:
                    yield ("drain", f"QFULL{x}", gi)
            for st in range(2):
                if gk > st:
                    yield ("drain", f"KFULL{st}", (gk - 1 - st) // 2 + 1)

    def vloader():
        gv = 0
        ok = True
        for n in items:
            for _ in range(n):
                if "vloader_vempty" not in skip:
                    ok = yield ("await", "VEMPTY", gv)
                    if not ok:
                        break
                yield ("tma", "V", ("V", gv), "VFULL")
                gv += 1
            if not ok:
                break
        if gv > 0 and "producer_drain" not in skip:
            yield ("drain", "VFULL", gv)

    def rope():
        gk = 0
        for i, n in enumerate(items):
            for x in range(2):
                if not (yield ("await", f"QFULL{x}", i + 1)):
                    return
                yield ("read", f"Q{x}", ("Qraw", i, x))
                yield ("write", f"Q{x}", ("Q", i, x))
                yield ("arrive", f"QREADY{x}")
            for _ in range(n):
                st = gk & 1
                if "rope_kfull" not in skip:
                    if not (yield ("await", f"KFULL{st}", (gk >> 1) + 1)):
                        return
                yield ("read", f"K{st}", ("Kraw", gk))
                yield ("write", f"K{st}", ("K", gk))
                yield ("arrive", f"KREADY{st}")
                gk += 1

    def mma():
        gk = gv = gp = 0
        issued = False

        def qk(i, x, b):
            yield ("mma", [(f"Q{x}", ("Q", i, x)), (f"K{b & 1}", ("K", b))], [(f"S{x}", ("S", x, b))])
            yield ("commit", f"SFULL{x}")

        def pv(i, x, j, b, first):
            if "mma_pfull" not in skip:
                if not (yield ("await", f"PFULL{x}", gp + 1)):
                    return False
            # (the O_EMPTY wait is implied by P_FULL: the softmax threads finish
            # the previous item's epilogue before they store this item's P)
            if first:
                if not (yield ("await", f"OEMPTY{x}", i)):
                    return False
            reads = [(f"S{x}", ("P", x, b)), ("V", ("V", gv))]
            if not first:
                reads.append((f"O{x}", ("Ors", x, i, j - 1)))
            yield ("mma", reads, [(f"O{x}", ("O", x, i, j))])
            yield ("commit", f"PVDONE{x}")
            return True

        def body():
            nonlocal gk, gv, gp, issued
            for i, n in enumerate(items):
                for w in (("QREADY0", i + 1), ("QREADY1", i + 1), (f"KREADY{gk & 1}", (gk >> 1) + 1)):
                    if not (yield ("await",) + w):
                        return
                yield from qk(i, 0, gk)
                issued = True
                yield from qk(i, 1, gk)
                yield ("commit", f"KEMPTY{gk & 1}")
                if n == 1:
                    yield ("commit", "QEMPTY")
                for j in range(n):
                    more = j + 1 < n
                    if not (yield ("await", "VFULL", gv + 1)):
                        return
                    if not (yield from pv(i, 0, j, gk, j == 0)):
                        return
                    if more:
                        if not (yield ("await", f"KREADY{(gk + 1) & 1}", ((gk + 1) >> 1) + 1)):
                            return
                        yield from qk(i, 0, gk + 1)
                    if not (yield from pv(i, 1, j, gk, j == 0)):
                        return
                    yield ("commit", "VEMPTY")
                    gv += 1
                    gp += 1
                    if more:
                        yield from qk(i, 1, gk + 1)
                        yield ("commit", f"KEMPTY{(gk + 1) & 1}")
                        if j + 1 == n - 1:
                            yield ("commit", "QEMPTY")
                    gk += 1

        yield from body()
        if issued and "mma_drain" not in skip:
            yield ("commit", "DRAIN")
            yield ("drain", "DRAIN", 1)

    def softmax(x):
        def role():
            gb = 0
            for i, n in enumerate(items):
                for j in range(n):
                    if not (yield ("await", f"SFULL{x}", gb + 1)):
                        return
                    yield ("read", f"S{x}", ("S", x, gb))
                    yield ("write", f"S{x}", ("P", x, gb))  # P over the S columns
                    if j > 0:
                        # (implied by S_FULL(j): QK(j) of this tile was issued
                        # after PV(j-1); the kernel waits all the same)
                        if not (yield ("await", f"PVDONE{x}", gb)):
                            return
                        yield ("read", f"O{x}", ("O", x, i, j - 1))
                        yield ("write", f"O{x}", ("Ors", x, i, j - 1))  # rescale
                    yield ("arrive", f"PFULL{x}")
                    gb += 1
                if not (yield ("await", f"PVDONE{x}", gb)):
                    return
                yield ("read", f"O{x}", ("O", x, i, n - 1))
                yield ("arrive", f"OEMPTY{x}")
        return role()

    roles = {"producer": producer(), "vloader": vloader(), "rope": rope(), "mma": mma(),
             "softmaxA": softmax(0), "softmaxB": softmax(1)}
    return roles, {EXIT_CHECK: True}


def band_roles(lanes, skip=(), nseg=9, R=12, stall=False):
    """sinkattn_band_kernel (SWA prefill) for one CTA whose contiguous range of
    tiles crosses `lanes`: (first tile index, number of tiles) per (sequence,
    KV head) lane.  A tile of 16 tokens sees the nwin = min(i + 1, nseg)
    16-key segments ending at its own; a tile that starts a run (the CTA's
    first, or the first of a lane) loads its whole window into the 12-slot
    segment ring, any other tile loads one new segment.  The MMA thread issues
    PV of the previous tile after this tile's QK^T (before it at a run start,
    which reloads the ring) and frees the segments leaving the window.  The two
    threads of a softmax row (modelled as two roles, one per half) swap partial
    maxima and sums through shared memory, paired by a barrier per parity.
    Every wait is bounded ("await"): a role whose wait returns False (the CTA
    is aborting) leaves its loop, and the copy and MMA threads then drain what
    they issued (the last copy into each Q stage and segment slot; a commit
    behind every MMA), as the kernel does before its final barrier.  With
    `stall`, the MMA thread first waits on a barrier nothing completes (the
    test build's stall), which can only end by running out."""
    tiles = []  # (tile index within its lane, run)
    for i0, n in lanes:
        for k in range(n):
            tiles.append((i0 + k, k == 0))

    def nwin_of(i):
        return min(i + 1, nseg)

    def producer():
        gq = gseg = 0
        ok = True
        for t, (i, run) in enumerate(tiles):
            qs = t & 1
            ok = yield ("await", f"QEMPTY{qs}", t >> 1)
            if not ok:
                break
            yield ("tma", f"Q{qs}", ("Qraw", t), f"QFULL{qs}")
            gq += 1
            for _ in range(nwin_of(i) if run else 1):
                slot = gseg % R
                if "producer_segempty" not in skip:
                    ok = yield ("await", f"SEGEMPTY{slot}", gseg // R)
                    if not ok:
                        break
                yield ("tma", f"SEG{slot}", ("Kraw", gseg), f"SEGFULL{slot}")
                gseg += 1
            if not ok:
                break
        # drain: the last copy into each stage and slot lands before the exit
        if "producer_drain" not in skip:
            for st in range(2):
                if gq > st:
                    yield ("drain", f"QFULL{st}", (gq - 1 - st) // 2 + 1)
            for st in range(R):
                if gseg > st:
                    yield ("drain", f"SEGFULL{st}", (gseg - 1 - st) // R + 1)

    def rope():
        gseg = 0
        for t, (i, run) in enumerate(tiles):
            qs = t & 1
            if not (yield ("await", f"QFULL{qs}", (t >> 1) + 1)):
                return
            yield ("read", f"Q{qs}", ("Qraw", t))
            yield ("write", f"Q{qs}", ("Q", t))
            yield ("arrive", f"QREADY{qs}")
            for _ in range(nwin_of(i) if run else 1):
                slot = gseg % R
                if not (yield ("await", f"SEGFULL{slot}", gseg // R + 1)):
                    return
                yield ("read", f"SEG{slot}", ("Kraw", gseg))
                yield ("write", f"SEG{slot}", ("KV", gseg))
                yield ("arrive", f"SEGREADY{slot}")
                gseg += 1

    def mma():
        gseg = 0
        prev = None  # (tile, nwin, first segment) of the tile whose PV is pending
        issued = False

        def issue_pv(t, nwin, seg0, nfree):
            b = t & 1
            if not (yield ("await", f"PFULL{b}", (t >> 1) + 1)):
                return False
            if "mma_oempty" not in skip:
                if not (yield ("await", "OEMPTY", t)):
                    return False
            reads = [(f"S{b}h0", ("P", t)), (f"S{b}h1", ("P", t))]
            reads += [(f"SEG{(seg0 + k) % R}", ("KV", seg0 + k)) for k in range(nwin)]
            yield ("mma", reads, [("Oh0", ("O", t)), ("Oh1", ("O", t))])
            for k in range(nfree):
                yield ("commit", f"SEGEMPTY{(seg0 + k) % R}")
            yield ("commit", "PVDONE")
            return True

        ok = True
        if stall:
            ok = yield ("await", "STALL", 1)
        for t, (i, run) in enumerate(tiles if ok else ()):
            nwin = nwin_of(i)
            nload = nwin if run else 1
            if prev is not None and run:
                ok = yield from issue_pv(*prev, prev[1])  # the reload needs the whole ring back
                if not ok:
                    break
            qs = t & 1
            ok = yield ("await", f"QREADY{qs}", (t >> 1) + 1)
            for j in range(nload):
                if not ok:
                    break
                g = gseg + j
                ok = yield ("await", f"SEGREADY{g % R}", g // R + 1)
            if not ok:
                break
            gseg += nload
            seg0 = gseg - nwin
            b = t & 1
            reads = [(f"Q{qs}", ("Q", t))] + [(f"SEG{(seg0 + k) % R}", ("KV", seg0 + k))
                                              for k in range(nwin)]
            yield ("mma", reads, [(f"S{b}h0", ("S", t)), (f"S{b}h1", ("S", t))])
            issued = True
            yield ("commit", f"SFULL{b}")
            yield ("commit", f"QEMPTY{qs}")
            if prev is not None and not run:
                ok = yield from issue_pv(*prev, 1 if nwin == prev[1] else 0)
                if not ok:
                    break
            prev = (t, nwin, seg0)
        if ok and prev is not None:
            yield from issue_pv(*prev, prev[1])
        # drain: every MMA done before TMEM goes back
        if issued and "mma_drain" not in skip:
            yield ("commit", "DRAIN")
            yield ("drain", "DRAIN", 1)

    def softmax(h):
        def role():
            for step in range(len(tiles) + 1):
                have = step < len(tiles)
                b = step & 1
                if have:
                    if not (yield ("await", f"SFULL{b}", (step >> 1) + 1)):
                        return
                    yield ("read", f"S{b}h{h}", ("S", step))
                par = step & 1  # swap with the other half of the row
                yield ("write", f"X{par}h{h}", ("X", step))
                yield ("arrive", f"PAIR{par}")
                if "softmax_pair" not in skip:
                    if not (yield ("await", f"PAIR{par}", (step >> 1) + 1)):
                        return
                yield ("read", f"X{par}h{1 - h}", ("X", step))
                if have:
                    yield ("write", f"S{b}h{h}", ("P", step))  # P over this half's S columns
                    yield ("arrive", f"PFULL{b}")
                if step > 0:
                    if not (yield ("await", "PVDONE", step)):
                        return
                    yield ("read", f"Oh{h}", ("O", step - 1))
                    yield ("arrive", "OEMPTY")
        return role()

    roles = {"producer": producer(), "rope": rope(), "mma": mma(), "half0": softmax(0),
             "half1": softmax(1)}
    counts = {"PFULL0": 2, "PFULL1": 2, "OEMPTY": 2, "PAIR0": 2, "PAIR1": 2,
              EXIT_CHECK: True}
    return roles, counts
