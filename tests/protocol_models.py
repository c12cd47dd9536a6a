"""Executable models of the mbarrier protocols of the tensor-core kernels.

Each model replays, for one CTA, the sequence of barrier waits, arrivals and
tensor-core commits of every role of a kernel (producer, MMA issuers,
compute warps) as Python generators, and a scheduler runs them in random
interleavings with asynchronous completions: TMA loads complete in any
order, the commits of one issuing thread in issue order. The run fails on

* a deadlock (no role can move and nothing is in flight),
* parity aliasing: a waiter two phases behind its barrier, or one that
  starts waiting for a phase two ahead of it (a parity wait cannot tell
  either apart from the phase it wants),
* a hazard: a stage reloaded while a role still reads it, a tensor-memory
  buffer or accumulator set written while another role reads or writes it.

The models follow the kernels' source (``fwd_tc16_kernel``,
``bwd_tc_kernel``, ``fwd_bf16_kernel``, ``fwd_tc_kernel``, ``wide_tc_kernel``
forward and backward, ``wide_tc_dw_kernel``, ``bwd_bf16_tc_kernel``): the same
item order, barrier counts, ring sizes and wait parities. ``mutation`` plants
a protocol mistake (a dropped wait, an early release) so that the tests can
check the checker. Where a kernel's compute warps arrive one per warp, the
model's single compute role arrives once on a barrier of count 1.
"""
import random

kRowItem = 16
kBwdSampleItem = 8
kChunkRing = 6
kLoBufs = 3


class Bar:
    """An mbarrier: ``count`` arrivals complete a phase."""

    def __init__(self, name, count):
        self.name, self.count, self.pending, self.completed = name, count, count, 0

    def arrive(self, n=1):
        self.pending -= n
        assert self.pending >= 0, ("over-arrival", self.name)
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count


def W(name, n):
    """Wait for phase n of a barrier (the kernels wait with parity n & 1)."""
    return ("wait", name, n)


def schedule(actors, bars, events, seed, limit=10 ** 6):
    """Run the role generators to completion in a random interleaving."""
    rnd = random.Random(seed)
    blocked = {k: None for k in actors}
    done = set()
    for _ in range(limit):
        if len(done) == len(actors):
            break
        runnable = []
        for k in actors:
            if k in done:
                continue
            w = blocked[k]
            if w is None or w[0] == "yield":
                runnable.append(k)
            else:
                b = bars[w[1]]
                assert b.completed <= w[2] + 1, ("parity aliasing", k, w, b.completed)
                if b.completed >= w[2] + 1:
                    runnable.append(k)
        queues = [q for q in events if events[q]]
        if queues and (not runnable or rnd.random() < 0.5):
            q = rnd.choice(queues)
            name, cb = events[q].pop(rnd.randrange(len(events[q])) if q == "tma" else 0)
            if cb:
                cb()
            bars[name].arrive()
            continue
        if not runnable:
            raise RuntimeError("deadlock: %s" % {k: blocked[k] for k in actors if k not in done})
        k = rnd.choice(runnable)
        blocked[k] = None
        try:
            blocked[k] = next(actors[k])
        except StopIteration:
            done.add(k)
            continue
        w = blocked[k]
        if w[0] == "wait":
            # a parity wait for phase n also passes while the barrier has
            # completed only n - 1 phases: a waiter may start at most one
            # phase ahead of the barrier
            assert bars[w[1]].completed >= w[2], ("parity aliasing ahead", k, w, bars[w[1]].completed)
    else:
        raise RuntimeError("no progress within the step limit")
    assert not any(events.values()), "completions left over"


def tiles(B, P, cta, K, S_max=None):
    """Sample counts of the CTA's tiles (the kernels' balanced split)."""
    if S_max is None:
        S_max = min(128 // K, 16)
    cb0 = B * cta // P
    n_c = B * (cta + 1) // P - cb0
    T = (n_c + S_max - 1) // S_max
    if T == 0:
        return []
    t_base, t_extra = n_c // T, n_c - (n_c // T) * T
    ts = lambda i: cb0 + i * t_base + min(i, t_extra)
    return [ts(i + 1) - ts(i) for i in range(T)]


def post_item(p, NSI, NRI):
    """The backward's item order after a tile's chunks: sample item 0, row
    items 0-3, the other sample items, the other row items."""
    if NSI > 0:
        if p == 0:
            return 1, 0
        p -= 1
    r1 = min(NRI, 4)
    if p < r1:
        return 2, p
    p -= r1
    s1 = NSI - 1 if NSI > 0 else 0
    if p < s1:
        return 1, 1 + p
    return 2, 4 + (p - s1)


# --------------------------------------------------------------- forward

def fwd_tc16(B, P, cta, K, SH2, NST, seed, mutation=None):
    """fwd_tc16_kernel: producer rounds (tile u's chunks, then tile u-1's h_s2
    rows), a main and a remainder MMA thread, the compute warps. A chunk
    signals full[s], a row item fullo[s]: the main MMA thread skips the row
    items, and with one barrier for both its parity waits could start two
    phases ahead."""
    S = tiles(B, P, cta, K)
    T, NC = len(S), SH2 // 32
    bars = {}
    for s in range(NST):
        bars["full%d" % s] = Bar("full", 1)
        bars["fullo%d" % s] = Bar("fullo", 1)
        bars["empty%d" % s] = Bar("empty", 2)
        bars["outdone%d" % s] = Bar("outdone", 1)
    for s in range(kChunkRing):
        bars["loready%d" % s] = Bar("loready", 1)
    for s in range(kLoBufs):
        bars["lofree%d" % s] = Bar("lofree", 1)
    for s in range(2):
        bars["mdone%d" % s] = Bar("mdone", 1)
        bars["accempty%d" % s] = Bar("accempty", 1)
    events = {"tma": [], "main": [], "corr": []}
    st_read = [set() for _ in range(NST)]
    lo_read = [0] * kLoBufs
    acc_w, acc_r = [0, 0], [None, None]
    rounds = lambda u: (NC if u < T else 0) + (1 if u >= 1 else 0)
    items = []
    for u in range(T + 1):
        items += ["chunk"] * (NC if u < T else 0) + (["out"] if u >= 1 else [])

    def producer():
        use = {"empty": [0] * NST, "outdone": [0] * NST}
        for pn in range(len(items)):
            if pn >= NST:
                rn = pn - NST
                b = "empty" if items[rn] == "chunk" else "outdone"
                st = rn % NST
                yield W("%s%d" % (b, st), use[b][st])
                use[b][st] += 1
            st = pn % NST
            assert not st_read[st], ("stage reloaded while read", st)
            one = mutation == "one_full_barrier"
            events["tma"].append((("full%d" if items[pn] == "chunk" or one else "fullo%d") % st, None))

    def main():
        tp = 0
        fuse = [0] * NST
        for t in range(T):
            if t >= 2 and mutation != "no_accempty_wait":
                yield W("accempty%d" % (t & 1), (t - 2) >> 1)
            assert acc_r[t & 1] is None, "main products into a set being read"
            for q in range(NC):
                it = tp + q
                st = it % NST
                yield W("full%d" % st, it // NST if mutation == "one_full_barrier" else fuse[st])
                fuse[st] += 1
                st_read[st].add(("m", it))
                acc_w[t & 1] += 1

                def done(st=st, it=it, s=t & 1):
                    st_read[st].discard(("m", it))
                    acc_w[s] -= 1
                events["main"].append(("empty%d" % st, done))
            events["main"].append(("mdone%d" % (t & 1), None))
            tp += rounds(t)

    def corr():
        tp = c = 0
        for t in range(T):
            if t >= 2:
                yield W("accempty%d" % (t & 1), (t - 2) >> 1)
            for q in range(NC):
                yield W("loready%d" % (c % kChunkRing), c // kChunkRing)
                assert acc_r[t & 1] is None, "remainder products into a set being read"
                bars["empty%d" % ((tp + q) % NST)].arrive()
                b = c % kLoBufs
                lo_read[b] += 1
                acc_w[t & 1] += 1

                def done(b=b, s=t & 1):
                    lo_read[b] -= 1
                    acc_w[s] -= 1
                events["corr"].append(("lofree%d" % b, done))
                c += 1
            tp += rounds(t)

    def compute():
        seq = c = 0
        one = mutation == "one_full_barrier"
        cuse, ouse = [0] * NST, [0] * NST

        def wait_item(kind, st):
            if one:
                return W("full%d" % st, seq // NST)
            u = cuse if kind == "chunk" else ouse
            u[st] += 1
            return W(("full%d" if kind == "chunk" else "fullo%d") % st, u[st] - 1)
        for t in range(T):
            for q in range(NC):
                st = seq % NST
                yield wait_item("chunk", st)
                st_read[st].add(("c", seq))
                if q > 0:
                    bars["loready%d" % ((c - 1) % kChunkRing)].arrive()
                    st_read[(seq - 1) % NST].discard(("c", seq - 1))
                if c >= kLoBufs and mutation != "no_lofree_wait":
                    yield W("lofree%d" % (c % kLoBufs), c // kLoBufs - 1)
                assert lo_read[c % kLoBufs] == 0, "remainder buffer written while read"
                seq += 1
                c += 1
            bars["loready%d" % ((c - 1) % kChunkRing)].arrive()
            st_read[(seq - 1) % NST].discard(("c", seq - 1))
            if t >= 1:
                st = seq % NST
                yield wait_item("out", st)
                st_read[st].add(("o", seq))
                yield ("yield",)
                st_read[st].discard(("o", seq))
                bars["outdone%d" % st].arrive()
                seq += 1
            yield W("mdone%d" % (t & 1), t >> 1)
            if mutation != "no_last_lofree_wait":
                yield W("lofree%d" % ((c - 1) % kLoBufs), (c - 1) // kLoBufs)
            assert acc_w[t & 1] == 0, "projections read while written"
            acc_r[t & 1] = t
            yield ("yield",)
            acc_r[t & 1] = None
            bars["accempty%d" % (t & 1)].arrive()
        if T:
            st = seq % NST
            yield wait_item("out", st)
            bars["outdone%d" % st].arrive()

    schedule({"p": producer(), "m": main(), "r": corr(), "c": compute()}, bars, events, seed)


def fwd_bf16(B, P, cta, K, SH2, NST, seed, mutation=None):
    """fwd_bf16_kernel: the same rounds with 64-column chunks and one MMA
    thread; a chunk stage is freed by the MMA commit and the compute warps.
    As in fwd_tc16, chunks signal full[s] and row items fullo[s]."""
    S = tiles(B, P, cta, K)
    T, NC = len(S), SH2 // 64
    bars = {}
    for s in range(NST):
        bars["full%d" % s] = Bar("full", 1)
        bars["fullo%d" % s] = Bar("fullo", 1)
        bars["empty%d" % s] = Bar("empty", 2)
        bars["outdone%d" % s] = Bar("outdone", 1)
    for s in range(2):
        bars["mdone%d" % s] = Bar("mdone", 1)
        bars["accempty%d" % s] = Bar("accempty", 1)
    events = {"tma": [], "mma": []}
    st_read = [set() for _ in range(NST)]
    acc_w, acc_r = [0, 0], [None, None]
    rounds = lambda u: (NC if u < T else 0) + (1 if u >= 1 else 0)
    items = []
    for u in range(T + 1):
        items += ["chunk"] * (NC if u < T else 0) + (["out"] if u >= 1 else [])

    def producer():
        use = {"empty": [0] * NST, "outdone": [0] * NST}
        for pn in range(len(items)):
            if pn >= NST:
                rn = pn - NST
                b = "empty" if items[rn] == "chunk" else "outdone"
                st = rn % NST
                yield W("%s%d" % (b, st), use[b][st])
                use[b][st] += 1
            st = pn % NST
            assert not st_read[st], ("stage reloaded while read", st)
            one = mutation == "one_full_barrier"
            events["tma"].append((("full%d" if items[pn] == "chunk" or one else "fullo%d") % st, None))

    def mma():
        tp = 0
        fuse = [0] * NST
        for t in range(T):
            if t >= 2 and mutation != "no_accempty_wait":
                yield W("accempty%d" % (t & 1), (t - 2) >> 1)
            assert acc_r[t & 1] is None, "products into a set being read"
            for q in range(NC):
                it = tp + q
                st = it % NST
                yield W("full%d" % st, it // NST if mutation == "one_full_barrier" else fuse[st])
                fuse[st] += 1
                st_read[st].add(("m", it))
                acc_w[t & 1] += 1

                def done(st=st, it=it, s=t & 1):
                    st_read[st].discard(("m", it))
                    acc_w[s] -= 1
                events["mma"].append(("empty%d" % st, done))
            events["mma"].append(("mdone%d" % (t & 1), None))
            tp += rounds(t)

    def compute():
        seq = 0
        one = mutation == "one_full_barrier"
        cuse, ouse = [0] * NST, [0] * NST

        def wait_item(kind, st):
            if one:
                return W("full%d" % st, seq // NST)
            u = cuse if kind == "chunk" else ouse
            u[st] += 1
            return W(("full%d" if kind == "chunk" else "fullo%d") % st, u[st] - 1)
        for t in range(T):
            for q in range(NC):
                st = seq % NST
                yield wait_item("chunk", st)
                if mutation == "early_empty":
                    bars["empty%d" % st].arrive()
                st_read[st].add(("c", seq))
                yield ("yield",)
                st_read[st].discard(("c", seq))
                if mutation != "early_empty":
                    bars["empty%d" % st].arrive()
                seq += 1
            if t >= 1:
                st = seq % NST
                yield wait_item("out", st)
                st_read[st].add(("o", seq))
                yield ("yield",)
                st_read[st].discard(("o", seq))
                bars["outdone%d" % st].arrive()
                seq += 1
            if mutation != "no_mdone_wait":
                yield W("mdone%d" % (t & 1), t >> 1)
            assert acc_w[t & 1] == 0, "projections read while written"
            acc_r[t & 1] = t
            yield ("yield",)
            acc_r[t & 1] = None
            bars["accempty%d" % (t & 1)].arrive()
        if T:
            st = seq % NST
            yield wait_item("out", st)
            bars["outdone%d" % st].arrive()

    schedule({"p": producer(), "m": mma(), "c": compute()}, bars, events, seed)


def fwd_tc(B, P, cta, K, SH2, NST, seed, mutation=None, D=8):
    """fwd_tc_kernel (D = 8 and 16 with the plain tf32 split): per tile the
    NC chunks, then one item of h_s2 rows; the compute warps split each chunk
    into one of two TMEM A buffers and free the stage themselves (the MMA
    thread reads only TMEM and the weights); one accumulator set. The MMA
    thread's wait on accempty is implied by the compute order (the next
    tile's first A buffer is handed over after the read-back), so dropping
    it is not a mistake this model can show."""
    S_max = min(128 // K, 32, 256 // D)
    S = tiles(B, P, cta, K, S_max)
    T, NC = len(S), SH2 // 32
    bars = {}
    for s in range(NST):
        bars["full%d" % s] = Bar("full", 1)
        bars["empty%d" % s] = Bar("empty", 1)
    for s in range(2):
        bars["aready%d" % s] = Bar("aready", 1)
        bars["afree%d" % s] = Bar("afree", 1)
    bars["accfull"] = Bar("accfull", 1)
    bars["accempty"] = Bar("accempty", 1)
    events = {"tma": [], "mma": []}
    st_read = [set() for _ in range(NST)]
    a_read = [0, 0]
    acc = {"w": 0, "r": False}
    n_items = T * (NC + 1)

    def producer():
        for pn in range(n_items):
            st, use = pn % NST, pn // NST
            if use > 0:
                yield W("empty%d" % st, use - 1)
            assert not st_read[st], ("stage reloaded while read", st)
            events["tma"].append(("full%d" % st, None))

    def mma():
        c = 0
        for t in range(T):
            if t > 0:
                yield W("accempty", t - 1)
            assert not acc["r"], "products into accumulators being read"
            for q in range(NC):
                yield W("aready%d" % (c & 1), c >> 1)
                a_read[c & 1] += 1
                acc["w"] += 1

                def done(b=c & 1):
                    a_read[b] -= 1
                    acc["w"] -= 1
                events["mma"].append(("afree%d" % (c & 1), done))
                c += 1
            events["mma"].append(("accfull", None))

    def compute():
        seq = c = 0
        for t in range(T):
            for q in range(NC):
                st = seq % NST
                yield W("full%d" % st, seq // NST)
                if mutation == "early_empty":
                    bars["empty%d" % st].arrive()
                st_read[st].add(seq)
                if c >= 2 and mutation != "no_afree_wait":
                    yield W("afree%d" % (c & 1), (c - 2) >> 1)
                assert a_read[c & 1] == 0, "A buffer written while read"
                yield ("yield",)
                st_read[st].discard(seq)
                bars["aready%d" % (c & 1)].arrive()
                if mutation != "early_empty":
                    bars["empty%d" % st].arrive()
                seq += 1
                c += 1
            if mutation != "no_accfull_wait":
                yield W("accfull", t)
            assert acc["w"] == 0, "accumulators read while written"
            acc["r"] = True
            yield ("yield",)
            acc["r"] = False
            bars["accempty"].arrive()
            st = seq % NST
            yield W("full%d" % st, seq // NST)
            st_read[st].add(seq)
            yield ("yield",)
            st_read[st].discard(seq)
            bars["empty%d" % st].arrive()
            seq += 1

    schedule({"p": producer(), "m": mma(), "c": compute()}, bars, events, seed)


# -------------------------------------------------------------- backward

def bwd_tc(B, P, cta, K, SH2, NST, seed, mutation=None):
    """bwd_tc_kernel: producer (chunks, then sample and row items; it stores
    an item's outputs before reusing its stage), the main MMA thread (main
    projection products, d_h halves, dW per row item), the remainder MMA
    thread, the compute warps."""
    S = tiles(B, P, cta, K)
    if not S:
        return
    NC = SH2 // 32
    NSI = lambda s: (s + kBwdSampleItem - 1) // kBwdSampleItem
    NRI = lambda s: (s * K + kRowItem - 1) // kRowItem
    bars = {}
    for s in range(NST):
        bars["full%d" % s] = Bar("full", 1)
        bars["empty%d" % s] = Bar("empty", 1)
        bars["cempty%d" % s] = Bar("cempty", 2)
    for s in range(kChunkRing):
        bars["loready%d" % s] = Bar("loready", 1)
    for s in range(kLoBufs):
        bars["lofree%d" % s] = Bar("lofree", 1)
    for s in range(2):
        for n in ("dhready", "dhfree", "htready", "htfree"):
            bars["%s%d" % (n, s)] = Bar(n, 1)
    for n in ("bready", "dwdone", "mdone"):
        bars[n] = Bar(n, 1)
    events = {"tma": [], "main": [], "corr": []}
    fl = {"main": 0, "corr": 0, "dh": 0, "dw": [0, 0], "lo": [0] * kLoBufs}
    st_read = [set() for _ in range(NST)]
    reading = {"P": False, "L": False}
    kinds = []
    for s in S:
        kinds += ["chunk"] * NC + ["item"] * (NSI(s) + NRI(s))

    def producer():
        use = {"cempty": [0] * NST, "empty": [0] * NST}
        for pn in range(len(kinds)):
            if pn >= NST:
                rn = pn - NST
                b = "cempty" if kinds[rn] == "chunk" else "empty"
                st = rn % NST
                yield W("%s%d" % (b, st), use[b][st])
                use[b][st] += 1
            st = pn % NST
            assert not st_read[st], ("stage reloaded while read", st)
            events["tma"].append(("full%d" % st, None))

    def main():
        seq = ri = 0
        for t, s in enumerate(S):
            nsi, nri = NSI(s), NRI(s)
            if t > 0 and mutation != "no_dhfree1_wait":
                yield W("dhfree1", t - 1)
            for q in range(NC):
                it = seq + q
                st = it % NST
                yield W("full%d" % st, it // NST)
                # d_h of the previous tile may still run: same thread, in order
                assert not reading["P"], "main products over P in use"
                st_read[st].add(("m", it))
                fl["main"] += 1

                def done(st=st, it=it):
                    st_read[st].discard(("m", it))
                    fl["main"] -= 1
                events["main"].append(("cempty%d" % st, done))
            events["main"].append(("mdone", None))
            seq += NC + nsi + nri
            yield W("bready", t)

            def dh():
                assert not reading["P"], "d_h over P in use"
                fl["dh"] += 1

                def done():
                    fl["dh"] -= 1
                return done
            events["main"].append(("dhready0", dh()))
            for k in range(nri):
                if k == 4:
                    yield W("dhfree0", t)
                    events["main"].append(("dhready1", dh()))
                yield W("htready%d" % (ri & 1), ri >> 1)
                p = ri & 1
                fl["dw"][p] += 1

                def done(p=p):
                    fl["dw"][p] -= 1
                events["main"].append(("htfree%d" % p, done))
                ri += 1
            if nri <= 4:
                yield W("dhfree0", t)
                events["main"].append(("dhready1", dh()))
        events["main"].append(("dwdone", None))

    def corr():
        seq = c = 0
        for s in S:
            for q in range(NC):
                yield W("loready%d" % (c % kChunkRing), c // kChunkRing)
                assert fl["dw"] == [0, 0] and not reading["L"], "remainder products over L in use"
                bars["cempty%d" % ((seq + q) % NST)].arrive()
                b = c % kLoBufs
                fl["lo"][b] += 1
                fl["corr"] += 1

                def done(b=b):
                    fl["lo"][b] -= 1
                    fl["corr"] -= 1
                events["corr"].append(("lofree%d" % b, done))
                c += 1
            seq += NC + NSI(s) + NRI(s)

    def compute():
        seq = c = ri = 0
        for t, s in enumerate(S):
            nsi, nri = NSI(s), NRI(s)
            if mutation != "no_htfree_wait":
                if ri >= 1:
                    yield W("htfree%d" % ((ri - 1) & 1), (ri - 1) >> 1)
                if ri >= 2:
                    yield W("htfree%d" % (ri & 1), (ri - 2) >> 1)
            for q in range(NC):
                st = seq % NST
                yield W("full%d" % st, seq // NST)
                st_read[st].add(("c", seq))
                if q > 0:
                    bars["loready%d" % ((c - 1) % kChunkRing)].arrive()
                    st_read[(seq - 1) % NST].discard(("c", seq - 1))
                if c >= kLoBufs:
                    yield W("lofree%d" % (c % kLoBufs), c // kLoBufs - 1)
                assert fl["lo"][c % kLoBufs] == 0 and fl["dw"] == [0, 0], \
                    "remainder written over L in use"
                seq += 1
                c += 1
            bars["loready%d" % ((c - 1) % kChunkRing)].arrive()
            st_read[(seq - 1) % NST].discard(("c", seq - 1))
            yield W("mdone", t)
            yield W("lofree%d" % ((c - 1) % kLoBufs), (c - 1) // kLoBufs)
            assert fl["main"] == 0 and fl["corr"] == 0 and fl["dh"] == 0, "projections read early"
            reading["P"] = reading["L"] = True
            yield ("yield",)
            reading["P"] = reading["L"] = False
            bars["bready"].arrive()
            for p in range(nsi + nri):
                kind, k = post_item(p, nsi, nri)
                st = seq % NST
                yield W("full%d" % st, seq // NST)
                if kind == 1:
                    bars["empty%d" % st].arrive()
                    seq += 1
                    continue
                if ri >= 2:
                    yield W("htfree%d" % (ri & 1), (ri - 2) >> 1)
                assert fl["dw"][ri & 1] == 0 and fl["corr"] == 0, "transposed rows over L in use"
                bars["htready%d" % (ri & 1)].arrive()
                rh = k >> 2
                if mutation == "early_row_empty":
                    bars["empty%d" % st].arrive()
                    st_read[st].add(("r", seq))
                    yield ("yield",)
                if (k & 3) == 0:
                    yield W("dhready%d" % rh, t)
                    assert fl["dh"] == 0 and fl["main"] == 0, "d_h read early"
                    reading["P"] = True
                assert fl["main"] == 0, "d_h overwritten while read"
                yield ("yield",)  # the item's d_h rows read back
                assert fl["main"] == 0, "d_h overwritten while read"
                if (k & 3) == 3 or k == nri - 1:
                    reading["P"] = False
                    bars["dhfree%d" % rh].arrive()
                if mutation == "early_row_empty":
                    st_read[st].discard(("r", seq))
                else:
                    bars["empty%d" % st].arrive()
                seq += 1
                ri += 1
            if nri <= 4:
                bars["dhfree1"].arrive()
        yield W("dwdone", 0)

    schedule({"p": producer(), "m": main(), "r": corr(), "c": compute()}, bars, events, seed)


# ------------------------------------------------- wide-state tile kernels

class Tmem:
    """Tensor-memory regions of 128 columns: MMA writers and readers in flight,
    compute readers and writers, checked against each other."""

    def __init__(self, n):
        self.mw, self.mr = [0] * n, [0] * n
        self.cr, self.cw = [0] * n, [0] * n

    def mma(self, writes, reads, what):
        for r in writes:
            assert self.cr[r] == 0 and self.cw[r] == 0, ("%s writes a region compute uses" % what, r)
        for r in reads:
            assert self.cw[r] == 0, ("%s reads a region compute writes" % what, r)
        for r in writes:
            self.mw[r] += 1
        for r in reads:
            self.mr[r] += 1

        def done():
            for r in writes:
                self.mw[r] -= 1
            for r in reads:
                self.mr[r] -= 1
        return done

    def compute(self, regions, write, what):
        for r in regions:
            assert self.mw[r] == 0, ("%s while the MMA writes it" % what, r)
            if write:
                assert self.mr[r] == 0, ("%s while the MMA reads it" % what, r)
        for r in regions:
            (self.cw if write else self.cr)[r] += 1

    def release(self, regions, write):
        for r in regions:
            (self.cw if write else self.cr)[r] -= 1


def wide_tiles(B, P, cta, K):
    """Tiles of the wide-state tile kernels: 128-row tiles of S_max samples
    handed out round-robin over min(n_tiles, P) CTAs."""
    S_max = min(128 // K, 16)
    n_tiles = -(-B // S_max)
    grid = min(n_tiles, P)
    if cta >= grid:
        return []
    return [min(S_max, B - t * S_max) for t in range(cta, n_tiles, grid)]


def wide_tc(B, P, cta, K, SH2, NST, seed, mutation=None, bwd=False):
    """wide_tc_kernel: per tile NQ = SH2/32 chunk stages (backward: then 2 NB
    stages of d_h weight tiles), a producer, one MMA thread, the compute warps
    and (backward) the loader of the split weights' remainders. Remainder buffer cq & 1 (shared with the A|B buffer); projections
    into TMEM regions 0-3 (chunk q into q mod 4); backward: d_h blocks into
    regions 0 and 1 in turn, dA|dB in regions 2 and 3."""
    S = wide_tiles(B, P, cta, K)
    T, NQ, NB = len(S), SH2 // 32, SH2 // 128
    bars = {"acc_full": Bar("acc_full", 1), "acc_free": Bar("acc_free", 1),
            "dab_ready": Bar("dab_ready", 1)}
    for s in range(NST):
        bars["full%d" % s] = Bar("full", 1)
        bars["empty%d" % s] = Bar("empty", 1)
        bars["split%d" % s] = Bar("split", 1)
    for b in range(2):
        bars["dh_full%d" % b] = Bar("dh_full", 1)
        bars["dh_free%d" % b] = Bar("dh_free", 1)
        bars["wlo_full%d" % b] = Bar("wlo_full", 1)
    bars["tile_done"] = Bar("tile_done", 1)
    events = {"tma": [], "mma": []}
    st_read = [set() for _ in range(NST)]
    lo_read, lo_write, ab_use = [0, 0], [0, 0], [0]
    wlo_pending = [0, 0]  # backward: W remainder copies in flight into buffer p
    tm = Tmem(4)
    per_tile = NQ + (2 * NB if bwd else 0)

    def producer():
        for pn in range(T * per_tile):
            st = pn % NST
            if pn >= NST:
                yield W("empty%d" % st, pn // NST - 1)
            assert not st_read[st], ("stage reloaded while read", st)
            events["tma"].append(("full%d" % st, None))

    def wlo_loader():
        # backward: the weights come split from the workspace; a chunk's W
        # remainders are copied into remainder buffer cq & 1 once the products
        # of stage use cq - 2 are done: for the first two chunks of a tile the
        # previous tile's products (tile_done), for the others chunk cq - 2.
        # "skip_dh_waits" is the form that waits on stage cq - 2 even across
        # the d_h stages it skips.
        cq = 0
        for t in range(T):
            if t > 0 and mutation not in ("no_wlo_free_wait", "skip_dh_waits"):
                yield W("tile_done", t - 1)
            for q in range(NQ):
                if mutation == "skip_dh_waits":
                    if cq >= 2:
                        yield W("empty%d" % ((cq - 2) % NST), (cq - 2) // NST)
                elif q >= 2 and mutation != "no_wlo_free_wait":
                    yield W("empty%d" % ((cq - 2) % NST), (cq - 2) // NST)
                p = cq & 1
                assert lo_read[p] == 0 and ab_use[0] == 0, "W remainder copied while the buffer is read"
                wlo_pending[p] += 1

                def landed(p=p):
                    wlo_pending[p] -= 1
                events["tma"].append(("wlo_full%d" % p, landed))
                cq += 1
            cq += 2 * NB

    def mma():
        cq = 0
        uses = [0, 0]
        wlo = [0, 0]
        for t in range(T):
            if bwd:
                if mutation != "no_dh_free_wait":
                    for b in range(2):
                        if uses[b]:
                            yield W("dh_free%d" % b, uses[b] - 1)
            elif t > 0 and mutation != "no_acc_free_wait":
                yield W("acc_free", t - 1)
            for q in range(NQ):
                st = cq % NST
                yield W("full%d" % st, cq // NST)
                yield W("split%d" % st, cq // NST)
                if bwd:
                    if mutation != "no_wlo_wait":
                        yield W("wlo_full%d" % (cq & 1), wlo[cq & 1])
                    wlo[cq & 1] += 1
                    assert wlo_pending[cq & 1] == 0, "W remainder read before it landed"
                assert lo_write[cq & 1] == 0 and ab_use[0] == 0, "remainder buffer read while written"
                st_read[st].add(("m", cq))
                lo_read[cq & 1] += 1
                fin = tm.mma([q & 3], [], "projection")

                def done(st=st, cq=cq, fin=fin):
                    st_read[st].discard(("m", cq))
                    lo_read[cq & 1] -= 1
                    fin()
                events["mma"].append(("empty%d" % st, done))
                cq += 1
            events["mma"].append(("acc_full", None))
            if not bwd:
                continue
            if mutation != "no_dab_ready_wait":
                yield W("dab_ready", t)
            for nb in range(NB):
                b = nb & 1
                if uses[b] and mutation != "no_dh_free_wait":
                    yield W("dh_free%d" % b, uses[b] - 1)
                uses[b] += 1
                for half in range(2):
                    st = cq % NST
                    yield W("full%d" % st, cq // NST)
                    yield W("split%d" % st, cq // NST)
                    assert lo_write[cq & 1] == 0 and ab_use[0] == 0, "remainder buffer read while written"
                    st_read[st].add(("m", cq))
                    lo_read[cq & 1] += 1
                    fin = tm.mma([b], [2, 3], "d_h")

                    def done(st=st, cq=cq, fin=fin):
                        st_read[st].discard(("m", cq))
                        lo_read[cq & 1] -= 1
                        fin()
                    events["mma"].append(("empty%d" % st, done))
                    cq += 1
                events["mma"].append(("dh_full%d" % b, None))
            if t + 1 < T:  # nobody waits for the last tile's: none is issued
                events["mma"].append(("tile_done", None))

    def compute():
        cq = 0
        reads = [0, 0]

        def stage():
            nonlocal cq
            st = cq % NST
            yield W("full%d" % st, cq // NST)
            if cq >= 2 and mutation != "no_lo_wait":
                yield W("empty%d" % ((cq - 2) % NST), (cq - 2) // NST)
            assert lo_read[cq & 1] == 0, "remainder buffer written while read"
            st_read[st].add(("c", cq))
            lo_write[cq & 1] += 1
            if mutation == "early_split":
                bars["split%d" % st].arrive()
            yield ("yield",)
            lo_write[cq & 1] -= 1
            st_read[st].discard(("c", cq))
            if mutation != "early_split":
                bars["split%d" % st].arrive()
            cq += 1

        def readback(nb):
            b = nb & 1
            if mutation != "no_dh_full_wait":
                yield W("dh_full%d" % b, reads[b])
            reads[b] += 1
            tm.compute([b], False, "d_h read back")
            yield ("yield",)
            tm.release([b], False)
            bars["dh_free%d" % b].arrive()

        for t in range(T):
            for q in range(NQ):
                yield from stage()
            if mutation != "no_acc_full_wait":
                yield W("acc_full", t)
            # partial sums of C / d_ctx, then A|B, in the buffer the remainders share
            assert lo_read == [0, 0], "A|B buffer written while remainders are read"
            assert wlo_pending == [0, 0], "A|B buffer written while a W remainder lands"
            ab_use[0] += 1
            tm.compute([0, 1, 2, 3], False, "projections read back")
            yield ("yield",)
            tm.release([0, 1, 2, 3], False)
            if not bwd:
                bars["acc_free"].arrive()
            yield ("yield",)  # scan (and output)
            if bwd:
                tm.compute([2, 3], True, "dA|dB into TMEM")
                yield ("yield",)
                tm.release([2, 3], True)
                bars["dab_ready"].arrive()
                ab_use[0] -= 1
                for nb in range(NB):
                    for half in range(2):
                        yield from stage()
                    if nb >= 1:
                        yield from readback(nb - 1)
                yield from readback(NB - 1)
            else:
                ab_use[0] -= 1

    roles = {"p": producer(), "m": mma(), "c": compute()}
    if bwd:
        roles["w"] = wlo_loader()
    schedule(roles, bars, events, seed)


def wide_tc_bwd(B, P, cta, K, SH2, NST, seed, mutation=None):
    return wide_tc(B, P, cta, K, SH2, NST, seed, mutation, bwd=True)


def wide_tc_dw(B, P, cta, K, SH2, NST, seed, mutation=None):
    """wide_tc_dw_kernel for the range of job (cta mod 3 nb) = dW_A|dW_B: NC
    stages of 32 rows, a producer, one MMA thread, the compute warps (the
    remainders, then the read-back of the accumulators once every product is
    done)."""
    Pr = min(B, 152)
    p = cta % Pr
    rows = (B * (p + 1) // Pr - B * p // Pr) * K
    NC = -(-rows // 32)
    bars = {"done": Bar("done", 1)}
    for s in range(NST):
        bars["full%d" % s] = Bar("full", 1)
        bars["empty%d" % s] = Bar("empty", 1)
        bars["split%d" % s] = Bar("split", 1)
    events = {"tma": [], "mma": []}
    st_read = [set() for _ in range(NST)]
    st_write = [0] * NST
    tm = Tmem(1)

    def producer():
        for c in range(NC):
            st = c % NST
            if c >= NST:
                yield W("empty%d" % st, c // NST - 1)
            assert not st_read[st] and not st_write[st], ("stage reloaded while used", st)
            events["tma"].append(("full%d" % st, None))

    def mma():
        for c in range(NC):
            st = c % NST
            yield W("full%d" % st, c // NST)
            if mutation != "no_split_wait":
                yield W("split%d" % st, c // NST)
            assert st_write[st] == 0, "operands read while their remainders are written"
            st_read[st].add(("m", c))
            fin = tm.mma([0], [], "dW")

            def done(st=st, c=c, fin=fin):
                st_read[st].discard(("m", c))
                fin()
            events["mma"].append(("empty%d" % st, done))
        events["mma"].append(("done", None))

    def compute():
        for c in range(NC):
            st = c % NST
            yield W("full%d" % st, c // NST)
            st_write[st] += 1
            if mutation == "early_split":
                bars["split%d" % st].arrive()
            yield ("yield",)
            st_write[st] -= 1
            if mutation != "early_split":
                bars["split%d" % st].arrive()
        if mutation != "no_done_wait":
            yield W("done", 0)
        tm.compute([0], False, "dW read back")
        yield ("yield",)
        tm.release([0], False)

    schedule({"p": producer(), "m": mma(), "c": compute()}, bars, events, seed)


# --------------------------------------------------- bf16 backward kernel

def bwd_bf16(B, P, cta, K, SH2, NST, seed, mutation=None):
    """bwd_bf16_tc_kernel: per tile NB = SH2/64 pass-1 stages then NB stages of
    the tile's h blocks again; a stage is freed by the MMA commit and the
    compute warps (empty: count 2 here). TMEM region X (projections, then
    d_h) is read back by the compute warps; T (dA|dB parts, shared memory) is
    written by the compute warps and read by the d_h and dW products."""
    S = tiles(B, P, cta, K)
    T_, NB = len(S), SH2 // 64
    bars = {"acc_full": Bar("acc_full", 1), "t_ready": Bar("t_ready", 1),
            "dh_full": Bar("dh_full", 1), "dh_free": Bar("dh_free", 1), "dw_done": Bar("dw_done", 1)}
    for s in range(NST):
        bars["full%d" % s] = Bar("full", 1)
        bars["empty%d" % s] = Bar("empty", 2)
    events = {"tma": [], "mma": []}
    st_read = [set() for _ in range(NST)]
    tm = Tmem(2)  # 0: X (projections, d_h), 1: the dW accumulators
    t_read, t_write = [0], [0]

    def producer():
        for pn in range(T_ * 2 * NB):
            st = pn % NST
            if pn >= NST:
                yield W("empty%d" % st, pn // NST - 1)
            assert not st_read[st], ("stage reloaded while read", st)
            events["tma"].append(("full%d" % st, None))

    def mma():
        n = 0
        for t in range(T_):
            if t > 0 and mutation != "no_dh_free_wait":
                yield W("dh_free", t - 1)
            for q in range(NB):
                st = n % NST
                yield W("full%d" % st, n // NST)
                st_read[st].add(("m", n))
                fin = tm.mma([0], [], "projection")

                def done(st=st, n=n, fin=fin):
                    st_read[st].discard(("m", n))
                    fin()
                events["mma"].append(("empty%d" % st, done))
                n += 1
            events["mma"].append(("acc_full", None))
            if mutation != "no_t_ready_wait":
                yield W("t_ready", t)
            assert t_write[0] == 0, "T read while written"
            t_read[0] += 1
            fin = tm.mma([0], [], "d_h")

            def dh_done(fin=fin):
                t_read[0] -= 1
                fin()
            events["mma"].append(("dh_full", dh_done))
            for q in range(NB):
                st = n % NST
                yield W("full%d" % st, n // NST)
                assert t_write[0] == 0, "T read while written"
                st_read[st].add(("m", n))
                t_read[0] += 1
                fin = tm.mma([1], [], "dW")

                def done(st=st, n=n, fin=fin):
                    st_read[st].discard(("m", n))
                    t_read[0] -= 1
                    fin()
                events["mma"].append(("empty%d" % st, done))
                n += 1
        events["mma"].append(("dw_done", None))

    def compute():
        n = 0

        def stage():
            nonlocal n
            st = n % NST
            yield W("full%d" % st, n // NST)
            st_read[st].add(("c", n))
            if mutation == "early_empty":
                bars["empty%d" % st].arrive()
            yield ("yield",)
            st_read[st].discard(("c", n))
            if mutation != "early_empty":
                bars["empty%d" % st].arrive()
            n += 1

        for t in range(T_):
            for q in range(NB):
                yield from stage()
            yield W("acc_full", t)
            tm.compute([0], False, "projections read back")
            yield ("yield",)
            tm.release([0], False)
            assert t_read[0] == 0, "T written while read"
            t_write[0] += 1
            yield ("yield",)  # scan: dA|dB parts into T
            t_write[0] -= 1
            bars["t_ready"].arrive()
            for q in range(NB):
                yield from stage()
            if mutation != "no_dh_full_wait":
                yield W("dh_full", t)
            tm.compute([0], False, "d_h read back")
            yield ("yield",)
            tm.release([0], False)
            bars["dh_free"].arrive()
        yield W("dw_done", 0)
        tm.compute([1], False, "dW read back")
        tm.release([1], False)

    schedule({"p": producer(), "m": mma(), "c": compute()}, bars, events, seed)


MODELS = {"fwd_tc16": fwd_tc16, "fwd_bf16": fwd_bf16, "bwd_tc": bwd_tc, "fwd_tc": fwd_tc,
          "wide_tc_fwd": wide_tc, "wide_tc_bwd": wide_tc_bwd, "wide_tc_dw": wide_tc_dw,
          "bwd_bf16": bwd_bf16}
