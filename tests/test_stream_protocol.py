"""CPU model of the streaming kernel's ring protocol (spec_stream_kernel.cuh), under random warp
interleavings.

The kernel's roles meet only at mbarriers: per ring slot a "full" barrier (one arrival: the
producer's bulk copy) and an "empty" barrier (15 arrivals: the data warps); per item the pass-1
statistics (15 arrivals), the decision (the control warp) and pass 2 (15 arrivals); per batch
three named barriers. The model runs each role's sequence of waits and arrivals exactly as the
kernel's loops issue them, with the ring sizes read from the kernel source, and checks:
  * the protocol completes (no deadlock) for every item mix, tile count and cluster size;
  * every wait on a "full" barrier finds the tile it expects (item, pass, tile), and no wait
    ever sees a barrier two phases ahead (the parity of an mbarrier cannot tell them apart);
  * pass 2 reads each draft tile where pass 1 left it: the slot was not refilled meanwhile.
Mistakes planted in the model (a draft ring one slot short, a producer that refills a slot
without waiting for it to be emptied, pass 1 streaming tiles for an item with no rows) fail it.
"""
import os
import random
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "speculative_decoding_verification_43_gb300", "csrc")
W = 15          # data warps
LAG = 1         # pass 2 of item i - 1 runs after pass 1 of item i
MAX_ITEMS = 22  # descriptors per batch


def kernel_constants():
    rows = open(os.path.join(SRC, "spec_rows.cuh")).read()
    stream = open(os.path.join(SRC, "spec_stream_kernel.cuh")).read()
    max_rows = int(re.search(r"constexpr int kMaxStreamRows = (\d+);", rows).group(1))
    items = int(re.search(r"constexpr int kMaxItems = (\d+);", rows).group(1))
    lag = int(re.search(r"constexpr int kStreamLag = (\d+);", rows).group(1))
    vpt = re.search(r"kVPT = \(DT == SPEC_BF16\) \? (\d+) : (\d+);", stream)
    tring = int(re.search(r"static constexpr int kTRing = (\d+);", stream).group(1))
    assert re.search(r"static constexpr int kDRing = 2 \* kMaxTiles;", stream)
    geos = []
    for v in (int(vpt.group(1)), int(vpt.group(2))):
        max_tiles = max_rows // v
        geos.append((tring, 2 * max_tiles, max_tiles))
    return geos, items, lag


class Bar:
    def __init__(self, n):
        self.n, self.cnt, self.done = n, 0, 0

    def arrive(self):
        self.cnt += 1
        if self.cnt == self.n:
            self.cnt, self.done = 0, self.done + 1


class CTA:
    def __init__(self, tr, dr, ntiles, planted):
        self.tr, self.dr, self.ntiles, self.planted = tr, dr, ntiles, planted
        self.tfull = [Bar(1) for _ in range(tr)]
        self.tempty = [Bar(W) for _ in range(tr)]
        self.dfull = [Bar(1) for _ in range(dr)]
        self.dempty = [Bar(W) for _ in range(dr)]
        self.tseq, self.dseq = {}, {}
        self.stats, self.p2, self.decs, self.xreach = {}, {}, set(), -1


def data_prog(c, batches):
    """One data warp: stream_pass1 / stream_pass2 and the data loop of the kernel."""
    tp = dp = 0
    g0 = 0
    for nb, batch in enumerate(batches):
        yield ("narrive", "BATCH")
        yield ("nwait", "BATCH", W + 1)
        db_prev = 0
        for i in range(len(batch) + LAG):
            db_cur = dp
            if i < len(batch):
                nr = batch[i]
                nt = c.ntiles if (nr >= 1 or c.planted == "rows_for_bad_shape") else 0
                for t in range(nt):
                    yield ("wfull", "t", tp, ("P1", nb, i, t))
                    if nr == 2:
                        yield ("wfull", "d", dp, (nb, i, t))
                    yield ("empty", "t", tp)
                    tp += 1
                    if nr == 2:
                        dp += 1
                yield ("stats", g0 + i)
            if i >= LAG:
                m = i - LAG
                yield ("dec", g0 + m)
                if batch[m] == 2:
                    for t in range(c.ntiles):
                        yield ("wfull", "t", tp, ("P2", nb, m, t))
                        yield ("still", db_prev + t, (nb, m, t))
                        yield ("empty", "t", tp)
                        yield ("empty", "d", db_prev + t)
                        tp += 1
                yield ("p2", g0 + m)
            db_prev = db_cur
        g0 += len(batch)


def producer_prog(c, kind, batches):
    """produce_targets / produce_drafts and the producer warps' batch loop."""
    pos = 0
    ring = c.tr if kind == "t" else c.dr
    for nb, batch in enumerate(batches):
        yield ("nwait_after_arrive", "SHAPES", 3)
        seq = []
        if kind == "t":
            for i in range(len(batch) + LAG):
                if i < len(batch) and batch[i] >= 1:
                    seq += [("P1", nb, i, t) for t in range(c.ntiles)]
                m = i - LAG
                if 0 <= m < len(batch) and batch[m] == 2:
                    seq += [("P2", nb, m, t) for t in range(c.ntiles)]
        else:
            for i in range(len(batch)):
                if batch[i] == 2:
                    seq += [(nb, i, t) for t in range(c.ntiles)]
        for tag in seq:
            if pos >= ring and c.planted != "no_empty_wait":
                yield ("wempty", kind, pos)
            yield ("issue", kind, pos, tag)
            pos += 1
        yield ("narrive", "PROD")


def control_prog(c, batches):
    """The control warp's batch and exchange loop."""
    g0 = e = 0
    for nb, batch in enumerate(batches):
        yield ("narrive", "SHAPES")
        yield ("narrive", "BATCH")
        for j in range(len(batch) + LAG + 1):
            g, m = g0 + j, j - LAG - 1
            if j < len(batch):
                yield ("wstats", g)
            if m >= 0:
                yield ("wp2", g0 + m)
            yield ("xarr", e)
            yield ("xwait", e)
            if j < len(batch):
                yield ("setdec", g)
            e += 1
        yield ("narrive", "PROD")
        yield ("nwait", "PROD", 3)
        g0 += len(batch)


def run(seed, rows, ntiles_of_cta, geo, planted=None):
    tr, dr, _ = geo
    if planted == "short_draft_ring":
        dr -= 1
    rng = random.Random(seed)
    batches = [rows[k:k + MAX_ITEMS] for k in range(0, len(rows), MAX_ITEMS)]
    ctas = [CTA(tr, dr, nt, planted) for nt in ntiles_of_cta]
    progs = []
    for ci, c in enumerate(ctas):
        pl = [(ci, data_prog(c, batches)) for _ in range(W)]
        pl += [(ci, producer_prog(c, "t", batches)), (ci, producer_prog(c, "d", batches)), (ci, control_prog(c, batches))]
        progs.append(pl)
    allp = [p for pl in progs for p in pl]
    pend = {id(p): next(p[1], None) for p in allp}
    named = {}   # (cta, name) -> {generation: arrivals}
    gen = {}     # (program, name) -> its generation
    sync_arrived = set()

    def ring(c, k):
        return (c.tfull, c.tempty, c.tr, c.tseq) if k == "t" else (c.dfull, c.dempty, c.dr, c.dseq)

    while True:
        runnable = []
        for p in allp:
            op = pend[id(p)]
            if op is None:
                continue
            c = ctas[p[0]]
            kind = op[0]
            if kind == "wfull":
                full, _, r, seq = ring(c, op[1])
                d = full[op[2] % r].done
                assert d <= op[2] // r + 1, "a full barrier two phases ahead of its waiter"
                if d == op[2] // r + 1:
                    assert seq[op[2]] == op[3], ("wrong tile", op, seq[op[2]])
                    runnable.append(p)
            elif kind == "still":
                assert c.dfull[op[1] % c.dr].done == op[1] // c.dr + 1 and c.dseq[op[1]] == op[2], \
                    "a draft tile was overwritten before pass 2 read it"
                runnable.append(p)
            elif kind == "wempty":
                _, empty, r, _ = ring(c, op[1])
                d = empty[op[2] % r].done
                assert d <= op[2] // r, "an empty barrier two phases ahead of its waiter"
                if d == op[2] // r:
                    runnable.append(p)
            elif kind in ("nwait", "nwait_after_arrive"):
                key = (id(p), op[1])
                if kind == "nwait_after_arrive" and key not in sync_arrived:
                    runnable.append(p)  # its arrival first
                elif named.get((p[0], op[1]), {}).get(gen.get(key, 0) - 1, 0) >= op[2]:
                    runnable.append(p)
            elif kind == "dec":
                if op[1] in c.decs:
                    runnable.append(p)
            elif kind == "wstats":
                if c.stats.get(op[1], 0) == W:
                    runnable.append(p)
            elif kind == "wp2":
                if c.p2.get(op[1], 0) == W:
                    runnable.append(p)
            elif kind == "xwait":
                if all(x.xreach >= op[1] for x in ctas):
                    runnable.append(p)
            else:
                runnable.append(p)
        if not runnable:
            left = [pend[id(p)] for p in allp if pend[id(p)] is not None]
            assert not left, ("deadlock", left[:4])
            return
        p = rng.choice(runnable)
        op = pend[id(p)]
        c = ctas[p[0]]
        kind = op[0]
        advance = True
        if kind in ("narrive", "nwait_after_arrive") and (kind == "narrive" or (id(p), op[1]) not in sync_arrived):
            key = (id(p), op[1])
            g = gen.get(key, 0)
            d = named.setdefault((p[0], op[1]), {})
            d[g] = d.get(g, 0) + 1
            gen[key] = g + 1
            if kind == "nwait_after_arrive":
                sync_arrived.add(key)
                advance = False
        elif kind == "nwait_after_arrive":
            sync_arrived.discard((id(p), op[1]))
        elif kind == "empty":
            _, empty, r, _ = ring(c, op[1])
            empty[op[2] % r].arrive()
        elif kind == "issue":
            full, _, r, seq = ring(c, op[1])
            assert full[op[2] % r].done == op[2] // r, "a slot refilled while its copy is still unread"
            seq[op[2]] = op[3]
            full[op[2] % r].arrive()
        elif kind == "stats":
            c.stats[op[1]] = c.stats.get(op[1], 0) + 1
        elif kind == "p2":
            c.p2[op[1]] = c.p2.get(op[1], 0) + 1
        elif kind == "xarr":
            c.xreach = op[1]
        elif kind == "setdec":
            c.decs.add(op[1])
        if advance:
            pend[id(p)] = next(p[1], None)


def cases(geo, n, seed0):
    rng = random.Random(seed0)
    for s in range(n):
        nitems = rng.choice([1, 2, 3, 5, 8, 9, 22, 23, 30, 45])
        rows = [rng.choice([1, 2, 2, 2, 0]) for _ in range(nitems)]
        C = rng.choice([1, 2, 4])
        yield s, rows, [rng.randint(1, geo[2]) for _ in range(C)]


def test_constants_match_the_model():
    geos, items, lag = kernel_constants()
    assert items == MAX_ITEMS and lag == LAG
    assert len(geos) == 2 and all(tr >= 1 and dr >= 2 for tr, dr, _ in geos)


@pytest.mark.parametrize("which", [0, 1], ids=["bf16", "f32"])
def test_ring_protocol_completes_and_reads_the_right_tiles(which):
    geo = kernel_constants()[0][which]
    for s, rows, nts in cases(geo, 25, 100 + which):
        run(s, rows, nts, geo)


@pytest.mark.parametrize("planted", ["short_draft_ring", "no_empty_wait", "rows_for_bad_shape"])
def test_planted_mistakes_are_caught(planted):
    geo = kernel_constants()[0][0]
    caught = False
    for s, rows, nts in cases(geo, 25, 7):
        if planted == "rows_for_bad_shape" and 0 not in rows:
            continue
        try:
            run(s, rows, [geo[2]] * len(nts), geo, planted)
        except AssertionError:
            caught = True
            break
    assert caught, planted
