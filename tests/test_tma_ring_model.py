"""A CPU model of the bulk-copy kernel's ring protocol (rmsnorm_tma.cuh).

The model follows the kernel's walk: producer lanes for x and the residual
each copy piece k of the block's rows, in order, into the next slot of their
ring once that slot's "empty" barrier has completed the phase before, and a
third copies the weight once into its own slots when it is resident (else the
consumers read it from global memory); 16 consumer warps wait on each
piece's "full" barrier (arrival + byte count), release residual slots after
pass 1 and x slots after pass 2, with a barrier over the consumer warps
between the passes.  Copies land after random
delays and actors run in random order.  For every ring split the library can
choose (``_native.tma_rings``, itself checked against the library's plan
validation in test_abi.py) it checks:

  - every copy's source lies inside its tensor and its destination inside the
    block's dynamic shared memory, both 16-byte aligned;
  - every consumer access lies inside the landed bytes of its slot;
  - no copy targets a slot that a warp has not released;
  - a consumer reads a piece only after it landed, and it is the piece it
    expects (tensor, row, k);
  - every walk ends: no deadlock for any shape, grid or block tried.

The failure path is modelled too: every wait has a budget of scheduler steps
(the kernel's time limit); a consumer warp whose wait ran out skips its
later waits and releases no slot from then on, a producer whose wait for an
empty slot ran out stops, and the block's last act waits for the copies in
flight.  With the test hook's withheld release, or with copies that land
after the consumers gave up on them, the model checks that no copy is ever
started into a slot whose previous copy has not landed (that would arrive
twice on one phase of the slot's "full" barrier), that every walk still
ends, and that nothing lands after the drain.  Releasing slots after a
failure, the order the kernel had before, fails that check.
"""
import random

import pytest

from row_reduction_norm_gb300 import _native as N

GT = 512
WARPS = 16
BAR_BYTES = 2 * 32 * 8
BUDGET = 227 * 1024 - 1024


class Bar:
    """An mbarrier: pending arrivals and transaction bytes of the current phase."""

    def __init__(self, count):
        self.count, self.pending, self.tx, self.phase = count, count, 0, 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self):
        assert self.pending > 0
        self.pending -= 1
        self._maybe_complete()

    def arrive_expect_tx(self, nbytes):
        assert self.pending > 0, "arrival on a phase that already has all its arrivals"
        self.tx += nbytes
        self.pending -= 1
        self._maybe_complete()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        assert self.tx >= 0, "more bytes landed than expected"
        self._maybe_complete()

    def done(self, parity):          # try_wait.parity
        return (self.phase & 1) != parity


def walk(rows, hidden, esz, pc, grid, block, res, w, seed, budget=None, withhold=False, max_delay=8,
         release_after_failure=False):
    """One block's walk.  ``budget``: scheduler steps a wait may take before it
    runs out (None: unbounded); ``withhold``: consumer warp 0 keeps its first x
    slot (the kernel's test hook); ``release_after_failure``: the order the
    kernel had before, where a warp that gave up still released its slots.
    Returns the number of actors that gave up."""
    rnd = random.Random(seed)
    row_bytes = hidden * esz
    nch = row_bytes // 16
    piece = GT * 16 * pc
    sx, sr, sw = N.tma_rings(row_bytes, pc, res, w)
    pieces = -(-row_bytes // piece)
    total = sx + sr + sw
    assert total <= 32
    smem = BAR_BYTES + total * piece
    assert smem <= BUDGET
    full = [Bar(1) for _ in range(total)]
    empty = [Bar(WARPS) for _ in range(total)]
    content = [None] * total
    landed = [False] * total
    readers = [set() for _ in range(total)]
    inflight = []
    my_rows = list(range(block, rows, grid))
    w_resident = w and sw >= pieces    # else the kernel reads the weight from global memory
    assert sw in (0, pieces), "a weight ring holds the whole weight or there is none"
    base = {"x": 0, "r": sx, "w": sx + sr}
    size = {"x": sx, "r": max(sr, 1), "w": max(sw, 1)}

    def producer(tensor, once):
        b, n = base[tensor], size[tensor]
        stride = 0 if tensor == "w" else row_bytes
        limit = row_bytes if tensor == "w" else rows * row_bytes
        q = 0
        for row in my_rows:
            for k in range(pieces):
                s, ph = q % n, q // n
                if ph > 0:
                    waited = 0
                    while not empty[b + s].done((ph - 1) & 1):
                        waited += 1
                        if budget is not None and waited > budget:
                            failed.append(tensor)
                            return
                        yield
                off = k * piece
                nbytes = min(piece, row_bytes - off)
                src = (0 if once else row * stride) + off
                assert nbytes > 0 and nbytes % 16 == 0 and src % 16 == 0 and src + nbytes <= limit
                g = b + s
                dst = BAR_BYTES + g * piece
                assert dst % 16 == 0 and dst + nbytes <= smem
                assert not readers[g], f"{tensor} copy into slot {g} still read by warps {readers[g]}"
                full[g].arrive_expect_tx(nbytes)
                content[g] = (tensor, None if once else row, k)
                landed[g] = False
                readers[g] = set(range(WARPS))
                inflight.append([rnd.randint(0, max_delay), g, nbytes])
                q += 1
                yield
            if once:
                break

    arrived = {}
    failed = []

    def wait_full(g, parity, st):
        """Consumer wait on a full barrier; st["ok"] turns False when it runs out."""
        if not st["ok"]:
            return
        waited = 0
        while not full[g].done(parity):
            waited += 1
            if budget is not None and waited > budget:
                st["ok"] = False
                failed.append("consumer")
                return
            yield

    def release(g, wid, st, withheld=False):
        if st["ok"] or release_after_failure:
            readers[g].discard(wid)
            if not withheld:
                empty[g].arrive()

    def reads(g, k, wid):
        for t in range(wid * 32, wid * 32 + 32):
            for j in range(pc):
                if (k * pc + j) * GT + t < nch:
                    so = (j * GT + t) * 16
                    assert so + 16 <= min(piece, row_bytes - k * piece)

    def consumer(wid):
        qx = qr = 0
        st = {"ok": True}
        for ri, row in enumerate(my_rows):
            for k in range(pieces):                       # pass 1
                g = (qx + k) % sx
                yield from wait_full(g, ((qx + k) // sx) & 1, st)
                if st["ok"]:
                    assert landed[g] and content[g] == ("x", row, k)
                    reads(g, k, wid)
                if res:
                    gr = sx + qr % sr
                    yield from wait_full(gr, (qr // sr) & 1, st)
                    if st["ok"]:
                        assert landed[gr] and content[gr] == ("r", row, k)
                        reads(gr, k, wid)
                    release(gr, wid, st)
                    qr += 1
                yield
            arrived[ri] = arrived.get(ri, 0) + 1          # barrier over the consumer warps
            while arrived[ri] < WARPS:
                yield
            for k in range(pieces):                       # pass 2
                g = (qx + k) % sx
                if st["ok"]:
                    assert content[g] == ("x", row, k)
                if w_resident:
                    gw = sx + sr + k
                    yield from wait_full(gw, 0, st)
                    if st["ok"]:
                        assert landed[gw] and content[gw] == ("w", None, k)
                        reads(gw, k, wid)
                elif w:
                    for t in range(wid * 32, wid * 32 + 32):   # the weight's chunks, straight from global memory
                        for j in range(pc):
                            u = (k * pc + j) * GT + t
                            if u < nch:
                                assert (u + 1) * 16 <= row_bytes
                release(g, wid, st, withheld=withhold and wid == 0 and qx + k == 0)
                yield
            qx += pieces

    actors = [producer("x", False)]
    if res:
        actors.append(producer("r", False))
    if w_resident:
        actors.append(producer("w", True))
    actors += [consumer(i) for i in range(WARPS)]
    alive = [True] * len(actors)
    steps = 0
    while any(alive):
        steps += 1
        assert steps < 2_000_000, "no progress: the walk deadlocked"
        for c in list(inflight):
            if c[0] == 0:
                inflight.remove(c)
                landed[c[1]] = True
                full[c[1]].complete_tx(c[2])
            else:
                c[0] -= 1
        order = list(range(len(actors)))
        rnd.shuffle(order)
        for i in order:
            if alive[i]:
                try:
                    next(actors[i])
                except StopIteration:
                    alive[i] = False
    if failed:
        # the block's drain: its last thread waits for every copy in flight
        while inflight:
            for c in list(inflight):
                if c[0] == 0:
                    inflight.remove(c)
                    landed[c[1]] = True
                    full[c[1]].complete_tx(c[2])
                else:
                    c[0] -= 1
    assert not inflight, "copies still in flight when every actor finished"
    return len(failed)


SHAPES = [(2, 65536), (2, 40000), (4, 16388), (4, 40960), (2, 8), (2, 8200)]


@pytest.mark.parametrize("esz,hidden", SHAPES)
@pytest.mark.parametrize("pc", N.TMA_PIECE_CHUNKS)
def test_ring_protocol_model(esz, hidden, pc):
    tried = 0
    for res in (False, True):
        for w in (False, True):
            if N.tma_rings(hidden * esz, pc, res, w) is None:
                continue
            for rows, grid in ((1, 1), (9, 2), (7, 152)):
                for block in sorted({0, min(grid, rows) - 1}):
                    walk(rows, hidden, esz, pc, grid, block, res, w, seed=rows * 31 + block + pc)
                    tried += 1
    if tried == 0:
        pytest.skip("row larger than the rings at this piece size")


def test_model_covers_every_ring_split():
    """Both weight modes (resident, read from global memory), with and without
    a residual, occur among the shapes above for every piece size."""
    seen = set()
    for esz, hidden in SHAPES:
        for pc in N.TMA_PIECE_CHUNKS:
            for res in (False, True):
                for w in (False, True):
                    r = N.tma_rings(hidden * esz, pc, res, w)
                    if r is not None and w:
                        seen.add((pc, res, r[2] >= -(-hidden * esz // (GT * 16 * pc))))
    for pc in N.TMA_PIECE_CHUNKS:
        for res in (False, True):
            assert (pc, res, True) in seen and (pc, res, False) in seen, (pc, res)


@pytest.mark.parametrize("esz,hidden", [(2, 40960), (2, 8200), (4, 16388)])
@pytest.mark.parametrize("pc", N.TMA_PIECE_CHUNKS)
def test_withheld_release_gives_up_safely(esz, hidden, pc):
    """The test hook: warp 0 keeps its first x slot.  The x producer's wait
    for that slot runs out, the consumers' waits for the pieces it no longer
    copies run out, nothing is copied into a slot still in use, and every walk
    ends (the kernel then counts the block in its timeout counter)."""
    tried = 0
    for res in (False, True):
        for w in (False, True):
            rings = N.tma_rings(hidden * esz, pc, res, w)
            if rings is None:
                continue
            sx, pieces = rings[0], -(-hidden * esz // (GT * 16 * pc))
            rows = 2 * -(-sx // pieces) + 1      # enough rows that slot 0 is needed again
            for grid in (1, 2):
                gave_up = walk(rows, hidden, esz, pc, grid, 0, res, w, seed=pc * 7 + grid, budget=60,
                               withhold=True)
                assert gave_up >= 1
                tried += 1
    if tried == 0:
        pytest.skip("row larger than the rings at this piece size")


def test_late_copies_with_failed_consumers_never_reuse_a_filling_slot():
    """Copies that land after the consumers gave up on them: with failed warps
    keeping their slots, no slot is refilled while its copy is in flight; the
    order the kernel had before (a failed warp still releasing) is caught by
    the model on at least one of the same walks."""
    walks = [(2, 8200, 1, res, w, seed) for res in (False, True) for w in (False, True) for seed in range(12)]
    old_order_caught = 0
    for esz, hidden, pc, res, w, seed in walks:
        if N.tma_rings(hidden * esz, pc, res, w) is None:
            continue
        walk(9, hidden, esz, pc, 1, 0, res, w, seed=seed, budget=6, max_delay=40)
        try:
            walk(9, hidden, esz, pc, 1, 0, res, w, seed=seed, budget=6, max_delay=40, release_after_failure=True)
        except AssertionError:
            old_order_caught += 1
    assert old_order_caught > 0
