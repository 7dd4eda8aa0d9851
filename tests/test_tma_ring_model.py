"""A CPU model of the bulk-copy kernel's ring protocol (rmsnorm_tma.cuh).

The model follows the kernel's walk: three producer lanes (x, residual,
weight) each copy piece k of the block's rows, in order, into the next slot of
their ring once that slot's "empty" barrier has completed the phase before;
16 consumer warps wait on each piece's "full" barrier (arrival + byte count),
release residual slots after pass 1 and x / weight slots after pass 2, with a
barrier over the consumer warps between the passes.  Copies land after random
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
        self.tx += nbytes
        self.pending -= 1
        self._maybe_complete()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        assert self.tx >= 0, "more bytes landed than expected"
        self._maybe_complete()

    def done(self, parity):          # try_wait.parity
        return (self.phase & 1) != parity


def walk(rows, hidden, esz, pc, grid, block, res, w, seed):
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
    w_resident = sw >= pieces
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
                    while not empty[b + s].done((ph - 1) & 1):
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
                inflight.append([rnd.randint(0, 8), g, nbytes])
                q += 1
                yield
            if once:
                break

    arrived = {}

    def reads(g, k, wid):
        for t in range(wid * 32, wid * 32 + 32):
            for j in range(pc):
                if (k * pc + j) * GT + t < nch:
                    so = (j * GT + t) * 16
                    assert so + 16 <= min(piece, row_bytes - k * piece)

    def consumer(wid):
        qx = qr = qw = 0
        for ri, row in enumerate(my_rows):
            for k in range(pieces):                       # pass 1
                g = (qx + k) % sx
                while not full[g].done(((qx + k) // sx) & 1):
                    yield
                assert landed[g] and content[g] == ("x", row, k)
                reads(g, k, wid)
                if res:
                    gr = sx + qr % sr
                    while not full[gr].done((qr // sr) & 1):
                        yield
                    assert landed[gr] and content[gr] == ("r", row, k)
                    reads(gr, k, wid)
                    readers[gr].discard(wid)
                    empty[gr].arrive()
                    qr += 1
                yield
            arrived[ri] = arrived.get(ri, 0) + 1          # barrier over the consumer warps
            while arrived[ri] < WARPS:
                yield
            for k in range(pieces):                       # pass 2
                g = (qx + k) % sx
                assert content[g] == ("x", row, k)
                if w:
                    gw = sx + sr + (k if w_resident else qw % sw)
                    while not full[gw].done(0 if w_resident else (qw // sw) & 1):
                        yield
                    assert landed[gw] and content[gw] == ("w", None if w_resident else row, k)
                    reads(gw, k, wid)
                readers[g].discard(wid)
                empty[g].arrive()
                if w and not w_resident:
                    readers[gw].discard(wid)
                    empty[gw].arrive()
                    qw += 1
                yield
            qx += pieces

    actors = [producer("x", False)]
    if res:
        actors.append(producer("r", False))
    if w:
        actors.append(producer("w", w_resident))
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
    assert not inflight, "copies still in flight when every actor finished"


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
    """Both weight modes (resident, streamed), with and without a residual,
    occur among the shapes above for every piece size."""
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
