"""CPU model of the tensor-core decode's dynamic item order (no GPU).

Each warp of the persistent grid has a producer that issues an item's pages
into a ring of ST stages and a consumer that takes them in order.  The
producer walks the warp's items -- its own index first, then items claimed
from one counter shared by the grid -- and writes a record of each (and of
the end) into a 32-entry ring that the consumer replays.  The producer stops
while 32 records are unread; at the end of each item the consumer tops the
copies in flight up to ST before it reads the next record.

The model runs the warps in random interleavings over random item lists
(many without pages: empty contexts) and checks that every item is consumed
exactly once, every page in the order it was issued, no record is read before
it is written or overwritten before it is read, and no warp ever has more than
ST pages in flight.  Two planted mistakes must be caught: the consumer moving
on without topping up (a page it waits for is never issued) and a producer
that ignores the ring's capacity."""
import random

import pytest

RING = 32


class _Fail(Exception):
    pass


def _run(items_pages, W, ST, seed, dynamic=True, top_up=True, ring_check=True):
    rng = random.Random(seed)
    n_items = len(items_pages)
    counter = [0]
    done = [0] * n_items

    class Warp:
        pass

    warps = []
    for gw in range(W):
        w = Warp()
        w.item, w.valid = gw, gw < n_items
        w.page, w.n_pages = 0, (items_pages[gw] if gw < n_items else 0)
        w.ring = [None] * RING
        w.n_rec = w.n_cons = 0
        w.claim = None
        w.issued = w.consumed = 0
        w.stages = []
        warps.append(w)

    def record(w):
        if w.ring[w.n_rec % RING] is not None and w.ring[w.n_rec % RING][1] >= w.n_cons:
            raise _Fail("record overwritten before it was read")
        w.ring[w.n_rec % RING] = ((w.item if w.valid else -1), w.n_rec)
        w.n_rec += 1

    def claim_next(w):
        w.claim = counter[0]
        counter[0] += 1

    def prod_advance(w):
        while w.valid and w.page >= w.n_pages:
            if ring_check and w.n_rec - w.n_cons >= RING:
                return False
            if dynamic:
                if w.claim is None:
                    claim_next(w)
                w.item = W + w.claim
            else:
                w.item += W
            w.valid = w.item < n_items
            w.page, w.n_pages = 0, (items_pages[w.item] if w.valid else 0)
            if dynamic and w.valid:
                claim_next(w)
            record(w)
        return w.valid

    def issue_next(w):
        if not prod_advance(w):
            return False
        w.stages.append((w.item, w.page))
        w.page += 1
        w.issued += 1
        if w.issued - w.consumed > ST:
            raise _Fail("more than ST pages in flight")
        return True

    def enter(w):
        if w.n_cons >= w.n_rec:
            raise _Fail("record read before it was written")
        it, seq = w.ring[w.n_cons % RING]
        if seq != w.n_cons:
            raise _Fail("record overwritten before it was read")
        w.c_item, w.c_valid, w.c_page = it, it >= 0, 0
        w.c_np = items_pages[it] if it >= 0 else 0

    for w in warps:
        record(w)
        for _ in range(ST):
            if not issue_next(w):
                break
        enter(w)
    active = [w for w in warps if w.c_valid]
    while active:
        w = rng.choice(active)
        if w.c_page < w.c_np:
            if not w.stages:
                raise _Fail("the consumer waits for a page that was never issued")
            page = w.stages.pop(0)
            if page != (w.c_item, w.c_page):
                raise _Fail("pages out of order")
            w.consumed += 1
            w.c_page += 1
            issue_next(w)
            if dynamic and w.claim is None and w.valid:
                claim_next(w)
        if w.c_page >= w.c_np:
            if done[w.c_item]:
                raise _Fail("item consumed twice")
            done[w.c_item] = 1
            w.n_cons += 1
            if top_up:
                while w.issued - w.consumed < ST and issue_next(w):
                    pass
            elif w.n_rec <= w.n_cons:
                prod_advance(w)
            enter(w)
            if not w.c_valid:
                if w.stages:
                    raise _Fail("pages issued but never consumed")
                active.remove(w)
    if not all(done):
        raise _Fail("items never consumed")


def _cases(n):
    for trial in range(n):
        r = random.Random(trial)
        n_items = r.randint(0, 300)
        p_empty = r.choice([0.0, 0.2, 0.9])
        pages = [0 if r.random() < p_empty else r.randint(1, 12) for _ in range(n_items)]
        yield pages, r.randint(1, 48), r.randint(1, 4), trial


@pytest.mark.parametrize("dynamic", [True, False])
def test_every_item_once_in_order(dynamic):
    for pages, W, ST, seed in _cases(1500):
        _run(pages, W, ST, seed, dynamic=dynamic)


def test_long_runs_of_items_without_pages():
    """Hundreds of empty items in a row: the producer stops at 32 unread
    records and the consumer drains them."""
    pages = [3] + [0] * 500 + [5, 0, 0, 7] + [0] * 200 + [2]
    for seed in range(50):
        _run(pages, 1, 2, seed)
        _run(pages, 3, 3, seed)


def test_moving_on_without_topping_up_is_caught():
    with pytest.raises(_Fail):
        for pages, W, ST, seed in _cases(1500):
            _run(pages, W, ST, seed, top_up=False)


def test_ignoring_the_ring_capacity_is_caught():
    with pytest.raises(_Fail):
        _run([1] + [0] * 100 + [4], 1, 2, 0, ring_check=False)
