"""The page-balanced split-K schedule of the FP8 decode, checked on the CPU
through a direct model of its arithmetic: the unit stream (sequence by
sequence, one unit per page, an empty context one unit) cut into runs of
q = max(ceil(U / groups), partition / 16) units, group j taking run j and
each of its warps one KV head; the piece of a run in a sequence starting at
unit A is piece floor(u / q) - floor(A / q) of
floor((A + u_s - 1) / q) - floor(A / q) + 1.

What the device code and the workspace size rely on: every page of every
(sequence, KV head) is processed exactly once; every (sequence, KV head)
has exactly one piece 0 (which records the piece count) and pieces
0 .. P - 1; P never exceeds the slots the workspace holds per row
(partitions of partition_size tokens in max_context_len, plus one); and
every warp gets the same number of units but for the stream's tail."""
import numpy as np
import pytest


def _units(ctx):
    return 1 if ctx <= 0 else (ctx + 15) // 16


def _schedule(ctx, num_kv_heads, partition, warps):
    tot = sum(_units(c) for c in ctx)
    groups = warps // num_kv_heads
    q = max(-(-tot // groups), max(partition // 16, 1))
    base = np.cumsum([0] + [_units(c) for c in ctx])
    pieces, load = {}, []
    for gw in range(groups * num_kv_heads):
        j, h = divmod(gw, num_kv_heads)
        u, u_end = j * q, min((j + 1) * q, tot)
        done = 0
        while u < u_end:
            s = int(np.searchsorted(base, u, side="right") - 1)
            us = _units(ctx[s])
            a = int(base[s])
            end = min(a + us, u_end)
            n_real = us if ctx[s] > 0 else 0
            pg0 = u - a
            n_pages = max(0, min(n_real, pg0 + (end - u)) - pg0)
            p = u // q - a // q
            P = (a + us - 1) // q - a // q + 1
            pieces.setdefault((s, h), []).append((p, P, pg0, n_pages))
            done += end - u
            u = end
        load.append(done)
    return pieces, load, q


@pytest.mark.parametrize("seed", range(40))
def test_balanced_pieces_cover_every_page_once_within_the_slots(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 70))
    H = int(rng.choice([1, 2, 4, 8]))
    ctx = rng.integers(0, 2500, size=B)
    if rng.random() < 0.4:
        ctx[rng.integers(0, B)] = int(rng.integers(5000, 40000))
    ctx[rng.random(B) < 0.1] = 0
    part = int(rng.choice([16, 48, 128, 512]))
    max_ctx = max(int(ctx.max()), 1)
    warps = int(rng.choice([8, 64, 1216, 1824, 2432]))
    if warps < H:
        return
    pieces, load, q = _schedule(ctx.tolist(), H, part, warps)
    p_part = -(-max_ctx // part)
    slots = p_part + 1 if p_part > 1 else 1
    for s in range(B):
        for h in range(H):
            ps = sorted(pieces[(s, h)])
            P = ps[0][1]
            assert [x[0] for x in ps] == list(range(P))   # pieces 0 .. P-1, one piece 0
            assert all(x[1] == P for x in ps)
            assert P <= slots
            pages = sorted(pg for (_, _, pg0, n) in ps for pg in range(pg0, pg0 + n))
            assert pages == list(range(_units(ctx[s]) if ctx[s] > 0 else 0))
    tot = sum(_units(c) for c in ctx)
    tail = tot % q
    # every warp's run is q units, except the stream's last (partial) run and
    # the runs past its end
    assert set(load) <= {0, q, tail}
    assert sum(1 for x in load if x not in (0, q)) <= H


def test_balanced_pieces_single_piece_sequences_need_no_workspace_slot_beyond_one():
    # a context shorter than the partition, inside one run: one piece, written directly
    pieces, _, _ = _schedule([100, 20, 0], 2, 512, 1824)
    assert all(v[0][1] == 1 for v in pieces.values())
