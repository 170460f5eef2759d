"""Two-phase continuous-batching scheduler (PhotonInfer README, "Technical
details > Continuous batching scheduler"): the plain-Python reference in
oracle/scheduler.py is pinned by invariants and a published generator test
vector, then the native C++ scheduler must reproduce it decision by decision
(admissions, preemptions, block ids, slot numbers) on seeded request
streams."""
import numpy as np
import pytest

import oracle
from oracle import scheduler as osched
from tests.helpers import ensure_built


# ---------------------------------------------------------------- oracle pins

def test_splitmix64_published_vector():
    # first outputs of splitmix64 seeded with 0 (Steele, Lea & Flood 2014;
    # the vector quoted with the reference implementation)
    st, out = 0, []
    for _ in range(3):
        st, z = osched.splitmix64_next(st)
        out.append(z)
    assert out == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_pool_is_a_permutation_and_lifo():
    p = osched.Pool(100, seed=4)
    assert sorted(p.free) == list(range(100)) and p.free != list(range(100))
    a = p.alloc(3)
    p.release(a[::-1])
    assert p.alloc(3) == a  # freed blocks come back first, in reverse release order


def _run_oracle(stream, pool_blocks, max_running, budget, width, seed, steps=400):
    pool = osched.Pool(pool_blocks, seed)
    s = osched.Scheduler(pool, max_running, budget, width)
    arrivals = {}
    for t, rid, plen, mnew in stream:
        arrivals.setdefault(t, []).append((rid, plen, mnew))
    log = []
    for step in range(steps):
        for rid, plen, mnew in arrivals.get(step, []):
            s.add_request(rid, plen, mnew)
        b = s.schedule()
        log.append(b)
        s.complete_step()
        if step > max(arrivals) and all(r.state == osched.FINISHED for r in s.reqs.values()):
            break
    return s, log


def _stream(seed, n=40, max_prompt=120, max_new=30, horizon=60):
    rng = np.random.default_rng(seed)
    out = []
    for rid in range(n):
        out.append((int(rng.integers(0, horizon)), rid, int(rng.integers(1, max_prompt)),
                    int(rng.integers(1, max_new))))
    return sorted(out)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_oracle_scheduler_invariants(seed):
    stream = _stream(seed)
    max_running, budget, width, bs = 8, 256, 16, 16
    s, log = _run_oracle(stream, pool_blocks=40, max_running=max_running, budget=budget,
                         width=width, seed=seed)
    reqs = s.reqs
    # every request finished with exactly max_new generated tokens, nothing held
    assert all(r.state == osched.FINISHED and r.generated == r.max_new and not r.blocks
               for r in reqs.values())
    assert sorted(s.pool.free) == list(range(40))
    preempted_any = False
    admitted_order = []
    for b in log:
        n = len(b["request_ids"])
        assert n <= max_running
        # live blocks are disjoint and cover each context
        used = [x for row in b["block_tables"] for x in row if x >= 0]
        assert len(used) == len(set(used))
        for row, ctx in zip(b["block_tables"], b["context_lens"]):
            assert sum(x >= 0 for x in row) == -(-ctx // bs)
        # tokens: positions num_computed .. L-1 of each row, slots in its blocks
        assert len(b["token_seq"]) == sum(b["num_new_tokens"])
        for t, (r, p, sl) in enumerate(zip(b["token_seq"], b["positions"], b["slot_mapping"])):
            assert p < b["context_lens"][r] and sl == b["block_tables"][r][p // bs] * bs + p % bs
        # admissions keep the token budget (running rows cost one token each)
        new_rows = b["num_admitted"]
        if new_rows:
            assert sum(b["num_new_tokens"]) <= budget or new_rows == 0
            admitted_order += b["request_ids"][n - new_rows:]
        preempted_any |= b["num_preempted"] > 0
    assert preempted_any, "the stream should exercise preemption"
    # first come first served: first admissions follow arrival order
    first = []
    for rid in admitted_order:
        if rid not in first:
            first.append(rid)
    assert first == [rid for _, rid, _, _ in stream]


def test_oracle_preempted_request_recomputes_from_zero():
    pool = osched.Pool(4, seed=0)  # 4 blocks of 16 tokens
    s = osched.Scheduler(pool, 4, 512, 8)
    s.add_request(0, 30, 10)   # 2 blocks
    s.add_request(1, 30, 10)   # 2 blocks
    b = s.schedule(); s.complete_step()
    assert b["request_ids"] == [0, 1] and b["num_new_tokens"] == [30, 30]
    b = s.schedule(); s.complete_step()
    assert b["num_new_tokens"] == [1, 1] and b["context_lens"] == [31, 31]
    b = s.schedule()  # both need a third block at L = 33 > 32... first request 0 grows
    # L = 32 still fits two blocks; the next step crosses into a third block
    s.complete_step()
    b = s.schedule()
    assert b["num_preempted"] == 1 and b["request_ids"] == [0]  # newest (1) preempted
    assert s.reqs[1].state == osched.PREEMPTED and s.reqs[1].computed == 0
    s.complete_step()


# ---------------------------------------------------------------- native parity

def _run_native(pk, stream, pool_blocks, max_running, budget, width, seed, steps=400):
    pool = pk.BlockPool(pool_blocks, seed)
    s = pk.Scheduler(pool, max_running, budget, width)
    arrivals = {}
    for t, rid, plen, mnew in stream:
        arrivals.setdefault(t, []).append((rid, plen, mnew))
    log = []
    for step in range(steps):
        for rid, plen, mnew in arrivals.get(step, []):
            s.add_request(rid, plen, mnew)
        log.append(s.schedule())
        s.complete_step()
        if step > max(arrivals) and s.counts()[2] == len(stream):
            break
    return s, log


@pytest.mark.parametrize("seed,pool_blocks,max_running,budget", [(0, 40, 8, 256), (1, 24, 4, 160),
                                                                 (2, 200, 16, 512), (3, 30, 8, 200)])
def test_native_scheduler_matches_oracle_decision_by_decision(seed, pool_blocks, max_running, budget):
    pk = ensure_built()
    stream = _stream(seed)
    width = 16
    _, ref = _run_oracle(stream, pool_blocks, max_running, budget, width, seed)
    s, got = _run_native(pk, stream, pool_blocks, max_running, budget, width, seed)
    assert len(got) == len(ref)
    for g, r in zip(got, ref):
        for key in ("request_ids", "num_new_tokens", "context_lens", "block_tables", "token_seq",
                    "positions", "slot_mapping"):
            assert np.array_equal(np.asarray(g[key]), np.asarray(r[key], dtype=np.asarray(g[key]).dtype).reshape(np.asarray(g[key]).shape)), key
        for key in ("max_context_len", "num_preempted", "num_admitted"):
            assert g[key] == r[key], key
    for _, rid, _, mnew in stream:
        st, nc, ng = s.request_state(rid)
        assert st == pk.REQ_FINISHED and ng == mnew
    assert s.pool.num_free() == pool_blocks


def test_native_scheduler_rejects_impossible_requests(pk=None):
    pk = ensure_built()
    pool = pk.BlockPool(10, 0)
    s = pk.Scheduler(pool, 4, 128, 8)
    with pytest.raises(pk.PhotonError):
        s.add_request(1, 0, 5)            # empty prompt
    with pytest.raises(pk.PhotonError):
        s.add_request(2, 120, 20)         # 140 tokens > 8 blocks of 16
    with pytest.raises(pk.PhotonError):
        s.add_request(3, 100, 40)         # recompute of 139 tokens > 128-token budget
    s.add_request(4, 10, 5)
    with pytest.raises(pk.PhotonError):
        s.add_request(4, 10, 5)           # duplicate id
    b = s.schedule()
    with pytest.raises(pk.PhotonError):
        s.schedule()                      # previous step not completed
    s.complete_step()
    assert list(b["request_ids"]) == [4]


def test_native_batch_tables_equal_a_fresh_rewrite_every_step():
    """The incremental block-table rows (same buffer every step) must equal the
    request's full block list every step, through admissions, finishes and
    preemptions (re-admitted requests get new blocks in possibly the same row)."""
    pk = ensure_built()
    stream = _stream(5, n=60)
    pool = pk.BlockPool(30, 5)
    s = pk.Scheduler(pool, 8, 256, 16)
    _, ref = _run_oracle(stream, 30, 8, 256, 16, 5)
    arrivals = {}
    for t, rid, plen, mnew in stream:
        arrivals.setdefault(t, []).append((rid, plen, mnew))
    preempts = 0
    for step, r in enumerate(ref):
        for rid, plen, mnew in arrivals.get(step, []):
            s.add_request(rid, plen, mnew)
        g = s.schedule(copy=False)
        preempts += g["num_preempted"]
        assert np.array_equal(g["block_tables"], np.asarray(r["block_tables"], np.int32).reshape(g["block_tables"].shape))
        s.complete_step()
    assert preempts > 0
