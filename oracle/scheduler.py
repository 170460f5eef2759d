"""Plain-Python reference of the two-phase continuous-batching scheduler.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py): it shares no code with the
product's C++ scheduler and is used by tests to check that scheduler decision
by decision.

Policy (PhotonInfer README, "Technical details > Continuous batching
scheduler"): phase 1 continues every RUNNING request; phase 2 admits WAITING
requests into the remaining capacity; states WAITING -> RUNNING -> FINISHED,
with PREEMPTED; num_computed_tokens marks where a request resumes.  Readings
taken where the page is silent:
  - a request knows L = prompt + generated tokens; when scheduled it processes
    tokens [num_computed, L) and holds ceil(L / block_size) blocks;
  - phase 1 preempts the most recently admitted running request while the
    free blocks cannot cover the running requests' next blocks (blocks freed,
    num_computed = 0, back to the front of the waiting queue);
  - phase 2 admits first come first served while a batch slot, the step's token
    budget and the request's blocks are available; the first misfit stops it;
  - after a step every scheduled request has computed L tokens and generated
    one more; reaching max_new_tokens finishes it and frees its blocks.

The block pool is a free list shuffled once by Fisher-Yates driven by
splitmix64 (Steele, Lea & Flood, OOPSLA 2014) with rejection sampling, handing
out blocks from the end of the list and taking freed blocks back at the end.
"""
from __future__ import annotations

MASK64 = (1 << 64) - 1
WAITING, RUNNING, FINISHED, PREEMPTED = 0, 1, 2, 3


def splitmix64_next(state: int):
    """One step of splitmix64: returns (new_state, output)."""
    state = (state + 0x9E3779B97F4A7C15) & MASK64
    z = state
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return state, z ^ (z >> 31)


class Pool:
    def __init__(self, num_blocks: int, seed: int):
        free = list(range(num_blocks))
        st = seed & MASK64
        for i in range(num_blocks - 1, 0, -1):
            n = i + 1
            limit = MASK64 - (MASK64 % n)  # accept draws below the largest multiple of n
            while True:
                st, r = splitmix64_next(st)
                if r < limit:
                    break
            j = r % n
            free[i], free[j] = free[j], free[i]
        self.free = free

    def alloc(self, n: int):
        assert n <= len(self.free)
        out = [self.free.pop() for _ in range(n)]
        return out

    def release(self, ids):
        self.free.extend(ids)


class Request:
    def __init__(self, rid, prompt_len, max_new):
        self.id, self.prompt_len, self.max_new = rid, prompt_len, max_new
        self.generated = 0
        self.computed = 0
        self.state = WAITING
        self.blocks = []

    @property
    def known(self):
        return self.prompt_len + self.generated


def _ceil(a, b):
    return -(-a // b)


class Scheduler:
    def __init__(self, pool: Pool, max_running, max_step_tokens, max_blocks_per_seq, block_size=16):
        self.pool, self.max_running, self.budget = pool, max_running, max_step_tokens
        self.width, self.bs = max_blocks_per_seq, block_size
        self.reqs, self.waiting, self.running, self.stepped = {}, [], [], None

    def add_request(self, rid, prompt_len, max_new):
        self.reqs[rid] = Request(rid, prompt_len, max_new)
        self.waiting.append(rid)

    def schedule(self):
        assert self.stepped is None
        bs = self.bs
        preempted = admitted = 0

        def extra():
            return sum(max(0, _ceil(self.reqs[i].known, bs) - len(self.reqs[i].blocks))
                       for i in self.running)

        # phase 1
        while self.running and extra() > len(self.pool.free):
            r = self.reqs[self.running.pop()]
            self.pool.release(r.blocks)
            r.blocks, r.computed, r.state = [], 0, PREEMPTED
            self.waiting.insert(0, r.id)
            preempted += 1
        tokens = 0
        for i in self.running:
            r = self.reqs[i]
            need = _ceil(r.known, bs) - len(r.blocks)
            if need > 0:
                r.blocks += self.pool.alloc(need)
            tokens += r.known - r.computed
        # phase 2
        while self.waiting and len(self.running) < self.max_running:
            r = self.reqs[self.waiting[0]]
            new = r.known - r.computed
            need = _ceil(r.known, bs)
            if tokens + new > self.budget or need > len(self.pool.free):
                break
            r.blocks = self.pool.alloc(need)
            r.state = RUNNING
            self.running.append(self.waiting.pop(0))
            tokens += new
            admitted += 1
        # batch
        rows, ts, pos, slots = [], [], [], []
        for row, i in enumerate(self.running):
            r = self.reqs[i]
            rows.append((r.id, r.known - r.computed, r.known,
                         r.blocks + [-1] * (self.width - len(r.blocks))))
            for p in range(r.computed, r.known):
                ts.append(row)
                pos.append(p)
                slots.append(r.blocks[p // bs] * bs + p % bs)
        self.stepped = list(self.running)
        return {"request_ids": [x[0] for x in rows], "num_new_tokens": [x[1] for x in rows],
                "context_lens": [x[2] for x in rows], "block_tables": [x[3] for x in rows],
                "token_seq": ts, "positions": pos, "slot_mapping": slots,
                "max_context_len": max((x[2] for x in rows), default=0),
                "num_preempted": preempted, "num_admitted": admitted}

    def complete_step(self):
        still = []
        for i in self.stepped:
            r = self.reqs[i]
            r.computed = r.known
            r.generated += 1
            if r.generated >= r.max_new:
                self.pool.release(r.blocks)
                r.blocks, r.state = [], FINISHED
            else:
                still.append(i)
        self.running, self.stepped = still, None
