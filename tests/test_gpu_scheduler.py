"""The native scheduler's step batches driven through the kernels: for a few
steps of a request stream (admissions, decode steps, a preemption), the
device cache write + decode attention must match the oracle's write +
attention on host copies of the caches, using the batch's metadata."""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import ensure_built

pytestmark = pytest.mark.gpu


def test_scheduler_steps_through_the_kernels():
    import torch
    pk = ensure_built()
    Hq, Hkv, d, bs, nb, width = 8, 2, 64, 16, 16, 16  # 16 blocks: the stream preempts once
    pool = pk.BlockPool(nb, seed=7)
    sched = pk.Scheduler(pool, max_running=6, max_step_tokens=400, max_blocks_per_seq=width)
    gen = torch.Generator(device="cuda").manual_seed(3)
    kc = (torch.randn((nb, Hkv, bs, d), generator=gen, device="cuda") * 0.5).bfloat16()
    vc = (torch.randn((nb, Hkv, bs, d), generator=gen, device="cuda") * 0.5).bfloat16()
    kc_h, vc_h = synth.to_storage_numpy(kc).copy(), synth.to_storage_numpy(vc).copy()
    rng = np.random.default_rng(0)
    for rid in range(10):
        sched.add_request(rid, int(rng.integers(5, 90)), int(rng.integers(2, 12)))
    saw_preempt = False
    for step in range(14):
        b = sched.schedule()
        saw_preempt |= b["num_preempted"] > 0
        B, T = len(b["request_ids"]), len(b["token_seq"])
        if B == 0:
            sched.complete_step()
            continue
        assert np.array_equal(b["slot_mapping"],
                              oracle.slot_mapping(b["block_tables"], b["token_seq"], b["positions"], bs))
        k = (torch.randn((T, Hkv, d), generator=gen, device="cuda") * 0.5).bfloat16()
        v = (torch.randn((T, Hkv, d), generator=gen, device="cuda") * 0.5).bfloat16()
        q = (torch.randn((B, Hq, d), generator=gen, device="cuda") * 0.5).bfloat16()
        pk.photon_kv_cache_write(k, v, torch.from_numpy(b["positions"]).cuda(),
                                 torch.from_numpy(b["slot_mapping"]).cuda(), kc, vc, 5e5)
        part = 32
        n = pk.photon_paged_attention_workspace_size(B, Hq, d, b["max_context_len"], part)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
        out = torch.empty((B, Hq, d), device="cuda")
        pk.photon_paged_attention_decode(q, kc, vc, torch.from_numpy(b["block_tables"]).cuda(),
                                         torch.from_numpy(b["context_lens"]).cuda(), 0.125, out,
                                         b["max_context_len"], part, ws)
        oracle.kv_cache_write(synth.to_storage_numpy(k), synth.to_storage_numpy(v), b["positions"],
                              b["slot_mapping"], kc_h, vc_h, 5e5)
        ref = oracle.paged_attention(synth.to_storage_numpy(q), kc_h, vc_h, b["block_tables"],
                                     b["context_lens"], 0.125)
        torch.cuda.synchronize()
        assert np.abs(out.cpu().numpy() - ref).max() <= 5e-3, step
        sched.complete_step()
    assert saw_preempt
    assert pk.photon_device_errors() == 0


def test_scheduler_steps_through_write_and_prefill():
    """A serving loop that attends every token the step computes (admitted
    prompts, recomputation after preemption, decode tokens): the scheduler's
    batch metadata drives the cache write and the tiled prefill over the
    batch's tokens; the oracle's causal definition on host copies agrees."""
    import torch
    pk = ensure_built()
    Hq, Hkv, d, bs, nb, width = 16, 4, 64, 16, 16, 16  # 16 blocks: the stream preempts once
    pool = pk.BlockPool(nb, seed=11)
    sched = pk.Scheduler(pool, max_running=6, max_step_tokens=300, max_blocks_per_seq=width)
    gen = torch.Generator(device="cuda").manual_seed(5)
    kc = (torch.randn((nb, Hkv, bs, d), generator=gen, device="cuda") * 0.5).bfloat16()
    vc = (torch.randn((nb, Hkv, bs, d), generator=gen, device="cuda") * 0.5).bfloat16()
    kc_h, vc_h = synth.to_storage_numpy(kc).copy(), synth.to_storage_numpy(vc).copy()
    rng = np.random.default_rng(1)
    for rid in range(12):
        sched.add_request(rid, int(rng.integers(3, 120)), int(rng.integers(2, 10)))
    saw_preempt = saw_prompt = False
    for step in range(16):
        b = sched.schedule()
        saw_preempt |= b["num_preempted"] > 0
        B, T = len(b["request_ids"]), len(b["token_seq"])
        if B == 0:
            sched.complete_step()
            continue
        saw_prompt |= max(b["num_new_tokens"]) > 1
        k = (torch.randn((T, Hkv, d), generator=gen, device="cuda") * 0.5).bfloat16()
        v = (torch.randn((T, Hkv, d), generator=gen, device="cuda") * 0.5).bfloat16()
        q = (torch.randn((T, Hq, d), generator=gen, device="cuda") * 0.5).bfloat16()
        ts = torch.from_numpy(np.ascontiguousarray(b["token_seq"], np.int32)).cuda()
        pos = torch.from_numpy(b["positions"]).cuda()
        pk.photon_kv_cache_write(k, v, pos, torch.from_numpy(b["slot_mapping"]).cuda(), kc, vc, 5e5)
        part, maxp = 32, int(b["positions"].max())
        n = pk.photon_paged_attention_workspace_size(T, Hq, d, maxp + 1, part)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
        out = torch.empty((T, Hq, d), device="cuda")
        pk.photon_paged_attention_prefill(q, ts, pos, kc, vc, torch.from_numpy(b["block_tables"]).cuda(),
                                          0.125, out, maxp, part, ws)
        oracle.kv_cache_write(synth.to_storage_numpy(k), synth.to_storage_numpy(v), b["positions"],
                              b["slot_mapping"], kc_h, vc_h, 5e5)
        ref = oracle.paged_attention_prefill(synth.to_storage_numpy(q), b["token_seq"], b["positions"],
                                             kc_h, vc_h, b["block_tables"], 0.125)
        torch.cuda.synchronize()
        assert np.abs(out.cpu().numpy() - ref).max() <= 5e-3, step
        sched.complete_step()
    assert saw_preempt and saw_prompt
    assert pk.photon_device_errors() == 0
