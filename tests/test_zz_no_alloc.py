"""photon_paged_attention_decode_static: the decode entry point for callers
that may not allocate device memory (for instance a plugin whose host
application owns the device-memory budget, or a serving loop where an
allocation could stall other streams).  Its split-K partials live in a fixed
scratch array inside the library.  Checked against
photon_paged_attention_decode with a caller workspace, on two calls in a row
(the second call reuses the array after the first left different data in it),
and for the size limit.  Collected last on purpose."""
import numpy as np
import pytest

import synth
from tests.helpers import ensure_built

pytestmark = pytest.mark.gpu


def _inputs(ctx, hq, hkv, d, seed):
    import torch
    wl = synth.make_custom(ctx, hq, hkv, d, kv_dtype="bf16", seed=seed, value_std=0.5,
                           tokens_per_seq=0)
    vals = synth.make_values(wl, device="cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    return wl, vals, bt, cl


def _with_workspace(pk, wl, vals, bt, cl, part):
    import torch
    n = pk.photon_paged_attention_workspace_size(wl.num_seqs, wl.num_q_heads, wl.head_dim,
                                                 wl.max_context_len, part)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    out = torch.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim), device="cuda")
    pk.photon_paged_attention_decode(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0], bt, cl,
                                     wl.scale, out, wl.max_context_len, part, ws)
    return out


def _static(pk, wl, vals, bt, cl, part):
    import torch
    out = torch.full((wl.num_seqs, wl.num_q_heads, wl.head_dim), float("nan"), device="cuda")
    pk.photon_paged_attention_decode_static(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0],
                                            bt, cl, wl.scale, out, wl.max_context_len, part)
    return out


def test_static_scratch_decode_matches_workspace_decode_twice():
    """Two calls in a row (the second finds the first's partials in the
    shared array): the same kernels as the workspace call, so the rows are
    bit-identical to it; and both are the oracle's attention within 5e-3."""
    import torch
    import oracle
    pk = ensure_built()
    cases = [([1, 700, 3000, 5000, 64], 32, 8, 64, 512, 1),
             ([9000, 17, 2500], 16, 8, 128, 256, 2)]
    for ctx, hq, hkv, d, part, seed in cases:
        wl, vals, bt, cl = _inputs(ctx, hq, hkv, d, seed)
        need = pk.photon_paged_attention_workspace_size(wl.num_seqs, hq, d, wl.max_context_len, part)
        assert 0 < need <= pk.STATIC_SCRATCH_BYTES
        ref = _with_workspace(pk, wl, vals, bt, cl, part)
        got = _static(pk, wl, vals, bt, cl, part)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
        want = oracle.paged_attention(synth.to_storage_numpy(vals["q"][0]),
                                      synth.to_storage_numpy(vals["k_cache"][0]),
                                      synth.to_storage_numpy(vals["v_cache"][0]),
                                      wl.block_tables, wl.context_lens, wl.scale)
        assert np.abs(got.cpu().numpy() - want).max() <= 5e-3
    assert pk.photon_device_errors() == 0


def test_static_scratch_decode_allocates_nothing():
    """After a first call (which looks up the array's address), further calls
    leave the device's free memory and torch's allocator untouched."""
    import torch
    pk = ensure_built()
    wl, vals, bt, cl = _inputs([2000, 40, 1300, 700], 32, 8, 64, 4)
    out = torch.empty((wl.num_seqs, 32, 64), device="cuda")
    call = lambda: pk.photon_paged_attention_decode_static(vals["q"][0], vals["k_cache"][0],
                                                           vals["v_cache"][0], bt, cl, wl.scale, out,
                                                           wl.max_context_len, 256)
    call()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    torch0 = torch.cuda.memory_allocated()
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == torch0
    assert pk.photon_device_errors() == 0


def test_static_scratch_rejects_requests_beyond_its_size():
    import torch
    pk = ensure_built()
    # 64 sequences x 32 heads x 64 partitions x (64 + 2) floats > 32 MiB
    wl, vals, bt, cl = _inputs([32768] + [16] * 63, 32, 8, 64, 3)
    need = pk.photon_paged_attention_workspace_size(64, 32, 64, 32768, 512)
    assert need > pk.STATIC_SCRATCH_BYTES
    out = torch.zeros((64, 32, 64), device="cuda")
    with pytest.raises(pk.PhotonError) as e:
        pk.photon_paged_attention_decode_static(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0],
                                                bt, cl, wl.scale, out, 32768, 512)
    assert e.value.status == -3
    torch.cuda.synchronize()
    assert float(out.abs().max()) == 0.0  # nothing was launched


def test_static_scratch_checks_arguments_before_the_size():
    """A request both too large for the array and malformed gets the
    argument's status, not the size one."""
    import torch
    pk = ensure_built()
    lib = pk.lib()
    q = torch.zeros((64, 32, 64), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((8, 8, 16, 64), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((64, 2048), dtype=torch.int32, device="cuda")
    cl = torch.ones(64, dtype=torch.int32, device="cuda")
    out = torch.zeros((64, 32, 64), device="cuda")
    p = lambda t: t.data_ptr()
    args = lambda hkv, hd: (p(q), p(kv), p(kv), p(bt), p(cl), 0.125, p(out), 64, 32, hkv, hd, 16, 8,
                            2048, 32768, 512, pk.BF16, pk.F32, None)
    assert lib.photon_paged_attention_decode_static(*args(8, 64)) == -3   # valid, too large
    assert lib.photon_paged_attention_decode_static(*args(7, 64)) == -1   # 32 % 7 != 0
    assert lib.photon_paged_attention_decode_static(*args(8, 96)) == -2   # head_dim 96
    torch.cuda.synchronize()
    assert float(out.abs().max()) == 0.0
