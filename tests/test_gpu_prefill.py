"""Paged prefill (causal attention of newly written prompt tokens over their
pages) on the device against the oracle's causal definition: whole prompts of
admitted requests, a chunk continuing a cached prefix, every storage path."""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import ensure_built

pytestmark = pytest.mark.gpu


def _prefill(pk, wl, vals, q, part, out_dtype=None):
    import torch
    ts = torch.from_numpy(wl.token_seq).cuda()
    pos = torch.from_numpy(wl.positions).cuda()
    bt = torch.from_numpy(wl.block_tables).cuda()
    maxp = int(wl.positions.max())
    n = pk.photon_paged_attention_workspace_size(wl.num_tokens, wl.num_q_heads, wl.head_dim, maxp + 1, part)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    out = torch.full((wl.num_tokens, wl.num_q_heads, wl.head_dim), float("nan"),
                     dtype=torch.float32 if out_dtype is None else out_dtype, device="cuda")
    pk.photon_paged_attention_prefill(q, ts, pos, vals["k_cache"][0], vals["v_cache"][0], bt,
                                      wl.scale, out, maxp, part, ws)
    torch.cuda.synchronize()
    return out


def _write(pk, wl, vals):
    import torch
    sm = pk.photon_slot_mapping(wl.block_tables, wl.token_seq, wl.positions)
    pk.photon_kv_cache_write(vals["k"][0], vals["v"][0], torch.from_numpy(wl.positions).cuda(),
                             torch.from_numpy(sm).cuda(), vals["k_cache"][0], vals["v_cache"][0],
                             wl.rope_theta)
    return sm


@pytest.mark.parametrize("part", [64, 512])
def test_prefill_of_admitted_prompts(part):
    """The continuous-batching step with 4 admitted 100-token prompts: after the
    write, every written token's causal attention (prompt and decode token)."""
    import torch
    pk = ensure_built()
    wl = synth.make("cb_batch16", seed=6)
    vals = synth.make_values(wl, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(11)
    q = (torch.randn((wl.num_tokens, wl.num_q_heads, wl.head_dim), generator=g, device="cuda") * 0.5).bfloat16()
    kc = synth.to_storage_numpy(vals["k_cache"][0]).copy()
    vc = synth.to_storage_numpy(vals["v_cache"][0]).copy()
    sm = _write(pk, wl, vals)
    oracle.kv_cache_write(synth.to_storage_numpy(vals["k"][0]), synth.to_storage_numpy(vals["v"][0]),
                          wl.positions, sm, kc, vc, wl.rope_theta)
    got = _prefill(pk, wl, vals, q, part).cpu().numpy()
    ref = oracle.paged_attention_prefill(synth.to_storage_numpy(q), wl.token_seq, wl.positions, kc, vc,
                                         wl.block_tables, wl.scale)
    assert np.isfinite(got).all() and np.abs(got - ref).max() <= 5e-3
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("bf16", 32), ("f32", 32), ("f32", 64)])
def test_chunked_prefill_over_a_cached_prefix(dtype, d):
    """Sequence 0 has 300 tokens cached and writes a 128-token chunk
    (positions 300..427); sequence 1 writes a 20-token prompt."""
    import torch
    pk = ensure_built()
    tol = 1e-5 if dtype == "f32" else 5e-3
    wl = synth.make_custom([428, 20], 8, 2, d, kv_dtype=dtype, seed=d, value_std=0.5)
    pos = np.concatenate([np.arange(300, 428), np.arange(20)]).astype(np.int32)
    ts = np.concatenate([np.zeros(128), np.ones(20)]).astype(np.int32)
    wl = synth.Workload(**{**wl.__dict__, "positions": pos, "token_seq": ts})
    vals = synth.make_values(wl, device="cuda")
    kc = synth.to_storage_numpy(vals["k_cache"][0]).copy()
    vc = synth.to_storage_numpy(vals["v_cache"][0]).copy()
    sm = _write(pk, wl, vals)
    oracle.kv_cache_write(synth.to_storage_numpy(vals["k"][0]), synth.to_storage_numpy(vals["v"][0]),
                          wl.positions, sm, kc, vc, wl.rope_theta)
    q = vals["k"][0].repeat_interleave(4, dim=1).contiguous()  # any [T, H_q, d] queries
    got = _prefill(pk, wl, vals, q, 128).cpu().numpy()
    ref = oracle.paged_attention_prefill(synth.to_storage_numpy(q), ts, pos, kc, vc, wl.block_tables,
                                         wl.scale)
    assert np.isfinite(got).all() and np.abs(got - ref).max() <= tol
    assert pk.photon_device_errors() == 0


def test_prefill_bad_sequence_row_gives_zero_and_flags():
    import torch
    pk = ensure_built()
    wl = synth.make_custom([40], 4, 2, 64, kv_dtype="bf16", seed=2, tokens_per_seq=3)
    vals = synth.make_values(wl, device="cuda")
    wl = synth.Workload(**{**wl.__dict__, "token_seq": np.array([0, 5, 0], np.int32)})
    pk.photon_device_errors(clear=True)
    out = _prefill(pk, wl, vals, vals["q"][0][:1].repeat(3, 1, 1).contiguous(), 512)
    assert pk.photon_device_errors(clear=True) & pk.DEVERR_BLOCK_RANGE
    assert float(out[1].abs().max()) == 0.0 and torch.isfinite(out).all()
