"""Paged prefill (causal attention of newly written prompt tokens over their
pages) on the device against the oracle's causal definition: whole prompts of
admitted requests, a chunk continuing a cached prefix, every storage path."""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import bf16_spacing, ensure_built

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


def _prefill_case(pk, ctx, spans, hq, hkv, d, seed, part, order=None, out_dtype=None):
    """Writes the span tokens (sequence, first, end positions) of a custom
    workload, runs the prefill of those tokens (in `order` if given) and
    returns (device result, oracle result)."""
    import torch
    wl = synth.make_custom(ctx, hq, hkv, d, kv_dtype="bf16", seed=seed, value_std=0.5)
    ts = np.concatenate([np.full(e - b, s) for s, b, e in spans]).astype(np.int32)
    pos = np.concatenate([np.arange(b, e) for s, b, e in spans]).astype(np.int32)
    if order is not None:
        ts, pos = ts[order], pos[order]
    wl = synth.Workload(**{**wl.__dict__, "positions": pos, "token_seq": ts})
    vals = synth.make_values(wl, device="cuda")
    kc = synth.to_storage_numpy(vals["k_cache"][0]).copy()
    vc = synth.to_storage_numpy(vals["v_cache"][0]).copy()
    sm = _write(pk, wl, vals)
    oracle.kv_cache_write(synth.to_storage_numpy(vals["k"][0]), synth.to_storage_numpy(vals["v"][0]),
                          wl.positions, sm, kc, vc, wl.rope_theta)
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = (torch.randn((len(ts), hq, d), generator=g, device="cuda") * 0.5).bfloat16()
    got = _prefill(pk, wl, vals, q, part, out_dtype).float().cpu().numpy()
    ref = oracle.paged_attention_prefill(synth.to_storage_numpy(q), ts, pos, kc, vc, wl.block_tables,
                                         wl.scale)
    return got, ref


@pytest.mark.parametrize("part", [64, 512])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_tiled_prefill_mixed_batch(d, G, part):
    """Tiled tensor-core prefill: a 150-token chunk over a 700-token cached
    prefix, prompts of 37 and 5 tokens, two decode tokens and a 100-token
    chunk at 1100, so row tiles hold one or several sequences, end ragged,
    and long rows span several partitions (partials + merge)."""
    pk = ensure_built()
    ctx = [850, 37, 5, 300, 64, 1200]
    spans = [(0, 700, 850), (1, 0, 37), (2, 0, 5), (3, 299, 300), (4, 63, 64), (5, 1100, 1200)]
    got, ref = _prefill_case(pk, ctx, spans, 2 * G, 2, d, seed=d + G + part, part=part)
    assert np.isfinite(got).all() and np.abs(got - ref).max() <= 5e-3
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("G", [1, 4])
def test_tiled_prefill_interleaved_tokens(G):
    """Two prompts whose tokens alternate in the batch: every row-tile segment
    is one token, and the same sequence recurs within a tile."""
    pk = ensure_built()
    spans = [(0, 0, 40), (1, 0, 40)]
    order = np.stack([np.arange(40), 40 + np.arange(40)], axis=1).reshape(-1)
    got, ref = _prefill_case(pk, [40, 40], spans, 2 * G, 2, 64, seed=3, part=16, order=order)
    assert np.abs(got - ref).max() <= 5e-3
    assert pk.photon_device_errors() == 0


def test_tiled_prefill_bf16_output():
    import torch
    pk = ensure_built()
    got, ref = _prefill_case(pk, [600, 90], [(0, 500, 600), (1, 0, 90)], 32, 8, 128, seed=5, part=128,
                             out_dtype=torch.bfloat16)
    assert (np.abs(got - ref) <= np.maximum(5e-3, bf16_spacing(ref) / 2 + 1e-6)).all()


def test_prefill_bad_row_spanning_partitions_gives_zero():
    """A token with an out-of-range sequence row at a position past several
    partitions: its row is zero (the merge must not combine partials that
    were never written); the other tokens are unaffected."""
    import torch
    pk = ensure_built()
    wl = synth.make_custom([60], 8, 2, 64, kv_dtype="bf16", seed=8, tokens_per_seq=4)
    vals = synth.make_values(wl, device="cuda")
    kc = synth.to_storage_numpy(vals["k_cache"][0]).copy()
    vc = synth.to_storage_numpy(vals["v_cache"][0]).copy()
    sm = _write(pk, wl, vals)
    oracle.kv_cache_write(synth.to_storage_numpy(vals["k"][0]), synth.to_storage_numpy(vals["v"][0]),
                          wl.positions, sm, kc, vc, wl.rope_theta)
    ts = np.array([0, 7, 0, 0], np.int32)
    wl = synth.Workload(**{**wl.__dict__, "token_seq": ts})
    q = vals["q"][0][:1].repeat(4, 1, 1).contiguous()
    pk.photon_device_errors(clear=True)
    out = _prefill(pk, wl, vals, q, 16)
    assert pk.photon_device_errors(clear=True) & pk.DEVERR_BLOCK_RANGE
    assert float(out[1].abs().max()) == 0.0
    good = [0, 2, 3]
    ref = oracle.paged_attention_prefill(synth.to_storage_numpy(q)[good], ts[good], wl.positions[good],
                                         kc, vc, wl.block_tables, wl.scale)
    assert np.abs(out.cpu().numpy()[good] - ref).max() <= 5e-3


def test_tiled_prefill_positions_beyond_the_bound_are_clamped():
    """Positions past the declared max_position are clamped to it (context
    max_position + 1) and flagged PHOTON_DEVERR_CONTEXT_RANGE."""
    import torch
    pk = ensure_built()
    wl = synth.make_custom([60], 8, 2, 64, kv_dtype="bf16", seed=12, tokens_per_seq=20)
    vals = synth.make_values(wl, device="cuda")
    kc = synth.to_storage_numpy(vals["k_cache"][0]).copy()
    vc = synth.to_storage_numpy(vals["v_cache"][0]).copy()
    sm = _write(pk, wl, vals)
    oracle.kv_cache_write(synth.to_storage_numpy(vals["k"][0]), synth.to_storage_numpy(vals["v"][0]),
                          wl.positions, sm, kc, vc, wl.rope_theta)
    maxp, part = 49, 16
    q = vals["q"][0][:1].repeat(wl.num_tokens, 1, 1).contiguous()
    ts = torch.from_numpy(wl.token_seq).cuda()
    pos = torch.from_numpy(wl.positions).cuda()
    bt = torch.from_numpy(wl.block_tables).cuda()
    n = pk.photon_paged_attention_workspace_size(wl.num_tokens, wl.num_q_heads, 64, maxp + 1, part)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    out = torch.full((wl.num_tokens, wl.num_q_heads, 64), float("nan"), device="cuda")
    pk.photon_device_errors(clear=True)
    pk.photon_paged_attention_prefill(q, ts, pos, vals["k_cache"][0], vals["v_cache"][0], bt, wl.scale,
                                      out, maxp, part, ws)
    assert pk.photon_device_errors(clear=True) & pk.DEVERR_CONTEXT_RANGE
    ref = oracle.paged_attention_prefill(synth.to_storage_numpy(q), wl.token_seq,
                                         np.minimum(wl.positions, maxp), kc, vc, wl.block_tables, wl.scale)
    assert np.abs(out.cpu().numpy() - ref).max() <= 5e-3


def test_tiled_prefill_long_batch_coarsened_partitions():
    """A long batch (3072 query tokens, 8 KV heads: the tcgen05 kernel's
    route): two whole 1024-token prompts and a 1024-token chunk at
    3900..4923 that crosses position 4096, with the caller's 64-token
    partitions.  A seeded sample of rows, including both sides of 4096,
    against the oracle."""
    import torch
    pk = ensure_built()
    ctx = [1024, 1024, 4924]
    spans = [(0, 0, 1024), (1, 0, 1024), (2, 3900, 4924)]
    wl = synth.make_custom(ctx, 32, 8, 64, kv_dtype="bf16", seed=31, value_std=0.5)
    ts = np.concatenate([np.full(e - b, s) for s, b, e in spans]).astype(np.int32)
    pos = np.concatenate([np.arange(b, e) for s, b, e in spans]).astype(np.int32)
    wl = synth.Workload(**{**wl.__dict__, "positions": pos, "token_seq": ts})
    vals = synth.make_values(wl, device="cuda")
    sm = _write(pk, wl, vals)
    kc = synth.to_storage_numpy(vals["k_cache"][0])
    vc = synth.to_storage_numpy(vals["v_cache"][0])
    g = torch.Generator(device="cuda").manual_seed(3)
    q = (torch.randn((len(ts), 32, 64), generator=g, device="cuda") * 0.5).bfloat16()
    got = _prefill(pk, wl, vals, q, 64).cpu().numpy()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.choice(len(ts), 120, replace=False),
                                     np.nonzero((pos >= 4090) & (pos <= 4100))[0], [0, 1023, len(ts) - 1]]))
    ref = oracle.paged_attention_prefill(synth.to_storage_numpy(q)[rows], ts[rows], pos[rows], kc, vc,
                                         wl.block_tables, wl.scale)
    assert np.isfinite(got).all() and np.abs(got[rows] - ref).max() <= 5e-3
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("seed", range(6))
def test_tiled_prefill_random_layouts(seed):
    """Seeded random batches for the tiled kernel: sequence count, contexts,
    which tokens are new (whole prompts, chunks over a cached prefix, single
    decode tokens), token order (sequence-contiguous or shuffled), head
    grouping, head_dim and partition size all drawn at random."""
    pk = ensure_built()
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 7))
    G = int(rng.choice([1, 2, 4, 8]))
    d = int(rng.choice([64, 128]))
    hkv = int(rng.choice([1, 2, 4]))
    part = int(rng.choice([16, 64, 256, 512]))
    ctx, spans = [], []
    for s in range(B):
        kind = rng.integers(0, 3)
        c = int(rng.integers(1, 700))
        n = c if kind == 0 else (1 if kind == 1 else int(rng.integers(1, c + 1)))
        ctx.append(c)
        spans.append((s, c - n, c))
    T = sum(e - b for _, b, e in spans)
    order = rng.permutation(T) if rng.random() < 0.3 else None
    got, ref = _prefill_case(pk, ctx, spans, hkv * G, hkv, d, seed=seed, part=part, order=order)
    assert np.isfinite(got).all() and np.abs(got - ref).max() <= 5e-3, (B, G, d, hkv, part, order is None)
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 64), (16, 8, 128)])
def test_tiled_prefill_bench_long_prompts_sampled_rows(hq, hkv, d):
    """The benchmark's long-prompt prefill as it times it (the tcgen05
    kernel): 8 whole 2048-token prompts, partition 512, Llama heads (d 64)
    and Qwen3 heads (d 128).  A seeded sample of rows -- every prompt's
    first and last token, tokens around each 128-key tile boundary, random
    others -- against the oracle."""
    import torch
    pk = ensure_built()
    wl = synth.make_custom([2048] * 8, hq, hkv, d, kv_dtype="bf16", seed=1, value_std=0.5,
                           tokens_per_seq=2048)
    vals = synth.make_values(wl, device="cuda")
    _write(pk, wl, vals)
    kc = synth.to_storage_numpy(vals["k_cache"][0])
    vc = synth.to_storage_numpy(vals["v_cache"][0])
    g = torch.Generator(device="cuda").manual_seed(d)
    q = (torch.randn((wl.num_tokens, hq, d), generator=g, device="cuda") * 0.5).bfloat16()
    got = _prefill(pk, wl, vals, q, 512).cpu().numpy()
    pos, ts = wl.positions, wl.token_seq
    rng = np.random.default_rng(d)
    edges = np.nonzero((pos == 0) | (pos == 2047) | np.isin(pos % 512, [0, 511]))[0]
    rows = np.unique(np.concatenate([rng.choice(wl.num_tokens, 96, replace=False),
                                     rng.choice(edges, 48, replace=False)]))
    ref = oracle.paged_attention_prefill(synth.to_storage_numpy(q)[rows], ts[rows], pos[rows], kc, vc,
                                         wl.block_tables, wl.scale)
    assert np.isfinite(got).all() and np.abs(got[rows] - ref).max() <= 5e-3
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 64), (16, 8, 128)])
def test_tc_prefill_long_prompts_are_deterministic(hq, hkv, d):
    """The long-prompt tcgen05 prefill computes every output with a fixed
    order of operations, so repeated calls give bit-identical rows.  (A race
    between the two key halves of a row -- one half's probabilities written
    over TMEM columns whose scores the other half had not read yet -- once
    showed here as rows differing by up to 0.02 between calls while a sample
    of rows still matched the oracle.)"""
    import torch
    pk = ensure_built()
    wl = synth.make_custom([2048] * 8, hq, hkv, d, kv_dtype="bf16", seed=3, value_std=0.5,
                           tokens_per_seq=2048)
    vals = synth.make_values(wl, device="cuda")
    _write(pk, wl, vals)
    g = torch.Generator(device="cuda").manual_seed(7 + d)
    q = (torch.randn((wl.num_tokens, hq, d), generator=g, device="cuda") * 0.5).bfloat16()
    first = _prefill(pk, wl, vals, q, 512).clone()
    assert torch.isfinite(first).all()
    for _ in range(6):
        assert torch.equal(_prefill(pk, wl, vals, q, 512), first)
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("G,d", [(4, 64), (2, 128), (8, 64)])
def test_tiled_prefill_is_deterministic(G, d):
    """The mma.sync tiled prefill (batches too small for the tcgen05 kernel):
    repeated calls give bit-identical rows."""
    import torch
    pk = ensure_built()
    hkv = 2
    spans = [(0, 0, 300), (1, 200, 260), (2, 0, 40), (3, 500, 900)]
    assert not _tc_route(pk, sum(e - b for _, b, e in spans), G, hkv)
    wl = synth.make_custom([300, 260, 40, 900], G * hkv, hkv, d, kv_dtype="bf16", seed=G + d, value_std=0.5)
    ts = np.concatenate([np.full(e - b, s_) for s_, b, e in spans]).astype(np.int32)
    pos = np.concatenate([np.arange(b, e) for _, b, e in spans]).astype(np.int32)
    wl = synth.Workload(**{**wl.__dict__, "positions": pos, "token_seq": ts})
    vals = synth.make_values(wl, device="cuda")
    _write(pk, wl, vals)
    g = torch.Generator(device="cuda").manual_seed(d)
    q = (torch.randn((wl.num_tokens, G * hkv, d), generator=g, device="cuda") * 0.5).bfloat16()
    first = _prefill(pk, wl, vals, q, 128).clone()
    assert torch.isfinite(first).all()
    for _ in range(4):
        assert torch.equal(_prefill(pk, wl, vals, q, 128), first)
    assert pk.photon_device_errors() == 0


# ---------------------------------------------------------------- tcgen05 kernel
# Batches whose 128-row tiles (128 / G query tokens x G heads) times the KV
# heads give every SM an item run on the tcgen05 / TMEM kernel; each test
# below asserts that its batch is that large.

def _tc_route(pk, num_tokens, G, hkv):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return -(-num_tokens // (128 // G)) * hkv >= sms


def _tc_spans(G, extra=0):
    """Chunks over cached prefixes, whole prompts of odd lengths and decode
    tokens, sized in 128 / G token tiles so that tiles hold one or several
    sequences and end ragged."""
    R = 128 // G
    spans = [(0, 700, 700 + 8 * R + 5), (1, 0, 5 * R + 37), (2, 299, 300), (3, 0, 3),
             (4, 1100, 1100 + 6 * R + extra), (5, 63, 64), (6, 0, R + 11)]
    ctx = [e for _, _, e in spans]
    return ctx, spans


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_tc_prefill_mixed_batch_every_row(d, G):
    pk = ensure_built()
    ctx, spans = _tc_spans(G)
    T = sum(e - b for _, b, e in spans)
    assert _tc_route(pk, T, G, 8)
    got, ref = _prefill_case(pk, ctx, spans, 8 * G, 8, d, seed=40 + d + G, part=128)
    err = np.abs(got - ref)
    assert np.isfinite(got).all() and err.max() <= 5e-3, err.max()
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("G", [2, 8])
def test_tc_prefill_interleaved_and_shuffled_tokens(G):
    """Tokens of three prompts in a shuffled order: tiles hold many one-token
    runs and the same sequence recurs within a tile."""
    pk = ensure_built()
    R = 128 // G
    n = 8 * R
    spans = [(0, 0, n), (1, 0, n), (2, 40, 40 + n)]
    T = 3 * n
    assert _tc_route(pk, T, G, 8)
    order = np.random.default_rng(G).permutation(T)
    got, ref = _prefill_case(pk, [n, n, 40 + n], spans, 8 * G, 8, 64, seed=50 + G, part=64,
                             order=order)
    assert np.isfinite(got).all() and np.abs(got - ref).max() <= 5e-3
    assert pk.photon_device_errors() == 0


def test_tc_prefill_bf16_output():
    import torch
    pk = ensure_built()
    ctx, spans = _tc_spans(4)
    T = sum(e - b for _, b, e in spans)
    assert _tc_route(pk, T, 4, 8)
    got, ref = _prefill_case(pk, ctx, spans, 32, 8, 128, seed=61, part=512, out_dtype=torch.bfloat16)
    assert (np.abs(got - ref) <= np.maximum(5e-3, bf16_spacing(ref) / 2 + 1e-6)).all()


def test_tc_prefill_bad_rows_and_clamped_positions():
    """A long batch with tokens naming a sequence row past the table (zero
    rows, PHOTON_DEVERR_BLOCK_RANGE), negative positions (empty contexts:
    zero rows) and positions past the declared bound (clamped,
    PHOTON_DEVERR_CONTEXT_RANGE); every other row equals the oracle."""
    import torch
    pk = ensure_built()
    G, hkv, d = 4, 8, 64
    ctx, spans = _tc_spans(G)
    wl = synth.make_custom(ctx, G * hkv, hkv, d, kv_dtype="bf16", seed=71, value_std=0.5)
    ts = np.concatenate([np.full(e - b, s) for s, b, e in spans]).astype(np.int32)
    pos = np.concatenate([np.arange(b, e) for s, b, e in spans]).astype(np.int32)
    wl = synth.Workload(**{**wl.__dict__, "positions": pos, "token_seq": ts})
    assert _tc_route(pk, len(ts), G, hkv)
    vals = synth.make_values(wl, device="cuda")
    kc = synth.to_storage_numpy(vals["k_cache"][0]).copy()
    vc = synth.to_storage_numpy(vals["v_cache"][0]).copy()
    sm = _write(pk, wl, vals)
    oracle.kv_cache_write(synth.to_storage_numpy(vals["k"][0]), synth.to_storage_numpy(vals["v"][0]),
                          pos, sm, kc, vc, wl.rope_theta)
    rng = np.random.default_rng(7)
    bad = rng.choice(len(ts), 9, replace=False)
    ts_dev = ts.copy()
    ts_dev[bad] = wl.num_seqs + 3
    # negative positions: empty contexts, zero rows -- scattered ones, and a
    # whole run (the 1100.. chunk's first 40 tokens) whose tiles have no keys
    neg = np.setdiff1d(np.concatenate([rng.choice(len(ts), 5, replace=False),
                                       np.nonzero(pos >= 1100)[0][:40]]), bad)
    pos_dev = pos.copy()
    pos_dev[neg] = -1
    maxp = 1000                       # positions of the 1100.. chunk exceed it
    g = torch.Generator(device="cuda").manual_seed(7)
    q = (torch.randn((len(ts), G * hkv, d), generator=g, device="cuda") * 0.5).bfloat16()
    n = pk.photon_paged_attention_workspace_size(len(ts), G * hkv, d, maxp + 1, 128)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    out = torch.full((len(ts), G * hkv, d), float("nan"), device="cuda")
    pk.photon_device_errors(clear=True)
    pk.photon_paged_attention_prefill(q, torch.from_numpy(ts_dev).cuda(), torch.from_numpy(pos_dev).cuda(),
                                      vals["k_cache"][0], vals["v_cache"][0],
                                      torch.from_numpy(wl.block_tables).cuda(), wl.scale, out, maxp,
                                      128, ws)
    flags = pk.photon_device_errors(clear=True)
    assert flags & pk.DEVERR_BLOCK_RANGE and flags & pk.DEVERR_CONTEXT_RANGE
    got = out.cpu().numpy()
    assert (got[bad] == 0).all() and (got[neg] == 0).all()
    good = np.setdiff1d(np.arange(len(ts)), np.concatenate([bad, neg]))
    ref = oracle.paged_attention_prefill(synth.to_storage_numpy(q)[good], ts[good],
                                         np.minimum(pos[good], maxp), kc, vc, wl.block_tables,
                                         wl.scale)
    assert np.isfinite(got).all() and np.abs(got[good] - ref).max() <= 5e-3
