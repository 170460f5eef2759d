"""Device parity of the full decode step (write, split-K partial attention,
log-sum-exp merge) against the fp64 oracle on identical seeded inputs, for
the five workloads, the degenerate contexts, every compiled head shape, and
the block-table gather checked bit-exactly with tagged values.

Tolerances (max abs error of the fp32 output): 1e-5 with fp32 storage,
5e-3 with bf16 storage and fp32 accumulation.  bf16 output additionally
allows half a bf16 step of the oracle value (its own rounding)."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from tests.helpers import bf16_spacing, ensure_built, gpu_step, host_inputs, oracle_step

pytestmark = pytest.mark.gpu


def _tol(wl):
    return 1e-5 if wl.kv_dtype == "f32" else 5e-3


def _check(wl, vals_seed=None, partition_size=None, out_dtype=None, split_calls=False, rows=None,
           max_context_len=None):
    import torch
    vals = synth.make_values(wl, device="cuda", seed=vals_seed)
    h = host_inputs(wl, vals)
    ref, _, _, _ = oracle_step(wl, h)
    out, _ = gpu_step(wl, vals, partition_size=partition_size, out_dtype=out_dtype,
                      split_calls=split_calls, max_context_len=max_context_len)
    got = out.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got, ref = got[rows], ref[rows]
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    tol = _tol(wl)
    if out_dtype is not None and out_dtype == torch.bfloat16:
        tol = np.maximum(tol, bf16_spacing(ref) / 2 + 1e-6)
    assert (err <= tol).all(), f"max err {err.max():.3g}"
    import paged_kv_decode_write_gb300 as pk
    assert pk.photon_device_errors() == 0
    return float(err.max())


@pytest.mark.parametrize("name", ["tiny_fp32", "llama1b_single", "cb_batch16", "qwen3_ragged64"])
def test_workload_parity(name):
    _check(synth.make(name))


def test_llama_single_all_16_layers():
    import torch
    wl = synth.make("llama1b_single")
    vals = synth.make_values(wl, device="cuda")
    for layer in range(wl.num_layers):
        h = host_inputs(wl, vals, layer)
        ref, _, _, _ = oracle_step(wl, h)
        out, _ = gpu_step(wl, vals, layer=layer)
        assert np.abs(out.cpu().numpy() - ref).max() <= 5e-3


def test_longctx_b256_every_row():
    """The full-size 256-sequence step (about 9 GB of KV) as the benchmark
    runs it, every output row against the oracle: host copies of the pools
    are taken before the device write, the oracle writes the step's tokens
    into them in place and attends over all 256 sequences."""
    wl = synth.make("longctx_b256")
    vals = synth.make_values(wl, device="cuda")
    q, k, v = (synth.to_storage_numpy(vals[n][0]) for n in ("q", "k", "v"))
    kc = synth.to_storage_numpy(vals["k_cache"][0])   # host copies (device -> host)
    vc = synth.to_storage_numpy(vals["v_cache"][0])
    sm = oracle.slot_mapping(wl.block_tables, wl.token_seq, wl.positions, wl.block_size)
    oracle.kv_cache_write(k, v, wl.positions, sm, kc, vc, wl.rope_theta)
    ref = oracle.paged_attention(q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    del kc, vc
    out, _ = gpu_step(wl, vals)
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert (err <= 5e-3).all(), f"max err {err.max():.3g}"
    import paged_kv_decode_write_gb300 as pk
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("ctx", [[1], [15, 16, 17], [31, 32, 33], [511, 512, 513], [1024, 1025, 1],
                                 [2049, 7, 0, 300]])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_degenerate_contexts(ctx, dtype):
    wl = synth.make_custom(ctx, 8, 2, 64 if dtype == "bf16" else 32, kv_dtype=dtype, seed=sum(ctx),
                           value_std=1.0)
    _check(wl)


@pytest.mark.parametrize("d", [32, 64, 128, 256])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_head_shapes_bf16(d, G):
    wl = synth.make_custom([3, 200, 700], 2 * G, 2, d, kv_dtype="bf16", seed=d + G, value_std=0.5)
    _check(wl, partition_size=256)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_head_shapes_f32(d, G):
    wl = synth.make_custom([5, 130, 600], G, 1, d, kv_dtype="f32", seed=7 * d + G)
    _check(wl, partition_size=128)


@pytest.mark.parametrize("part", [16, 48, 128, 512, 4096])
def test_partition_sizes_agree(part):
    wl = synth.make_custom([1, 100, 1000, 3000], 32, 8, 64, kv_dtype="bf16", seed=11, value_std=0.5)
    _check(wl, partition_size=part)


@pytest.mark.parametrize("d,G", [(64, 1), (64, 4), (128, 2), (128, 8)])
@pytest.mark.parametrize("part", [16, 128])
def test_long_and_empty_contexts_mixed(d, G, part):
    """One long context among short and empty ones: the bf16 tensor-core
    decode's fixed partitions (hundreds for the long one with 16-token
    partitions, a single one for most others, empty contexts as zero rows)
    and the merge's partition counts.  The FP8 decode runs the same shapes
    through its page-balanced pieces (tests/test_gpu_fp8.py)."""
    rng = np.random.default_rng(31 + d + G + part)
    ctx = [0, 30000, 1, 17, 0] + rng.integers(1, 900, size=11).tolist() + [4097, 16, 0]
    wl = synth.make_custom(ctx, 2 * G, 2, d, kv_dtype="bf16", seed=d * G + part, value_std=0.5)
    _check(wl, partition_size=part)


@pytest.mark.parametrize("d,hq", [(64, 32), (128, 16)])
def test_l2_lookahead_path(d, hq):
    """64 sequences declared with a 32k maximum context: the page bound
    (64 x 2048 pages x 8 KV heads) exceeds 384 pages per resident warp, so
    the tensor-core kernel prefetches pages into L2 ahead of its ring.  The
    real contexts are short and ragged, and the 1024-token partitions make
    items longer than one 32-page block-table window."""
    rng = np.random.default_rng(21 + d)
    ctx = rng.integers(1, 1600, size=64)
    ctx[:6] = [1, 16, 512, 513, 1024, 1025]
    wl = synth.make_custom(ctx.tolist(), hq, 8, d, kv_dtype="bf16", seed=d, value_std=0.5,
                           partition_size=1024)
    pad = -np.ones((wl.num_seqs, 2048 - wl.max_blocks_per_seq), np.int32)
    wl = dataclasses.replace(wl, block_tables=np.concatenate([wl.block_tables, pad], axis=1))
    _check(wl, max_context_len=32768)


def test_split_calls_and_bf16_output():
    import torch
    wl = synth.make_custom([10, 900, 2000], 16, 8, 128, kv_dtype="bf16", seed=12, value_std=0.5)
    _check(wl, split_calls=True)
    _check(wl, out_dtype=torch.bfloat16)


def test_block_table_gather_is_bit_exact():
    """fp32 cache; in every sequence one token's key gives a score 1000 above
    all others, so the softmax weight is exactly 1 for it and exactly 0
    elsewhere: the output must equal that token's (index-tagged) V bit for bit,
    whatever partition it sits in."""
    import torch
    pk = ensure_built()
    ctx = [1, 17, 600, 1500]
    wl = synth.make_custom(ctx, 4, 2, 32, kv_dtype="f32", seed=5, tokens_per_seq=0)
    vals = synth.make_values(wl, device="cuda")
    kc, vc = vals["k_cache"][0], vals["v_cache"][0]
    kc.zero_()
    n = vc.numel()
    vc.copy_((torch.arange(n, device="cuda", dtype=torch.float64) % 8191 + 1).float().view_as(vc))
    q = torch.zeros_like(vals["q"][0])
    q[..., 0] = 1.0
    rng = np.random.default_rng(2)
    hot = [int(rng.integers(0, c)) for c in ctx]
    for s, j in enumerate(hot):
        b, o = wl.block_tables[s, j // 16], j % 16
        kc[b, :, o, 0] = 1000.0
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    out = torch.empty((4, 4, 32), device="cuda")
    ws_b = pk.photon_paged_attention_workspace_size(4, 4, 32, max(ctx), 512)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    pk.photon_paged_attention_decode(q, kc, vc, bt, cl, 1.0, out, max(ctx), 512, ws)
    for s, j in enumerate(hot):
        b, o = wl.block_tables[s, j // 16], j % 16
        for g in range(4):
            assert torch.equal(out[s, g], vc[b, g // 2, o]), (s, g)
    assert pk.photon_device_errors() == 0


def test_bad_block_id_is_skipped_and_flagged():
    import torch
    pk = ensure_built()
    wl = synth.make_custom([40], 4, 2, 64, kv_dtype="bf16", seed=1, tokens_per_seq=0)
    vals = synth.make_values(wl, device="cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    bt[0, 1] = wl.num_blocks + 5          # second page points outside the pool
    cl = torch.from_numpy(wl.context_lens).cuda()
    out = torch.empty((1, 4, 64), device="cuda")
    pk.photon_device_errors(clear=True)
    pk.photon_paged_attention_decode(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0], bt, cl,
                                     wl.scale, out, 40, 512, None)
    assert pk.photon_device_errors(clear=True) == pk.DEVERR_BLOCK_RANGE
    # the result is the oracle's attention over the pages that remained
    # (tokens 0-15 and 32-39): a block table without the bad page
    h = host_inputs(wl, vals)
    bt_kept = np.array([[wl.block_tables[0, 0], wl.block_tables[0, 2]]], np.int32)
    ref = oracle.paged_attention(h["q"], h["k_cache"], h["v_cache"], bt_kept,
                                 np.array([24], np.int32), wl.scale)
    assert np.abs(out.cpu().numpy() - ref).max() <= 5e-3


def test_context_beyond_bound_is_clamped_and_flagged():
    import torch
    pk = ensure_built()
    wl = synth.make_custom([64], 4, 2, 64, kv_dtype="bf16", seed=4, tokens_per_seq=0)
    vals = synth.make_values(wl, device="cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.tensor([64], dtype=torch.int32, device="cuda")
    out = torch.empty((1, 4, 64), device="cuda")
    pk.photon_device_errors(clear=True)
    # claims max_context_len 48: the device value 64 is clamped to 48
    pk.photon_paged_attention_decode(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0], bt, cl,
                                     wl.scale, out, 48, 512, None)
    assert pk.photon_device_errors(clear=True) & pk.DEVERR_CONTEXT_RANGE
    h = host_inputs(wl, vals)
    ref = oracle.paged_attention(h["q"], h["k_cache"], h["v_cache"], wl.block_tables,
                                 np.array([48], np.int32), wl.scale)
    assert np.abs(out.cpu().numpy() - ref).max() <= 5e-3


@pytest.mark.parametrize("d,hq,hkv", [(64, 32, 8), (128, 16, 8), (64, 8, 8), (128, 64, 8)])
def test_block_table_gather_is_bit_exact_bf16(d, hq, hkv):
    """bf16 cache (the tensor-core path for head_dim 64/128): one dominant key
    per (sequence, KV head) makes its softmax weight exactly 1 and all others
    exactly 0, so every output element must equal that token's V element bit
    for bit -- checking the permuted head-dim and token orders of the fragment
    loads, the 128-byte swizzle and the split-K merge."""
    import torch
    pk = ensure_built()
    ctx = [1, 17, 600, 1500, 16, 33]
    wl = synth.make_custom(ctx, hq, hkv, d, kv_dtype="bf16", seed=6, tokens_per_seq=0)
    vals = synth.make_values(wl, device="cuda")
    kc, vc = vals["k_cache"][0], vals["v_cache"][0]
    kc.zero_()
    n = vc.numel()
    idx = torch.arange(n, device="cuda", dtype=torch.int64)
    vc.copy_(((idx % 251) - 125).to(torch.bfloat16).view_as(vc))  # small integers: exact in bf16
    q = torch.zeros_like(vals["q"][0])
    q[..., 0] = 1.0
    rng = np.random.default_rng(3)
    hot = [[int(rng.integers(0, c)) for _ in range(hkv)] for c in ctx]
    for s, js in enumerate(hot):
        for h, j in enumerate(js):
            kc[wl.block_tables[s, j // 16], h, j % 16, 0] = 1000.0  # 2^-1442 underflows to 0
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    out = torch.empty((len(ctx), hq, d), device="cuda")
    part = 256
    ws_b = pk.photon_paged_attention_workspace_size(len(ctx), hq, d, max(ctx), part)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    pk.photon_paged_attention_decode(q, kc, vc, bt, cl, 1.0, out, max(ctx), part, ws)
    G = hq // hkv
    for s, js in enumerate(hot):
        for g in range(hq):
            j = js[g // G]
            ref = vc[wl.block_tables[s, j // 16], g // G, j % 16].float()
            assert torch.equal(out[s, g], ref), (s, g)
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("name,fp8", [("qwen3_ragged64", False), ("qwen3_ragged64", True),
                                      ("longctx_b256", False), ("longctx_b256", True)])
def test_decode_is_deterministic(name, fp8):
    """Each decode row comes from a fixed schedule of pages, pieces and merge
    order: repeated calls give bit-identical rows (bf16 partitions, FP8
    page-balanced pieces)."""
    import torch
    pk = ensure_built()
    wl = synth.make(name)
    if name == "longctx_b256":
        wl = synth.truncate(wl, 48)
    vals = (synth.make_values_fp8 if fp8 else synth.make_values)(wl, device="cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    part = wl.partition_size
    n = pk.photon_paged_attention_workspace_size(wl.num_seqs, wl.num_q_heads, wl.head_dim,
                                                 wl.max_context_len, part)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")

    def run():
        out = torch.full((wl.num_seqs, wl.num_q_heads, wl.head_dim), float("nan"), device="cuda")
        if fp8:
            pk.photon_paged_attention_decode_fp8(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0],
                                                 vals["k_scale"][0], vals["v_scale"][0], bt, cl,
                                                 wl.scale, out, wl.max_context_len, part, ws)
        else:
            pk.photon_paged_attention_decode(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0], bt,
                                             cl, wl.scale, out, wl.max_context_len, part, ws)
        torch.cuda.synchronize()
        return out

    first = run()
    assert torch.isfinite(first).all()
    for _ in range(4):
        assert torch.equal(run(), first)
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("d,dtype", [(32, "bf16"), (256, "bf16"), (64, "f32")])
def test_cuda_core_decode_is_deterministic(d, dtype):
    """The CUDA-core decode (fp32 pools; bf16 d 32 and 256), whose warps of a
    CTA split an item's pages and merge through shared memory: repeated
    calls give bit-identical rows."""
    import torch
    pk = ensure_built()
    rng = np.random.default_rng(d)
    ctx = rng.integers(1, 3000, size=24).tolist()
    wl = synth.make_custom(ctx, 16, 4, d, kv_dtype=dtype, seed=d, value_std=0.5, tokens_per_seq=0)
    vals = synth.make_values(wl, device="cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    n = pk.photon_paged_attention_workspace_size(wl.num_seqs, 16, d, wl.max_context_len, 256)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(4):
        out = torch.full((wl.num_seqs, 16, d), float("nan"), device="cuda")
        pk.photon_paged_attention_decode(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0], bt, cl,
                                         wl.scale, out, wl.max_context_len, 256, ws)
        torch.cuda.synchronize()
        outs.append(out)
    assert torch.isfinite(outs[0]).all()
    assert all(torch.equal(o, outs[0]) for o in outs[1:])
    assert pk.photon_device_errors() == 0


def _ctl_offset(wl, part):
    """Byte offset of the workspace's 16-byte control block (after the
    partials and the per-row piece counts with the mode word)."""
    al = lambda x: (x + 255) // 256 * 256
    rows = wl.num_seqs * wl.num_q_heads
    n = rows * (-(-wl.max_context_len // part) + 1)
    return 2 * al(n * 4) + al(n * wl.head_dim * 4) + (rows + 1 + 3) // 4 * 16


def test_dynamic_item_order_control_block():
    """With a workspace the tensor-core decode hands items out in dynamic
    order through a control block in the workspace.  With every byte of the
    workspace random before the first call (the block neither zero nor in
    use), every row matches the oracle; each call leaves the block zeroed;
    and replays of a CUDA graph of the call (the same arguments every time)
    give the eager call's rows bit for bit."""
    import torch
    pk = ensure_built()
    wl = synth.make("qwen3_ragged64")
    vals = synth.make_values(wl, device="cuda")
    h = host_inputs(wl, vals)
    ref = oracle.paged_attention(h["q"], h["k_cache"], h["v_cache"], wl.block_tables,
                                 wl.context_lens, wl.scale)
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    part = wl.partition_size
    n = pk.photon_paged_attention_workspace_size(wl.num_seqs, wl.num_q_heads, wl.head_dim,
                                                 wl.max_context_len, part)
    x = _ctl_offset(wl, part)
    assert x + 16 <= n
    gen = torch.Generator(device="cuda").manual_seed(5)
    ws = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=gen)
    stream = torch.cuda.Stream()

    def call(out):
        pk.photon_paged_attention_decode(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0], bt,
                                         cl, wl.scale, out, wl.max_context_len, part, ws)

    shape = (wl.num_seqs, wl.num_q_heads, wl.head_dim)
    out = torch.full(shape, float("nan"), device="cuda")
    with torch.cuda.stream(stream):
        call(out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= 5e-3
    assert not ws[x:x + 16].any()
    g = torch.cuda.CUDAGraph()
    out_g = torch.full(shape, float("nan"), device="cuda")
    with torch.cuda.graph(g, stream=stream):
        call(out_g)
    for _ in range(3):
        out_g.fill_(float("nan"))
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g, out)
        assert not ws[x:x + 16].any()
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("G", [2, 8])
def test_deep_ring_dynamic_order(G):
    """A d 128 batch whose declared context bound (32768 tokens) makes the
    launcher pick the two-warp, three-stage ring with the dynamic item order,
    while the actual contexts are short and ragged: every row against the
    oracle."""
    rng = np.random.default_rng(70 + G)
    ctx = rng.integers(1, 2500, size=24).tolist() + [0, 1, 16, 17]
    wl = synth.make_custom(ctx, 8 * G, 8, 128, kv_dtype="bf16", seed=G, value_std=0.5)
    # block-table rows wide enough for the declared bound (unused entries -1)
    bt = np.full((wl.num_seqs, 32768 // 16), -1, dtype=np.int32)
    bt[:, :wl.block_tables.shape[1]] = wl.block_tables
    wl = dataclasses.replace(wl, block_tables=bt)
    _check(wl, partition_size=512, max_context_len=32768)


@pytest.mark.parametrize("d,G", [(64, 4), (128, 2)])
def test_runs_of_empty_contexts_dynamic_order(d, G):
    """Hundreds of empty contexts between a few long ones on a full grid:
    long runs of items without pages (zero rows) fill the producer's
    32-entry ring of item records, which the consumer then drains; every
    row against the oracle."""
    rng = np.random.default_rng(d + G)
    ctx = [0] * 300
    for i in rng.choice(300, size=24, replace=False):
        ctx[i] = int(rng.integers(1, 3000))
    wl = synth.make_custom(ctx, 8 * G // 2, 4, d, kv_dtype="bf16", seed=d + G, value_std=0.5)
    bt = np.full((wl.num_seqs, 8192 // 16), -1, dtype=np.int32)
    bt[:, :wl.block_tables.shape[1]] = wl.block_tables
    wl = dataclasses.replace(wl, block_tables=bt)
    _check(wl, partition_size=128, max_context_len=8192)
