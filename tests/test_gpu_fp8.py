"""FP8 (E4M3) KV cache: the quantising write and the tensor-core decode over
FP8 pools, against the oracle's FP8 definitions (exact E4M3 encode/decode,
pinned against torch's float8 type) on identical seeded inputs."""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import bf16_spacing, ensure_built

pytestmark = pytest.mark.gpu


def _fp8_step_values(name, seed=0, ctx=None):
    wl = synth.make(name, seed=seed) if ctx is None else synth.make_custom(
        ctx, 32, 8, 64, kv_dtype="bf16", seed=seed, value_std=0.5)
    return wl, synth.make_values_fp8(wl, device="cuda")


@pytest.mark.parametrize("name", ["cb_batch16", "llama1b_single"])
def test_fp8_write_matches_oracle(name):
    import torch
    pk = ensure_built()
    wl, vals = _fp8_step_values(name, seed=2)
    kc_h = vals["k_cache"][0].cpu().numpy().copy()
    vc_h = vals["v_cache"][0].cpu().numpy().copy()
    ks, vs = vals["k_scale"][0].cpu().numpy(), vals["v_scale"][0].cpu().numpy()
    sm = oracle.slot_mapping(wl.block_tables, wl.token_seq, wl.positions, 16)
    oracle.kv_cache_write_fp8(synth.to_storage_numpy(vals["k"][0]), synth.to_storage_numpy(vals["v"][0]),
                              wl.positions, sm, kc_h, vc_h, ks, vs, wl.rope_theta)
    pk.photon_kv_cache_write_fp8(vals["k"][0], vals["v"][0], torch.from_numpy(wl.positions).cuda(),
                                 torch.from_numpy(sm).cuda(), vals["k_cache"][0], vals["v_cache"][0],
                                 vals["k_scale"][0], vals["v_scale"][0], wl.rope_theta)
    torch.cuda.synchronize()
    kc, vc = vals["k_cache"][0].cpu().numpy(), vals["v_cache"][0].cpu().numpy()
    assert np.array_equal(vc, vc_h)                      # V codes bit-exact
    diff = kc.astype(np.int32) - kc_h.astype(np.int32)   # K codes: same sign, at most one step
    assert (np.abs(diff) <= 1).all() and ((kc ^ kc_h) & 0x80 == 0).all()
    assert (diff != 0).mean() < 1e-3
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_write_codes_on_exact_midpoints(d):
    """fp32 inputs whose quotient by the head's scale is exactly a midpoint of
    two E4M3 values (scales of 19 significant bits, so no reciprocal is
    exact), a hair beside one, or random: K (no rotation) and V codes must
    equal the oracle's, the nearest E4M3 of the exact quotient with ties to
    the even code, bit for bit."""
    import torch
    pk = ensure_built()
    rng = np.random.default_rng(40 + d)
    H, T, bs, nb = 8, 48, 16, 8
    vals = sorted({oracle.fp8_decode(c) for c in range(0x7E + 1)})
    mids = np.array([(a + b) / 2 for a, b in zip(vals, vals[1:])])
    scales = np.array([float(int(rng.integers(2 ** 18, 2 ** 19)) | 1) * 2.0 ** -24 for _ in range(H)])
    assert (scales.astype(np.float32) == scales).all()
    m = mids[rng.integers(0, len(mids), size=(T, H, d))] * rng.choice([-1.0, 1.0], size=(T, H, d))
    x = m * scales[None, :, None]                       # exact midpoints times the scale
    near = rng.random((T, H, d)) < 0.25                 # a hair beside the midpoint
    x = np.where(near, x * (1 + rng.choice([-1, 1], size=x.shape) * 2.0 ** -22), x)
    rnd = rng.random((T, H, d)) < 0.25                  # and random values
    x = np.where(rnd, rng.standard_normal(x.shape) * scales[None, :, None] * 100, x)
    k = x.astype(np.float32)
    assert (k[~near & ~rnd] == x[~near & ~rnd]).all()  # midpoints exact in float
    v = (-k).copy()
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    pos = rng.integers(0, 5000, size=T).astype(np.int32)
    sc = scales.astype(np.float32)
    kc_h = np.full((nb, H, bs, d), 0x5A, np.uint8)
    vc_h = np.full((nb, H, d, bs), 0x5A, np.uint8)
    oracle.kv_cache_write_fp8(k, v, pos, slots, kc_h, vc_h, sc, sc, 1e4, oracle.ROPE_NONE)
    kc = torch.from_numpy(np.full((nb, H, bs, d), 0x5A, np.uint8)).cuda()
    vc = torch.from_numpy(np.full((nb, H, d, bs), 0x5A, np.uint8)).cuda()
    sc_t = torch.from_numpy(sc).cuda()
    pk.photon_kv_cache_write_fp8(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                                 torch.from_numpy(pos).cuda(), torch.from_numpy(slots).cuda(), kc, vc,
                                 sc_t, sc_t, 1e4, "none")
    torch.cuda.synchronize()
    assert np.array_equal(kc.cpu().numpy(), kc_h)
    assert np.array_equal(vc.cpu().numpy(), vc_h)
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("ctx,part", [([1, 17, 600, 1500, 33], 256), ([3000, 9, 700], 512),
                                      ([16, 31, 32, 33, 511, 512, 513], 64)])
@pytest.mark.parametrize("hq", [8, 16, 32, 64])
@pytest.mark.parametrize("d", [64, 128])
def test_fp8_decode_matches_oracle(ctx, part, hq, d):
    import torch
    pk = ensure_built()
    wl = synth.make_custom(ctx, hq, 8, d, kv_dtype="bf16", seed=len(ctx) + hq + d, value_std=0.5,
                           tokens_per_seq=0)
    vals = synth.make_values_fp8(wl, device="cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    n = pk.photon_paged_attention_workspace_size(wl.num_seqs, hq, d, wl.max_context_len, part)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    out = torch.full((wl.num_seqs, hq, d), float("nan"), device="cuda")
    pk.photon_paged_attention_decode_fp8(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0],
                                         vals["k_scale"][0], vals["v_scale"][0], bt, cl, wl.scale,
                                         out, wl.max_context_len, part, ws)
    ref = oracle.paged_attention_fp8(synth.to_storage_numpy(vals["q"][0]),
                                     vals["k_cache"][0].cpu().numpy(), vals["v_cache"][0].cpu().numpy(),
                                     vals["k_scale"][0].cpu().numpy(), vals["v_scale"][0].cpu().numpy(),
                                     wl.block_tables, wl.context_lens, wl.scale)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.isfinite(got).all() and np.abs(got - ref).max() <= 5e-3
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_gather_is_bit_exact(d):
    """One dominant key per (sequence, KV head): the output must be exactly
    fp32(decode(code) * v_scale) of that token, checking the dim-major V
    fragment loads and the in-page token order."""
    import torch
    pk = ensure_built()
    ctx = [1, 17, 600, 1500, 16, 33]
    hq, hkv = 32, 8
    wl = synth.make_custom(ctx, hq, hkv, d, kv_dtype="bf16", seed=9, tokens_per_seq=0)
    vals = synth.make_values_fp8(wl, device="cuda")
    kc, vc = vals["k_cache"][0], vals["v_cache"][0]
    kc.zero_()
    q = torch.zeros_like(vals["q"][0])
    q[..., 0] = 1.0
    rng = np.random.default_rng(4)
    hot = [[int(rng.integers(0, c)) for _ in range(hkv)] for c in ctx]
    ks = vals["k_scale"][0].cpu().numpy()
    for s, js in enumerate(hot):
        for h, j in enumerate(js):
            kc[wl.block_tables[s, j // 16], h, j % 16, 0] = 0x7E  # 448: score 448*ks*... >> others
    # make the dominant score large in absolute terms: scale so that 448*ks*scale >> 150 / log2(e)
    scale = 1000.0 / float(448 * ks.min())
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    out = torch.empty((len(ctx), hq, d), device="cuda")
    n = pk.photon_paged_attention_workspace_size(len(ctx), hq, d, max(ctx), 256)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    pk.photon_paged_attention_decode_fp8(q, kc, vc, vals["k_scale"][0], vals["v_scale"][0], bt, cl,
                                         scale, out, max(ctx), 256, ws)
    vc_h = vc.cpu().numpy()
    vs = vals["v_scale"][0].cpu().numpy()
    G = hq // hkv
    for s, js in enumerate(hot):
        for g in range(hq):
            j = js[g // G]
            codes = vc_h[wl.block_tables[s, j // 16], g // G, :, j % 16]
            ref = (np.array([oracle.fp8_decode(c) for c in codes]) * np.float64(vs[g // G])).astype(np.float32)
            assert np.array_equal(out[s, g].cpu().numpy(), ref), (s, g)
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("name", ["cb_batch16", "qwen3_ragged64"])
def test_fp8_write_then_decode_step(name):
    """Write through the FP8 path, then decode: equals the oracle's FP8 write +
    attention over the same pools (head_dim 64 and 128)."""
    import torch
    pk = ensure_built()
    wl = synth.make(name, seed=4)
    d = wl.head_dim
    vals = synth.make_values_fp8(wl, device="cuda")
    ks, vs = vals["k_scale"][0], vals["v_scale"][0]
    kc_h = vals["k_cache"][0].cpu().numpy().copy()
    vc_h = vals["v_cache"][0].cpu().numpy().copy()
    sm = pk.photon_slot_mapping(wl.block_tables, wl.token_seq, wl.positions)
    pk.photon_kv_cache_write_fp8(vals["k"][0], vals["v"][0], torch.from_numpy(wl.positions).cuda(),
                                 torch.from_numpy(sm).cuda(), vals["k_cache"][0], vals["v_cache"][0],
                                 ks, vs, wl.rope_theta)
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    n = pk.photon_paged_attention_workspace_size(wl.num_seqs, wl.num_q_heads, d, wl.max_context_len,
                                                 wl.partition_size)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    out = torch.empty((wl.num_seqs, wl.num_q_heads, d), device="cuda")
    pk.photon_paged_attention_decode_fp8(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0], ks, vs,
                                         bt, cl, wl.scale, out, wl.max_context_len, wl.partition_size, ws)
    oracle.kv_cache_write_fp8(synth.to_storage_numpy(vals["k"][0]), synth.to_storage_numpy(vals["v"][0]),
                              wl.positions, sm, kc_h, vc_h, ks.cpu().numpy(), vs.cpu().numpy(),
                              wl.rope_theta)
    ref = oracle.paged_attention_fp8(synth.to_storage_numpy(vals["q"][0]), kc_h, vc_h,
                                     ks.cpu().numpy(), vs.cpu().numpy(), wl.block_tables,
                                     wl.context_lens, wl.scale)
    torch.cuda.synchronize()
    assert np.abs(out.cpu().numpy() - ref).max() <= 5e-3
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_decode_bf16_output(d):
    """bf16 output rows from the FP8 decode (single-partition rows written by
    the decode kernel, split rows by the merge): the oracle value within the
    tolerance or half a bf16 step of it."""
    import torch
    from tests.helpers import bf16_spacing
    pk = ensure_built()
    ctx = [3, 200, 1300, 16, 700]
    wl = synth.make_custom(ctx, 16, 8, d, kv_dtype="bf16", seed=17 + d, value_std=0.5, tokens_per_seq=0)
    vals = synth.make_values_fp8(wl, device="cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    part = 256
    n = pk.photon_paged_attention_workspace_size(wl.num_seqs, 16, d, wl.max_context_len, part)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    out = torch.empty((wl.num_seqs, 16, d), dtype=torch.bfloat16, device="cuda")
    pk.photon_paged_attention_decode_fp8(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0],
                                         vals["k_scale"][0], vals["v_scale"][0], bt, cl, wl.scale,
                                         out, wl.max_context_len, part, ws)
    ref = oracle.paged_attention_fp8(synth.to_storage_numpy(vals["q"][0]),
                                     vals["k_cache"][0].cpu().numpy(), vals["v_cache"][0].cpu().numpy(),
                                     vals["k_scale"][0].cpu().numpy(), vals["v_scale"][0].cpu().numpy(),
                                     wl.block_tables, wl.context_lens, wl.scale)
    got = out.float().cpu().numpy()
    assert (np.abs(got - ref) <= np.maximum(5e-3, bf16_spacing(ref) / 2 + 1e-6)).all()
    assert pk.photon_device_errors() == 0


def test_fp8_longctx_b256_every_row():
    """The full-size 256-sequence FP8 step as the benchmark runs it (FP8
    write of the new tokens, then decode with 512-token partitions), every
    output row against the oracle.  The oracle's FP8 attention dequantises
    the pools it is given to fp64, so it runs over groups of 32 sequences,
    each on a compact copy of that group's blocks (taken before the write,
    relabelled), through its own FP8 write and attention."""
    import torch
    pk = ensure_built()
    wl = synth.make("longctx_b256")
    vals = synth.make_values_fp8(wl, device="cuda")
    ks, vs = vals["k_scale"][0], vals["v_scale"][0]
    ks_h, vs_h = ks.cpu().numpy(), vs.cpu().numpy()
    k_h, v_h = synth.to_storage_numpy(vals["k"][0]), synth.to_storage_numpy(vals["v"][0])
    q_h = synth.to_storage_numpy(vals["q"][0])
    ref = np.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim))
    for g0 in range(0, wl.num_seqs, 32):
        pick = list(range(g0, min(g0 + 32, wl.num_seqs)))
        bt = wl.block_tables[pick]
        used = np.unique(bt[bt >= 0])
        remap = -np.ones(wl.num_blocks, np.int64)
        remap[used] = np.arange(len(used))
        bt_c = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
        idx = torch.from_numpy(used).cuda()
        kc_c = vals["k_cache"][0].index_select(0, idx).cpu().numpy()
        vc_c = vals["v_cache"][0].index_select(0, idx).cpu().numpy()
        tok = np.nonzero(np.isin(wl.token_seq, pick))[0]
        ts_c = (wl.token_seq[tok] - g0).astype(np.int32)
        sm_c = oracle.slot_mapping(bt_c, ts_c, wl.positions[tok], 16)
        oracle.kv_cache_write_fp8(k_h[tok], v_h[tok], wl.positions[tok], sm_c, kc_c, vc_c, ks_h, vs_h,
                                  wl.rope_theta)
        ref[pick] = oracle.paged_attention_fp8(q_h[pick], kc_c, vc_c, ks_h, vs_h, bt_c,
                                               wl.context_lens[pick], wl.scale)
    sm = pk.photon_slot_mapping(wl.block_tables, wl.token_seq, wl.positions)
    pk.photon_kv_cache_write_fp8(vals["k"][0], vals["v"][0], torch.from_numpy(wl.positions).cuda(),
                                 torch.from_numpy(sm).cuda(), vals["k_cache"][0], vals["v_cache"][0],
                                 ks, vs, wl.rope_theta)
    n = pk.photon_paged_attention_workspace_size(wl.num_seqs, wl.num_q_heads, wl.head_dim,
                                                 wl.max_context_len, wl.partition_size)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    out = torch.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim), device="cuda")
    pk.photon_paged_attention_decode_fp8(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0], ks, vs,
                                         torch.from_numpy(wl.block_tables).cuda(),
                                         torch.from_numpy(wl.context_lens).cuda(), wl.scale, out,
                                         wl.max_context_len, wl.partition_size, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert (err <= 5e-3).all(), f"max err {err.max():.3g}"
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("d,out_dtype", [(64, "f32"), (128, "bf16")])
def test_fp8_partial_then_reduce_equals_decode(d, out_dtype):
    """photon_paged_attention_partial_fp8 followed by
    photon_paged_attention_reduce runs the same kernels as
    photon_paged_attention_decode_fp8: bit-identical rows (split and
    single-partition sequences, an empty context), and the oracle's values."""
    import torch
    pk = ensure_built()
    ctx = [0, 5, 300, 1100, 16, 2049]
    wl = synth.make_custom(ctx, 32, 8, d, kv_dtype="bf16", seed=61 + d, value_std=0.5, tokens_per_seq=0)
    vals = synth.make_values_fp8(wl, device="cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    part = 256
    n = pk.photon_paged_attention_workspace_size(wl.num_seqs, 32, d, wl.max_context_len, part)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    args = (vals["q"][0], vals["k_cache"][0], vals["v_cache"][0], vals["k_scale"][0],
            vals["v_scale"][0], bt, cl, wl.scale)
    one = torch.full((wl.num_seqs, 32, d), float("nan"), dtype=dt, device="cuda")
    two = torch.full((wl.num_seqs, 32, d), float("nan"), dtype=dt, device="cuda")
    pk.photon_paged_attention_decode_fp8(*args, one, wl.max_context_len, part, ws)
    pk.photon_paged_attention_partial_fp8(*args, two, wl.max_context_len, part, ws)
    pk.photon_paged_attention_reduce(cl, two, wl.max_context_len, part, ws)
    torch.cuda.synchronize()
    assert torch.equal(one, two)
    ref = oracle.paged_attention_fp8(synth.to_storage_numpy(vals["q"][0]),
                                     vals["k_cache"][0].cpu().numpy(), vals["v_cache"][0].cpu().numpy(),
                                     vals["k_scale"][0].cpu().numpy(), vals["v_scale"][0].cpu().numpy(),
                                     wl.block_tables, wl.context_lens, wl.scale)
    got = two.float().cpu().numpy()
    tol = 5e-3 if out_dtype == "f32" else np.maximum(5e-3, bf16_spacing(ref) / 2 + 1e-6)
    assert (np.abs(got - ref) <= tol).all()
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_fp8_page_balanced_pieces(d, G):
    """The FP8 decode's page-balanced pieces (a long context cut over many
    warps, empty and one-page contexts, pieces starting on odd pages inside
    the two-page pipeline steps, runs crossing several short sequences;
    16-token partitions let a run be as short as one page) against the
    oracle, at every head size and group size."""
    import torch
    pk = ensure_built()
    hq = 8 * G
    rng = np.random.default_rng(5 * d + G)
    ctx = [0, 20000, 1, 33, 0, 16, 4097, 250] + rng.integers(1, 700, size=9).tolist()
    wl = synth.make_custom(ctx, hq, 8, d, kv_dtype="bf16", seed=77 + d + G, value_std=0.5, tokens_per_seq=0)
    vals = synth.make_values_fp8(wl, device="cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    for part in (16, 128):
        n = pk.photon_paged_attention_workspace_size(wl.num_seqs, hq, d, wl.max_context_len, part)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
        out = torch.full((wl.num_seqs, hq, d), float("nan"), device="cuda")
        pk.photon_paged_attention_decode_fp8(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0],
                                             vals["k_scale"][0], vals["v_scale"][0], bt, cl, wl.scale,
                                             out, wl.max_context_len, part, ws)
        ref = oracle.paged_attention_fp8(synth.to_storage_numpy(vals["q"][0]),
                                         vals["k_cache"][0].cpu().numpy(), vals["v_cache"][0].cpu().numpy(),
                                         vals["k_scale"][0].cpu().numpy(), vals["v_scale"][0].cpu().numpy(),
                                         wl.block_tables, wl.context_lens, wl.scale)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.isfinite(got).all() and np.abs(got - ref).max() <= 5e-3
    assert pk.photon_device_errors() == 0


def test_fp8_context_beyond_bound_is_clamped_and_flagged():
    """A device context length above max_context_len: the balanced walker
    (which counts the page stream from the context lengths) clamps it as the
    fixed partitions do, sets the context-range bit, and the rows equal the
    oracle's over the clamped context."""
    import torch
    pk = ensure_built()
    ctx = [64, 700, 3, 300]
    wl = synth.make_custom(ctx, 16, 8, 64, kv_dtype="bf16", seed=44, value_std=0.5, tokens_per_seq=0)
    vals = synth.make_values_fp8(wl, device="cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    cap, part = 512, 128  # the 700-token context is clamped to 512
    n = pk.photon_paged_attention_workspace_size(wl.num_seqs, 16, 64, cap, part)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    out = torch.full((wl.num_seqs, 16, 64), float("nan"), device="cuda")
    pk.photon_device_errors(clear=True)
    pk.photon_paged_attention_decode_fp8(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0],
                                         vals["k_scale"][0], vals["v_scale"][0], bt, cl, wl.scale,
                                         out, cap, part, ws)
    assert pk.photon_device_errors(clear=True) & pk.DEVERR_CONTEXT_RANGE
    ref = oracle.paged_attention_fp8(synth.to_storage_numpy(vals["q"][0]),
                                     vals["k_cache"][0].cpu().numpy(), vals["v_cache"][0].cpu().numpy(),
                                     vals["k_scale"][0].cpu().numpy(), vals["v_scale"][0].cpu().numpy(),
                                     wl.block_tables, np.minimum(wl.context_lens, cap).astype(np.int32),
                                     wl.scale)
    got = out.cpu().numpy()
    assert np.isfinite(got).all() and np.abs(got - ref).max() <= 5e-3
