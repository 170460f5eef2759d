"""Device parity of photon_kv_cache_write (the batched, RoPE-fused cache
write) against the oracle: placement bit-exact with index-tagged values,
untouched slots keep their canary bits, RoPE'd K within one unit in the last
place of the storage type, V bit-exact, slot -1 and out-of-pool slots write
nothing."""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import bf16_spacing, ensure_built, host_inputs, oracle_step

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


def _tag_tensor(shape, dtype, start):
    # distinct small integers: exact in bf16 (|x| < 256) and fp32
    torch = _torch()
    n = int(np.prod(shape))
    vals = (torch.arange(n, dtype=torch.float64) % 251 + start) * torch.where(
        torch.arange(n) % 2 == 0, 1.0, -1.0).double()
    return vals.reshape(shape).to(dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_write_placement_is_bit_exact_and_leaves_canaries(dtype):
    torch = _torch()
    pk = ensure_built()
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    T, H, d, nb = 37, 4, 64, 20
    rng = np.random.default_rng(1)
    slots = rng.choice(nb * 16, size=T, replace=False).astype(np.int64)
    slots[[3, 10]] = -1
    pos = rng.integers(0, 5000, size=T).astype(np.int32)
    k = _tag_tensor((T, H, d), dt, 1).cuda()
    v = _tag_tensor((T, H, d), dt, 2).cuda()
    canary = -123.0
    kc = torch.full((nb, H, 16, d), canary, dtype=dt, device="cuda")
    vc = torch.full((nb, H, 16, d), canary, dtype=dt, device="cuda")
    pk.photon_kv_cache_write(k, v, torch.from_numpy(pos).cuda(), torch.from_numpy(slots).cuda(),
                             kc, vc, 1e4, "none")
    torch.cuda.synchronize()
    kc_h, vc_h = kc.cpu(), vc.cpu()
    written = torch.zeros((nb, H, 16), dtype=torch.bool)
    for t in range(T):
        if slots[t] < 0:
            continue
        b, o = int(slots[t]) // 16, int(slots[t]) % 16
        written[b, :, o] = True
        assert torch.equal(kc_h[b, :, o].view(torch.int16 if dtype == "bf16" else torch.int32),
                           k[t].cpu().view(torch.int16 if dtype == "bf16" else torch.int32))
        assert torch.equal(vc_h[b, :, o], v[t].cpu())
    assert (kc_h[~written] == canary).all() and (vc_h[~written] == canary).all()
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("style", ["neox", "gptj"])
@pytest.mark.parametrize("name", ["tiny_fp32", "cb_batch16", "qwen3_ragged64"])
def test_write_rope_within_one_ulp_of_oracle(name, style):
    torch = _torch()
    pk = ensure_built()
    wl = synth.make(name, seed=3)
    vals = synth.make_values(wl, device="cuda")
    h = host_inputs(wl, vals)
    code = {"neox": oracle.ROPE_NEOX, "gptj": oracle.ROPE_GPTJ}[style]
    _, kc_ref, vc_ref, sm = oracle_step(wl, h, rope_style=code)
    sm_t = torch.from_numpy(sm).cuda()
    pos_t = torch.from_numpy(wl.positions).cuda()
    pk.photon_kv_cache_write(vals["k"][0], vals["v"][0], pos_t, sm_t, vals["k_cache"][0],
                             vals["v_cache"][0], wl.rope_theta, style)
    torch.cuda.synchronize()
    kc = synth.to_storage_numpy(vals["k_cache"][0])
    vc = synth.to_storage_numpy(vals["v_cache"][0])
    assert np.array_equal(vc, vc_ref)                       # V bit-exact everywhere
    b, o = sm // 16, sm % 16
    got = oracle.to_f64(kc[b, :, o])
    ref = oracle.to_f64(kc_ref[b, :, o])
    if wl.kv_dtype == "bf16":
        tol = bf16_spacing(ref)
    else:
        tol = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert (np.abs(got - ref) <= tol).all()
    mism = (kc != kc_ref)
    mism[b, :, o] = False
    assert not mism.any()                                   # nothing else changed
    assert pk.photon_device_errors() == 0


def test_write_out_of_pool_slot_is_skipped_and_flagged():
    torch = _torch()
    pk = ensure_built()
    k = torch.ones((2, 1, 32), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((2, 1, 16, 32), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    pk.photon_device_errors(clear=True)
    pk.photon_kv_cache_write(k, k, torch.zeros(2, dtype=torch.int32, device="cuda"),
                             torch.tensor([5, 32], dtype=torch.int64, device="cuda"), kc, vc, 1e4)
    assert pk.photon_device_errors(clear=True) == pk.DEVERR_SLOT_RANGE
    assert float(kc.float().sum()) == 32.0                  # only slot 5 was written
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("style", ["neox", "gptj", "none"])
@pytest.mark.parametrize("name", ["tiny_fp32", "cb_batch16", "qwen3_ragged64"])
def test_fused_q_rope_write_matches_oracle_and_the_plain_write(name, style):
    """photon_rope_q_kv_cache_write: q rows rotated in place within one unit in
    the last place of the oracle's rotation (left bit-identical with no
    rotation), and K/V caches bit-identical to photon_kv_cache_write on the
    same inputs, for every RoPE style."""
    torch = _torch()
    pk = ensure_built()
    wl = synth.make(name, seed=5)
    vals = synth.make_values(wl, device="cuda")
    q = vals["q"][0].clone()
    q_pos = torch.from_numpy((wl.context_lens - 1).clip(min=0).astype(np.int32)).cuda()
    code = {"neox": oracle.ROPE_NEOX, "gptj": oracle.ROPE_GPTJ, "none": oracle.ROPE_NONE}[style]
    q_ref = oracle.rope_rows(synth.to_storage_numpy(q), (wl.context_lens - 1).clip(min=0),
                             wl.rope_theta, code)
    sm = torch.from_numpy(oracle.slot_mapping(wl.block_tables, wl.token_seq, wl.positions, 16)).cuda()
    pos = torch.from_numpy(wl.positions).cuda()
    kc2, vc2 = vals["k_cache"][0].clone(), vals["v_cache"][0].clone()
    pk.photon_rope_q_kv_cache_write(q, q_pos, vals["k"][0], vals["v"][0], pos, sm,
                                    vals["k_cache"][0], vals["v_cache"][0], wl.rope_theta, style)
    pk.photon_kv_cache_write(vals["k"][0], vals["v"][0], pos, sm, kc2, vc2, wl.rope_theta, style)
    torch.cuda.synchronize()
    assert torch.equal(vals["k_cache"][0], kc2) and torch.equal(vals["v_cache"][0], vc2)
    got = oracle.to_f64(synth.to_storage_numpy(q))
    ref = oracle.to_f64(q_ref)
    if style == "none":
        tol = 0.0
    elif wl.kv_dtype == "bf16":
        tol = bf16_spacing(ref)
    else:
        tol = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert (np.abs(got - ref) <= tol).all()
    assert pk.photon_device_errors() == 0


def test_fused_q_rope_step_decode_parity():
    """Unrotated q -> fused write -> decode equals the oracle's rotate q, write,
    attend."""
    torch = _torch()
    pk = ensure_built()
    wl = synth.make("cb_batch16", seed=8)
    vals = synth.make_values(wl, device="cuda")
    h = host_inputs(wl, vals)
    q_pos_np = (wl.context_lens - 1).astype(np.int32)
    h["q"] = oracle.rope_rows(h["q"], q_pos_np, wl.rope_theta)
    ref, _, _, _ = oracle_step(wl, h)
    sm = torch.from_numpy(pk.photon_slot_mapping(wl.block_tables, wl.token_seq, wl.positions)).cuda()
    pk.photon_rope_q_kv_cache_write(vals["q"][0], torch.from_numpy(q_pos_np).cuda(), vals["k"][0],
                                    vals["v"][0], torch.from_numpy(wl.positions).cuda(), sm,
                                    vals["k_cache"][0], vals["v_cache"][0], wl.rope_theta)
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    n = pk.photon_paged_attention_workspace_size(wl.num_seqs, wl.num_q_heads, wl.head_dim,
                                                 wl.max_context_len, wl.partition_size)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    out = torch.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim), device="cuda")
    pk.photon_paged_attention_decode(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0], bt, cl,
                                     wl.scale, out, wl.max_context_len, wl.partition_size, ws)
    torch.cuda.synchronize()
    assert np.abs(out.cpu().numpy() - ref).max() <= 5e-3
    assert pk.photon_device_errors() == 0


def _cancelling_rows(wl, positions, rows, rng, style, dtype):
    """[len(positions), rows, d] values whose RoPE nearly cancels: each pair
    (x0, x1) = (r(tan(angle)), 1) * 2^e with r() the rounding to the storage
    type, so x0 cos - x1 sin = (r(tan) - tan) cos is ~2^-9 (bf16) of the
    inputs and, for pairs whose tangent lies near a representable number,
    far less."""
    torch = _torch()
    d = wl.head_dim
    half = d // 2
    inv = wl.rope_theta ** (-2.0 * np.arange(half) / d)
    tan = np.tan(np.asarray(positions, np.float64)[:, None] * inv[None, :])
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    b = torch.from_numpy(tan).to(tdt).double().numpy()
    scale = 2.0 ** rng.integers(-3, 4, size=(len(positions), rows, 1))
    x = np.zeros((len(positions), rows, d))
    i = np.arange(half)
    e0, e1 = (i, i + half) if style == "neox" else (2 * i, 2 * i + 1)
    x[:, :, e0] = b[:, None, :] * scale
    x[:, :, e1] = scale
    return torch.from_numpy(x).to(tdt)   # exact: a storage value times a power of two


@pytest.mark.parametrize("style", ["neox", "gptj"])
@pytest.mark.parametrize("dtype,d,hkv", [("bf16", 32, 4), ("bf16", 64, 8), ("bf16", 128, 8),
                                         ("bf16", 256, 8), ("bf16", 256, 16)])
def test_rope_near_cancellation_within_one_ulp(dtype, d, hkv, style):
    """bf16 K and q rows built so that the first element of every rotated pair
    nearly cancels -- where a rotation computed in fp32 alone could round
    wrongly and the kernels' fp64 decision takes over -- at every head size
    (d 256: two pairs per thread; 16 KV heads: several rounds of loads per
    CTA).  Rotated K (cache) and q (fused write, in place) within one unit in
    the last place of the oracle's exact rotation; V bit-exact.  (Here bf16
    inputs cancel down to ~2^-28 of their size: an fp32-only rotation would be
    off by many units, while two fp64 cosines -- the oracle's and the
    device's -- would only disagree in the result below ~2^-45.  fp32 inputs
    can cancel that far, so fp32 caches are checked on random values below.)"""
    torch = _torch()
    pk = ensure_built()
    rng = np.random.default_rng(d + hkv)
    wl = synth.make_custom([40, 300, 1000, 17, 4100], 2 * hkv if hkv < 16 else 16, hkv, d,
                           kv_dtype=dtype, seed=d, tokens_per_seq=3, rope_theta=5e5)
    vals = synth.make_values(wl, device="cuda")
    vals["k"][0].copy_(_cancelling_rows(wl, wl.positions, hkv, rng, style, dtype).cuda())
    q_pos = (wl.context_lens - 1).clip(min=0).astype(np.int32)
    q = _cancelling_rows(wl, q_pos, wl.num_q_heads, rng, style, dtype).cuda()
    h = host_inputs(wl, vals)
    code = {"neox": oracle.ROPE_NEOX, "gptj": oracle.ROPE_GPTJ}[style]
    _, kc_ref, vc_ref, sm = oracle_step(wl, h, rope_style=code)
    q_ref = oracle.rope_rows(synth.to_storage_numpy(q), q_pos, wl.rope_theta, code)
    pk.photon_rope_q_kv_cache_write(q, torch.from_numpy(q_pos).cuda(), vals["k"][0], vals["v"][0],
                                    torch.from_numpy(wl.positions).cuda(), torch.from_numpy(sm).cuda(),
                                    vals["k_cache"][0], vals["v_cache"][0], wl.rope_theta, style)
    torch.cuda.synchronize()
    kc = synth.to_storage_numpy(vals["k_cache"][0])
    assert np.array_equal(synth.to_storage_numpy(vals["v_cache"][0]), vc_ref)
    b, o = sm // 16, sm % 16
    for got, ref in ((oracle.to_f64(kc[b, :, o]), oracle.to_f64(kc_ref[b, :, o])),
                     (oracle.to_f64(synth.to_storage_numpy(q)), oracle.to_f64(q_ref))):
        if dtype == "bf16":
            tol = bf16_spacing(ref)
        else:
            tol = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
        assert (np.abs(got - ref) <= tol).all()
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("style", ["neox", "gptj"])
@pytest.mark.parametrize("dtype,d,hkv", [("f32", 256, 16), ("bf16", 256, 16), ("f32", 128, 8)])
def test_rope_write_large_heads_random_values(dtype, d, hkv, style):
    """Random K / V / q at head sizes whose rows take several rounds of loads
    per CTA (16 KV heads of 256 dims: four rounds of rotations, two of V
    chunks) and the fp32 cache's all-fp64 rotation: K and q within one unit in
    the last place of the oracle, V bit-exact."""
    torch = _torch()
    pk = ensure_built()
    wl = synth.make_custom([33, 700, 2049, 5], 16, hkv, d, kv_dtype=dtype, seed=7 + d,
                           tokens_per_seq=4, rope_theta=5e5)
    vals = synth.make_values(wl, device="cuda")
    q = vals["q"][0].clone()
    q_pos = (wl.context_lens - 1).clip(min=0).astype(np.int32)
    h = host_inputs(wl, vals)
    code = {"neox": oracle.ROPE_NEOX, "gptj": oracle.ROPE_GPTJ}[style]
    _, kc_ref, vc_ref, sm = oracle_step(wl, h, rope_style=code)
    q_ref = oracle.rope_rows(synth.to_storage_numpy(q), q_pos, wl.rope_theta, code)
    pk.photon_rope_q_kv_cache_write(q, torch.from_numpy(q_pos).cuda(), vals["k"][0], vals["v"][0],
                                    torch.from_numpy(wl.positions).cuda(), torch.from_numpy(sm).cuda(),
                                    vals["k_cache"][0], vals["v_cache"][0], wl.rope_theta, style)
    torch.cuda.synchronize()
    kc = synth.to_storage_numpy(vals["k_cache"][0])
    assert np.array_equal(synth.to_storage_numpy(vals["v_cache"][0]), vc_ref)
    b, o = sm // 16, sm % 16
    for got, ref in ((oracle.to_f64(kc[b, :, o]), oracle.to_f64(kc_ref[b, :, o])),
                     (oracle.to_f64(synth.to_storage_numpy(q)), oracle.to_f64(q_ref))):
        if dtype == "bf16":
            tol = bf16_spacing(ref)
        else:
            tol = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
        assert (np.abs(got - ref) <= tol).all()
    assert pk.photon_device_errors() == 0
