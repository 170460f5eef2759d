"""Guard regions around every buffer the decode and prefill calls write
(output rows, split-K workspace) must come back untouched, and the caches they
only read must come back bit-identical -- the stand-in for a memory checker
on this pool, for each kernel path: tensor-core bf16 (d 64, 128), CUDA-core
fp32, FP8, tiled prefill."""
import numpy as np
import pytest

import synth
from tests.helpers import ensure_built

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes of canary on each side (keeps 256-byte alignment)


def _guarded(n_bytes, dtype):
    """A device buffer of n_bytes between two canary regions; returns
    (whole uint8 buffer, typed view of the middle)."""
    import torch
    whole = torch.full((GUARD + n_bytes + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    mid = whole[GUARD:GUARD + n_bytes].view(dtype)
    return whole, mid


def _intact(whole):
    h = whole.cpu().numpy()
    return (h[:GUARD] == 0xA5).all() and (h[-GUARD:] == 0xA5).all()


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 64)])
def test_decode_writes_only_out_and_workspace(dtype, d):
    import torch
    pk = ensure_built()
    wl = synth.make_custom([1, 37, 600, 1500, 16], 16, 4, d, kv_dtype=dtype, seed=d, tokens_per_seq=0)
    vals = synth.make_values(wl, device="cuda")
    kc0, vc0 = vals["k_cache"][0].clone(), vals["v_cache"][0].clone()
    part = 128
    n_out = wl.num_seqs * wl.num_q_heads * d
    out_w, out = _guarded(4 * n_out, torch.float32)
    out = out.view(wl.num_seqs, wl.num_q_heads, d)
    ws_bytes = pk.photon_paged_attention_workspace_size(wl.num_seqs, wl.num_q_heads, d, wl.max_context_len, part)
    ws_w, ws = _guarded(ws_bytes, torch.uint8)
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    pk.photon_paged_attention_decode(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0], bt, cl, wl.scale,
                                     out, wl.max_context_len, part, ws)
    torch.cuda.synchronize()
    assert _intact(out_w) and _intact(ws_w)
    assert torch.equal(kc0, vals["k_cache"][0]) and torch.equal(vc0, vals["v_cache"][0])
    assert torch.isfinite(out).all()
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_decode_writes_only_out_and_workspace(d):
    import torch
    pk = ensure_built()
    wl = synth.make_custom([5, 333, 1200], 32, 8, d, kv_dtype="bf16", seed=3 + d, tokens_per_seq=0)
    vals = synth.make_values_fp8(wl, device="cuda")
    kc0, vc0 = vals["k_cache"][0].clone(), vals["v_cache"][0].clone()
    part = 256
    n_out = wl.num_seqs * wl.num_q_heads * d
    out_w, out = _guarded(4 * n_out, torch.float32)
    out = out.view(wl.num_seqs, wl.num_q_heads, d)
    ws_bytes = pk.photon_paged_attention_workspace_size(wl.num_seqs, wl.num_q_heads, d, wl.max_context_len, part)
    ws_w, ws = _guarded(ws_bytes, torch.uint8)
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    pk.photon_paged_attention_decode_fp8(vals["q"][0], vals["k_cache"][0], vals["v_cache"][0],
                                         vals["k_scale"][0], vals["v_scale"][0], bt, cl, wl.scale, out,
                                         wl.max_context_len, part, ws)
    torch.cuda.synchronize()
    assert _intact(out_w) and _intact(ws_w)
    assert torch.equal(kc0, vals["k_cache"][0]) and torch.equal(vc0, vals["v_cache"][0])
    assert torch.isfinite(out).all()
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_tiled_prefill_writes_only_out_and_workspace(d):
    import torch
    pk = ensure_built()
    ctx = [700, 40, 5]
    wl = synth.make_custom(ctx, 16, 4, d, kv_dtype="bf16", seed=9 + d, tokens_per_seq=0)
    ts = np.concatenate([np.zeros(100), np.ones(40), np.full(1, 2)]).astype(np.int32)
    pos = np.concatenate([np.arange(600, 700), np.arange(40), [4]]).astype(np.int32)
    vals = synth.make_values(wl, device="cuda")
    kc0, vc0 = vals["k_cache"][0].clone(), vals["v_cache"][0].clone()
    T, part = len(ts), 64
    q = (torch.randn((T, 16, d), device="cuda") * 0.5).bfloat16()
    out_w, out = _guarded(4 * T * 16 * d, torch.float32)
    out = out.view(T, 16, d)
    maxp = int(pos.max())
    ws_bytes = pk.photon_paged_attention_workspace_size(T, 16, d, maxp + 1, part)
    ws_w, ws = _guarded(ws_bytes, torch.uint8)
    pk.photon_paged_attention_prefill(q, torch.from_numpy(ts).cuda(), torch.from_numpy(pos).cuda(),
                                      vals["k_cache"][0], vals["v_cache"][0],
                                      torch.from_numpy(wl.block_tables).cuda(), wl.scale, out, maxp, part, ws)
    torch.cuda.synchronize()
    assert _intact(out_w) and _intact(ws_w)
    assert torch.equal(kc0, vals["k_cache"][0]) and torch.equal(vc0, vals["v_cache"][0])
    assert torch.isfinite(out).all()
    assert pk.photon_device_errors() == 0


@pytest.mark.parametrize("d,G", [(64, 4), (128, 2), (128, 8)])
def test_tc_prefill_writes_only_out(d, G):
    """The tcgen05 prefill (a batch long enough for its route): output rows
    in guard regions, bf16 output included, caches untouched."""
    import torch
    pk = ensure_built()
    hkv, R = 8, 128 // G
    ctx = [20 * R + 50, 3 * R, 7]
    wl = synth.make_custom(ctx, G * hkv, hkv, d, kv_dtype="bf16", seed=19 + d, tokens_per_seq=0)
    ts = np.concatenate([np.zeros(20 * R), np.ones(3 * R), np.full(7, 2)]).astype(np.int32)
    pos = np.concatenate([np.arange(50, 50 + 20 * R), np.arange(3 * R), np.arange(7)]).astype(np.int32)
    T = len(ts)
    assert -(-T // R) * hkv >= torch.cuda.get_device_properties(0).multi_processor_count
    vals = synth.make_values(wl, device="cuda")
    kc0, vc0 = vals["k_cache"][0].clone(), vals["v_cache"][0].clone()
    q = (torch.randn((T, G * hkv, d), device="cuda") * 0.5).bfloat16()
    maxp = int(pos.max())
    for odt, es in ((torch.float32, 4), (torch.bfloat16, 2)):
        out_w, out = _guarded(es * T * G * hkv * d, odt)
        out = out.view(T, G * hkv, d)
        ws_bytes = pk.photon_paged_attention_workspace_size(T, G * hkv, d, maxp + 1, 512)
        ws_w, ws = _guarded(ws_bytes, torch.uint8)
        pk.photon_paged_attention_prefill(q, torch.from_numpy(ts).cuda(), torch.from_numpy(pos).cuda(),
                                          vals["k_cache"][0], vals["v_cache"][0],
                                          torch.from_numpy(wl.block_tables).cuda(), wl.scale, out, maxp,
                                          512, ws)
        torch.cuda.synchronize()
        assert _intact(out_w) and _intact(ws_w)
        assert torch.isfinite(out.float()).all()
    assert torch.equal(kc0, vals["k_cache"][0]) and torch.equal(vc0, vals["v_cache"][0])
    assert pk.photon_device_errors() == 0
