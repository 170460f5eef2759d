"""Shared test plumbing: run one decode step through the library (device) and
through the oracle (host), on the same seeded inputs."""
from __future__ import annotations

import numpy as np

import oracle
import synth


def ensure_built():
    import paged_kv_decode_write_gb300 as pk
    import os
    if not os.path.exists(pk.lib_path):
        from paged_kv_decode_write_gb300 import _build
        _build.build()
    return pk


def host_inputs(wl, vals, layer=0):
    """Host storage copies (float32 or bf16 bit patterns) of one layer's inputs,
    taken before the device step mutates the caches."""
    return {name: synth.to_storage_numpy(vals[name][layer]).copy()
            for name in ("q", "k", "v", "k_cache", "v_cache")}


def oracle_step(wl, h, rope_style=oracle.ROPE_NEOX, block_tables=None, context_lens=None):
    bt = wl.block_tables if block_tables is None else block_tables
    cl = wl.context_lens if context_lens is None else context_lens
    sm = oracle.slot_mapping(bt, wl.token_seq, wl.positions, wl.block_size)
    kc, vc = h["k_cache"].copy(), h["v_cache"].copy()
    oracle.kv_cache_write(h["k"], h["v"], wl.positions, sm, kc, vc, wl.rope_theta, rope_style)
    out = oracle.paged_attention(h["q"], kc, vc, bt, cl, wl.scale)
    return out, kc, vc, sm


def gpu_step(wl, vals, layer=0, partition_size=None, out_dtype=None, rope_style="neox",
             split_calls=False, max_context_len=None):
    """Write + decode on the device through the C ABI.  Mutates the layer's
    caches in `vals`.  max_context_len: the bound declared to the decode call
    (default: the batch's longest context).  Returns (out, slot_mapping used)."""
    import torch
    pk = ensure_built()
    dev = vals["q"].device
    sm_host = pk.photon_slot_mapping(wl.block_tables, wl.token_seq, wl.positions, wl.block_size)
    sm = torch.from_numpy(sm_host).to(dev)
    pos = torch.from_numpy(wl.positions.astype(np.int32)).to(dev)
    kc, vc = vals["k_cache"][layer], vals["v_cache"][layer]
    if wl.num_tokens:
        pk.photon_kv_cache_write(vals["k"][layer], vals["v"][layer], pos, sm, kc, vc,
                                 wl.rope_theta, rope_style)
    bt = torch.from_numpy(wl.block_tables).to(dev)
    cl = torch.from_numpy(wl.context_lens.astype(np.int32)).to(dev)
    part = wl.partition_size if partition_size is None else partition_size
    mcl = wl.max_context_len if max_context_len is None else int(max_context_len)
    ws_bytes = pk.photon_paged_attention_workspace_size(wl.num_seqs, wl.num_q_heads, wl.head_dim,
                                                        mcl, part)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) if ws_bytes else None
    od = torch.float32 if out_dtype is None else out_dtype
    out = torch.full((wl.num_seqs, wl.num_q_heads, wl.head_dim), float("nan"), dtype=od, device=dev)
    args = (vals["q"][layer], kc, vc, bt, cl, wl.scale, out, mcl, part, ws)
    if split_calls:
        pk.photon_paged_attention_partial(*args)
        pk.photon_paged_attention_reduce(cl, out, mcl, part, ws)
    else:
        pk.photon_paged_attention_decode(*args)
    torch.cuda.synchronize()
    return out, sm_host


def bf16_spacing(x: np.ndarray) -> np.ndarray:
    """Distance from |x| to the next bf16 number (x exactly bf16 or fp64)."""
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 2.0 ** -126)))
    return 2.0 ** (np.maximum(e, -126) - 7)
