"""Seeded synthetic workloads for the paged-KV decode step.

This module is shared by the product tests, the benchmark and the oracle
tests.  It holds none of the method's arithmetic: it draws context lengths,
assigns physical blocks to sequences (the "scheduler state" before a step),
lists which (sequence, position) pairs the step writes, and fills tensors with
seeded normal values.  Slot numbers, RoPE and attention are computed
elsewhere (by the product's metadata builder and kernels, and independently by
the oracle).

Workloads (head shapes from Llama-3.2-1B and Qwen3, the two model families
the PhotonInfer README names under "Performance highlights"):

  tiny_fp32        2 sequences, context {5, 19}, 4 q / 2 kv heads, d 32,
                   fp32, pool of 8 blocks, RoPE theta 1e4.
  llama1b_single   1 sequence, context 1024, 32 q / 8 kv heads, d 64, bf16,
                   16 layers (one cache pair each) sharing a block table of 64
                   pages drawn from 1024, theta 5e5.
  cb_batch16       16 sequences, Llama heads; 12 running with context
                   U[100, 2048]; 4 newly admitted write a 100-token prompt and
                   then decode (context 101); pool 4096 shuffled blocks.
  qwen3_ragged64   64 sequences, 16 q / 8 kv heads, d 128, bf16, context
                   lognormal(median 1500, sigma 0.8) clipped to [16, 8192];
                   blocks from an allocator with interleaved frees (phantom
                   sequences give their blocks back), so pages are fragmented;
                   theta 1e6.
  longctx_b256     256 sequences, Llama heads, context U[512, 32768] with 3
                   (1 %) forced to context 1; split-K partition 512 tokens;
                   pool = 1.05 x the blocks needed, shuffled.

Split-K partition sizes: 512 tokens for longctx_b256 (fixed by that
workload); 32 and 64 tokens for llama1b_single and cb_batch16, the smallest
multiple of the block size that still gives every warp of the persistent grid
work; 128 for qwen3_ragged64 (about 4.6 items per resident warp: with a cold
L2 its step was shortest there, 256 giving fewer, longer items and a longer
tail); 512 for tiny_fp32.

All draws come from numpy's default_rng(seed) (metadata) and a seeded
torch.Generator (values).  Values are N(0, 1) * value_std, rounded to the
storage dtype.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

WORKLOADS = ("tiny_fp32", "llama1b_single", "cb_batch16", "qwen3_ragged64", "longctx_b256")


@dataclasses.dataclass
class Workload:
    name: str
    kv_dtype: str                 # "f32" or "bf16": storage type of q, k, v and the caches
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    num_layers: int
    context_lens: np.ndarray      # int32 [B], counting the tokens written in this step
    block_tables: np.ndarray      # int32 [B, max_blocks_per_seq], -1 padded
    token_seq: np.ndarray         # int32 [T], sequence of each token written this step
    positions: np.ndarray         # int32 [T], position of each written token in its sequence
    rope_theta: float
    scale: float
    partition_size: int
    value_std: float
    seed: int

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.positions.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def elem_bytes(self) -> int:
        return 4 if self.kv_dtype == "f32" else 2


def _tables_from_lists(lists, width=None) -> np.ndarray:
    width = width if width is not None else max((len(x) for x in lists), default=0)
    bt = np.full((len(lists), max(width, 1)), -1, dtype=np.int32)
    for i, row in enumerate(lists):
        bt[i, :len(row)] = row
    return bt


def _decode_tokens(context_lens):
    """One new token per sequence, at its last position (context - 1)."""
    cl = np.asarray(context_lens, dtype=np.int64)
    live = np.nonzero(cl > 0)[0]
    return live.astype(np.int32), (cl[live] - 1).astype(np.int32)


def _sequential_alloc(rng, context_lens, block_size, num_blocks):
    free = list(rng.permutation(num_blocks))
    lists = []
    for c in context_lens:
        n = -(-int(c) // block_size)
        lists.append([int(x) for x in free[:n]])
        del free[:n]
    return lists


def _fragmenting_alloc(rng, context_lens, block_size, num_blocks, num_phantom):
    """Round-robin, one block per live sequence per round, with phantom
    sequences that are freed at random rounds and whose blocks go back to the
    free list at random places."""
    need = [-(-int(c) // block_size) for c in context_lens]
    total_real = sum(need)
    phantom_need = list(rng.integers(4, 64, size=num_phantom))
    phantom_free_round = list(rng.integers(1, 64, size=num_phantom))
    free = list(rng.permutation(num_blocks))
    real = [[] for _ in need]
    ph = [[] for _ in phantom_need]
    rnd = 0
    while sum(len(r) for r in real) < total_real:
        for i in range(len(need)):
            if len(real[i]) < need[i]:
                real[i].append(int(free.pop(0)))
        for j in range(num_phantom):
            if ph[j] is not None and rnd < phantom_free_round[j] and len(ph[j]) < phantom_need[j] and free:
                ph[j].append(int(free.pop(0)))
            if ph[j] is not None and rnd == phantom_free_round[j]:
                for b in ph[j]:
                    free.insert(int(rng.integers(0, len(free) + 1)), b)
                ph[j] = None
        rnd += 1
        if not free and sum(len(r) for r in real) < total_real:
            raise RuntimeError("pool too small for the fragmenting allocator")
    return real


def make(name: str, seed: int = 0) -> Workload:
    """Builds the named workload's metadata (values come from make_values)."""
    rng = np.random.default_rng(seed)
    if name == "tiny_fp32":
        ctx = np.array([5, 19], dtype=np.int32)
        perm = rng.permutation(8)
        lists = [[int(perm[0])], [int(perm[1]), int(perm[2])]]
        ts, pos = _decode_tokens(ctx)
        return Workload(name, "f32", 4, 2, 32, 16, 8, 1, ctx, _tables_from_lists(lists), ts, pos,
                        1e4, 1.0 / math.sqrt(32), 512, 1.0, seed)
    if name == "llama1b_single":
        ctx = np.array([1024], dtype=np.int32)
        pages = rng.choice(1024, size=64, replace=False)
        ts, pos = _decode_tokens(ctx)
        return Workload(name, "bf16", 32, 8, 64, 16, 1024, 16, ctx,
                        _tables_from_lists([[int(x) for x in pages]]), ts, pos,
                        5e5, 1.0 / 8.0, 32, 0.5, seed)
    if name == "cb_batch16":
        B, n_new, prompt = 16, 4, 100
        ctx = rng.integers(100, 2049, size=B).astype(np.int32)
        admitted = np.sort(rng.choice(B, size=n_new, replace=False))
        ctx[admitted] = prompt + 1
        lists = _sequential_alloc(rng, ctx, 16, 4096)
        ts, pos = [], []
        for s in range(B):
            if s in admitted:   # prompt tokens 0..99, then the decode token at 100
                ts += [s] * (prompt + 1)
                pos += list(range(prompt + 1))
            else:
                ts.append(s)
                pos.append(int(ctx[s]) - 1)
        return Workload(name, "bf16", 32, 8, 64, 16, 4096, 1, ctx, _tables_from_lists(lists),
                        np.array(ts, np.int32), np.array(pos, np.int32), 5e5, 1.0 / 8.0, 64,
                        0.5, seed)
    if name == "qwen3_ragged64":
        B = 64
        ctx = np.clip(np.rint(rng.lognormal(math.log(1500.0), 0.8, size=B)), 16, 8192).astype(np.int32)
        need = int(sum(-(-int(c) // 16) for c in ctx))
        nb = int(math.ceil(need * 1.25))
        lists = _fragmenting_alloc(rng, ctx, 16, nb, num_phantom=32)
        ts, pos = _decode_tokens(ctx)
        return Workload(name, "bf16", 16, 8, 128, 16, nb, 1, ctx, _tables_from_lists(lists), ts, pos,
                        1e6, 1.0 / math.sqrt(128), 128, 0.5, seed)
    if name == "longctx_b256":
        B = 256
        ctx = rng.integers(512, 32769, size=B).astype(np.int32)
        ones = rng.choice(B, size=3, replace=False)
        ctx[ones] = 1
        need = int(sum(-(-int(c) // 16) for c in ctx))
        nb = int(math.ceil(need * 1.05))
        lists = _sequential_alloc(rng, ctx, 16, nb)
        ts, pos = _decode_tokens(ctx)
        return Workload(name, "bf16", 32, 8, 64, 16, nb, 1, ctx, _tables_from_lists(lists), ts, pos,
                        5e5, 1.0 / 8.0, 512, 0.5, seed)
    raise KeyError(f"unknown workload {name!r}; choose from {WORKLOADS}")


def truncate(wl: Workload, n: int) -> Workload:
    """The first n sequences of a workload, with a pool cut down to the
    blocks they use (relabelled in order of first use)."""
    n = min(int(n), wl.num_seqs)
    bt = wl.block_tables[:n]
    used = np.unique(bt[bt >= 0])
    remap = -np.ones(max(wl.num_blocks, 1), np.int64)
    remap[used] = np.arange(len(used))
    bt2 = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    keep = wl.token_seq < n
    return dataclasses.replace(wl, name=f"{wl.name}[:{n}]", num_blocks=max(len(used), 1),
                               context_lens=wl.context_lens[:n].copy(), block_tables=bt2,
                               token_seq=wl.token_seq[keep].copy(),
                               positions=wl.positions[keep].copy())


def make_custom(context_lens, num_q_heads, num_kv_heads, head_dim, kv_dtype="bf16",
                block_size=16, pool_factor=1.5, partition_size=512, rope_theta=1e4,
                value_std=1.0, seed=0, tokens_per_seq=1, num_layers=1) -> Workload:
    """A shuffled-pool workload with the given context lengths.  Each sequence
    writes its last `tokens_per_seq` positions in this step."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int32)
    need = int(sum(-(-int(c) // block_size) for c in ctx))
    nb = max(1, int(math.ceil(max(need, 1) * pool_factor)))
    lists = _sequential_alloc(rng, ctx, block_size, nb)
    ts, pos = [], []
    for s, c in enumerate(ctx):
        for p in range(max(0, int(c) - tokens_per_seq), int(c)):
            ts.append(s)
            pos.append(p)
    width = max(1, max((len(x) for x in lists), default=1))
    return Workload("custom", kv_dtype, num_q_heads, num_kv_heads, head_dim, block_size, nb,
                    num_layers, ctx, _tables_from_lists(lists, width), np.array(ts, np.int32),
                    np.array(pos, np.int32), rope_theta, 1.0 / math.sqrt(head_dim),
                    partition_size, value_std, seed)


# ---- values -------------------------------------------------------------------

def _torch_dtype(wl):
    import torch
    return torch.float32 if wl.kv_dtype == "f32" else torch.bfloat16


def fill_normal_(t, gen, std, chunk=1 << 26):
    """Fills a tensor with N(0,1)*std drawn from `gen`, a chunk at a time (so a
    multi-GB bf16 pool never needs an fp32 copy of itself)."""
    import torch
    flat = t.view(-1)
    for i in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - i)
        flat[i:i + n] = (torch.randn(n, generator=gen, device=t.device, dtype=torch.float32)
                         * std).to(t.dtype)
    return t


def make_values(wl: Workload, device="cpu", seed=None, layers=None):
    """Seeded tensors for a workload, on `device`:
      q [L, B, H_q, d], k, v [L, T, H_kv, d], k_cache, v_cache
      [L, num_blocks, H_kv, bs, d] (the whole pool, history included)."""
    import torch
    L = wl.num_layers if layers is None else layers
    gen = torch.Generator(device=device)
    gen.manual_seed(int(wl.seed if seed is None else seed) + 0x5EED)
    dt = _torch_dtype(wl)
    B, T = wl.num_seqs, wl.num_tokens
    shp_c = (L, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    out = {
        "q": fill_normal_(torch.empty((L, B, wl.num_q_heads, wl.head_dim), dtype=dt, device=device), gen, wl.value_std),
        "k": fill_normal_(torch.empty((L, T, wl.num_kv_heads, wl.head_dim), dtype=dt, device=device), gen, wl.value_std),
        "v": fill_normal_(torch.empty((L, T, wl.num_kv_heads, wl.head_dim), dtype=dt, device=device), gen, wl.value_std),
        "k_cache": fill_normal_(torch.empty(shp_c, dtype=dt, device=device), gen, wl.value_std),
        "v_cache": fill_normal_(torch.empty(shp_c, dtype=dt, device=device), gen, wl.value_std),
    }
    return out


def make_values_fp8(wl: Workload, device="cpu", seed=None, layers=None):
    """FP8 (E4M3) pools for a workload: per-KV-head scales 4*value_std/448
    (times a seeded factor in [0.5, 1.5]) and cache codes of N(0,1)*value_std
    values (torch's float8 conversion; test data only).  Layouts: K
    [L, nb, H_kv, bs, d], V [L, nb, H_kv, d, bs] (dims outer).  q, k, v as in
    make_values (bf16)."""
    import torch
    L = wl.num_layers if layers is None else layers
    base = make_values(dataclasses.replace(wl, kv_dtype="bf16", num_blocks=1), device, seed, L)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(wl.seed if seed is None else seed) + 0xF8)
    H, bs, d = wl.num_kv_heads, wl.block_size, wl.head_dim
    ks = (4 * wl.value_std / 448) * (0.5 + torch.rand((L, H), generator=gen, device=device))
    vs = (4 * wl.value_std / 448) * (0.5 + torch.rand((L, H), generator=gen, device=device))
    kc = torch.empty((L, wl.num_blocks, H, bs, d), dtype=torch.uint8, device=device)
    vc = torch.empty((L, wl.num_blocks, H, d, bs), dtype=torch.uint8, device=device)
    for l in range(L):
        for cache, sc in ((kc[l], ks[l]), (vc[l], vs[l])):
            flat = cache.view(wl.num_blocks, H, -1)
            for b0 in range(0, wl.num_blocks, 4096):
                b1 = min(b0 + 4096, wl.num_blocks)
                x = torch.randn((b1 - b0, H, flat.shape[2]), generator=gen, device=device) * wl.value_std
                flat[b0:b1] = ((x / sc.view(1, H, 1)).clamp(-448, 448)
                               .to(torch.float8_e4m3fn).view(torch.uint8))
    base.update({"k_cache": kc, "v_cache": vc, "k_scale": ks.float().contiguous(),
                 "v_scale": vs.float().contiguous()})
    return base


def to_storage_numpy(t) -> np.ndarray:
    """Host numpy view of a float32 tensor, or the uint16 bit patterns of a
    bf16 tensor (the oracle's storage format)."""
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)


def kv_bytes_read(wl: Workload, kv_elem_bytes=None) -> int:
    """Algorithmic bytes the attention reads per layer: every context token's K
    and V row for every KV head (kv_elem_bytes per value: the storage type's
    size, or 1 for FP8 pools), the query, the output (fp32), the block-table
    entries in use and the context lengths."""
    ctx = wl.context_lens.astype(np.int64)
    kvb = wl.elem_bytes if kv_elem_bytes is None else kv_elem_bytes
    kv = int(ctx.sum()) * wl.num_kv_heads * wl.head_dim * 2 * kvb
    qo = wl.num_seqs * wl.num_q_heads * wl.head_dim * (wl.elem_bytes + 4)
    tables = int(sum(-(-int(c) // wl.block_size) for c in ctx)) * 4 + wl.num_seqs * 4
    return kv + qo + tables


def write_bytes(wl: Workload) -> int:
    """Algorithmic bytes of the cache write per layer: read k, v; write both
    cache rows; read positions and slot numbers."""
    T = wl.num_tokens
    return T * wl.num_kv_heads * wl.head_dim * 2 * 2 * wl.elem_bytes + T * (4 + 8)
