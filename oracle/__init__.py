"""fp64 CPU oracle for one paged-KV decode step (write + attention).

TEST INFRASTRUCTURE ONLY.  The product library never imports, loads or calls
anything in this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` do.  The oracle
shares no code with the CUDA path: its arithmetic lives in ``photon_oracle.c``
(plain C, fp64, compiled with gcc) and this module only marshals numpy arrays.

Source of the method: the PhotonInfer README (zh-CN / fr / ja pages),
"Technical details > Paged attention" (block-level KV cache, per-sequence
cache offsets, one batched K/V write for many sequences) and "Key features >
GPU-optimised kernels" (batched RoPE, numerically stable attention softmax).

Every function here has a pin in ``tests/test_oracle_*.py`` that checks it
against something other than itself (closed forms, invariants, a library
routine on a special case, brute force on tiny inputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

F32 = 0
BF16 = 1
F64 = 3
ROPE_NEOX = 0
ROPE_GPTJ = 1
ROPE_NONE = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "photon_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compiles photon_oracle.c into liboracle.so beside it (gcc, OpenMP).

    ``-ffp-contract=off`` keeps gcc from fusing multiply-adds, so x86 and Arm
    hosts produce the same bits."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.orc_round_bf16.argtypes = [dbl]
    lib.orc_round_bf16.restype = ctypes.c_uint16
    lib.orc_slot_mapping.argtypes = [P, i32, P, P, i32, i32, P]
    lib.orc_slot_mapping.restype = None
    lib.orc_rope.argtypes = [P, i32, i32, dbl, ctypes.c_int]
    lib.orc_rope.restype = None
    lib.orc_kv_cache_write.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i64,
                                       ctypes.c_int, dbl, ctypes.c_int]
    lib.orc_kv_cache_write.restype = ctypes.c_int
    lib.orc_rope_rows.argtypes = [P, P, i32, i32, i32, ctypes.c_int, dbl, ctypes.c_int]
    lib.orc_rope_rows.restype = None
    lib.orc_paged_attention.argtypes = [P, P, P, P, P, dbl, P, i32, i32, i32, i32, i32,
                                        i32, ctypes.c_int, P, i32]
    lib.orc_paged_attention.restype = None
    lib.orc_paged_attention_split.argtypes = [P, P, P, P, P, dbl, P, i32, i32, i32, i32,
                                              i32, i32, ctypes.c_int, i32]
    lib.orc_paged_attention_split.restype = None
    lib.orc_fp8_decode.argtypes = [ctypes.c_uint8]
    lib.orc_fp8_decode.restype = dbl
    lib.orc_fp8_encode.argtypes = [dbl]
    lib.orc_fp8_encode.restype = ctypes.c_uint8
    lib.orc_kv_cache_write_fp8.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i64,
                                           ctypes.c_int, dbl, ctypes.c_int]
    lib.orc_kv_cache_write_fp8.restype = ctypes.c_int
    lib.orc_fp8_dequant.argtypes = [P, P, P, P, i64, i32, i32, i32, P, P]
    lib.orc_fp8_dequant.restype = None
    lib.orc_num_threads.argtypes = []
    lib.orc_num_threads.restype = ctypes.c_int
    lib.orc_set_num_threads.argtypes = [ctypes.c_int]
    lib.orc_set_num_threads.restype = None
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float64:
        return F64
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:  # bf16 bit patterns
        return BF16
    raise TypeError(f"oracle storage arrays are float32 or uint16 (bf16 bits), got {a.dtype}")


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> None:
    """Host threads for the OpenMP loops (launchers such as torchrun may have
    limited them through OMP_NUM_THREADS)."""
    _load().orc_set_num_threads(int(n))


# ---- bf16 storage helpers --------------------------------------------------

def round_bf16(x: float) -> int:
    """Nearest bf16 bit pattern to the double x, ties to even, one rounding."""
    return int(_load().orc_round_bf16(float(x)))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of a storage array (float32 or bf16 bits) to float64."""
    return bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


# ---- FP8 E4M3 -------------------------------------------------------------------

def fp8_decode(code: int) -> float:
    """Exact value of an E4M3 code (NaN for 0x7F / 0xFF)."""
    return float(_load().orc_fp8_decode(int(code) & 0xFF))


def fp8_encode(x: float) -> int:
    """Nearest E4M3 code to x, ties to even, saturating at +-448."""
    return int(_load().orc_fp8_encode(float(x)))


def kv_cache_write_fp8(k, v, positions, slot_mapping_, k_cache, v_cache, k_scale, v_scale,
                       rope_theta, rope_style=ROPE_NEOX):
    """In-place quantising write into FP8 pools (K [nb][H][bs][d] codes, V
    [nb][H][d][bs] codes) with per-KV-head scales (float32 [H])."""
    T, H, d = k.shape
    nb, H2, bs, d2 = k_cache.shape
    assert k_cache.dtype == v_cache.dtype == np.uint8 and v_cache.shape == (nb, H, d, bs)
    ks = np.ascontiguousarray(k_scale, np.float32)
    vs = np.ascontiguousarray(v_scale, np.float32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    sm = np.ascontiguousarray(slot_mapping_, dtype=np.int64)
    rc = _load().orc_kv_cache_write_fp8(_ptr(np.ascontiguousarray(k)), _ptr(np.ascontiguousarray(v)),
                                        _ptr(pos), _ptr(sm), _ptr(k_cache), _ptr(v_cache), _ptr(ks),
                                        _ptr(vs), T, H, d, bs, nb, _dtype_code(k),
                                        float(rope_theta), int(rope_style))
    if rc != 0:
        raise ValueError("slot_mapping points outside the cache pool")


def fp8_dequant(k_cache, v_cache, k_scale, v_scale):
    """fp64 K and V pools in the plain [nb][H][bs][d] layout from FP8 pools."""
    nb, H, bs, d = k_cache.shape
    ko = np.empty((nb, H, bs, d), np.float64)
    vo = np.empty((nb, H, bs, d), np.float64)
    _load().orc_fp8_dequant(_ptr(np.ascontiguousarray(k_cache)), _ptr(np.ascontiguousarray(v_cache)),
                            _ptr(np.ascontiguousarray(k_scale, np.float32)),
                            _ptr(np.ascontiguousarray(v_scale, np.float32)), nb, H, d, bs,
                            _ptr(ko), _ptr(vo))
    return ko, vo


def paged_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale):
    """Decode attention over FP8 pools: the same definition as
    paged_attention, on the exactly dequantised values."""
    kd, vd = fp8_dequant(k_cache, v_cache, k_scale, v_scale)
    return paged_attention(np.ascontiguousarray(to_f64(q)), kd, vd, block_tables, context_lens, scale)


# ---- metadata ----------------------------------------------------------------

def slot_mapping(block_tables: np.ndarray, token_seq: np.ndarray, positions: np.ndarray,
                 block_size: int) -> np.ndarray:
    """slot = block_tables[s][p // bs] * bs + p % bs per new token, -1 if unmapped."""
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ts = np.ascontiguousarray(token_seq, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    out = np.empty(len(pos), dtype=np.int64)
    _load().orc_slot_mapping(_ptr(bt), bt.shape[1], _ptr(ts), _ptr(pos), len(pos),
                             block_size, _ptr(out))
    return out


# ---- RoPE ---------------------------------------------------------------------

def rope(x: np.ndarray, position: int, theta: float, style: int = ROPE_NEOX) -> np.ndarray:
    """Rotary embedding of one head vector (float64 in, float64 out)."""
    v = np.ascontiguousarray(x, dtype=np.float64).copy()
    _load().orc_rope(_ptr(v), v.shape[0], int(position), float(theta), int(style))
    return v


def rope_rows(x: np.ndarray, positions: np.ndarray, theta: float, style: int = ROPE_NEOX) -> np.ndarray:
    """Copy of the storage array x [rows, heads, d] with every head vector of
    row r rotated at positions[r] and rounded once into the storage type."""
    y = np.ascontiguousarray(x).copy()
    code = _dtype_code(y)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    n, h, d = y.shape
    assert pos.shape == (n,)
    _load().orc_rope_rows(_ptr(y), _ptr(pos), n, h, d, code, float(theta), int(style))
    return y


# ---- the two kernels' definitions -------------------------------------------

def kv_cache_write(k: np.ndarray, v: np.ndarray, positions: np.ndarray,
                   slot_mapping_: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                   rope_theta: float, rope_style: int = ROPE_NEOX) -> None:
    """In-place write of RoPE(k) and v into the host caches through slot_mapping.

    k, v: [T, H_kv, d]; k_cache, v_cache: [num_blocks, H_kv, bs, d]; all the
    same storage dtype (float32, or uint16 holding bf16 bits)."""
    code = _dtype_code(k_cache)
    assert k.dtype == v.dtype == k_cache.dtype == v_cache.dtype
    T, H, d = k.shape
    nb, H2, bs, d2 = k_cache.shape
    assert (H, d) == (H2, d2) and v.shape == k.shape and v_cache.shape == k_cache.shape
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    sm = np.ascontiguousarray(slot_mapping_, dtype=np.int64)
    rc = _load().orc_kv_cache_write(_ptr(np.ascontiguousarray(k)), _ptr(np.ascontiguousarray(v)),
                                    _ptr(pos), _ptr(sm), _ptr(k_cache), _ptr(v_cache),
                                    T, H, d, bs, nb, code, float(rope_theta), int(rope_style))
    if rc != 0:
        raise ValueError("slot_mapping points outside the cache pool")


def paged_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                    block_tables: np.ndarray, context_lens: np.ndarray, scale: float,
                    return_weights: bool = False):
    """Decode attention, fp64 result [B, H_q, d] (and weights [B, H_q, max_ctx])."""
    code = _dtype_code(k_cache)
    assert q.dtype == k_cache.dtype == v_cache.dtype
    B, Hq, d = q.shape
    nb, Hkv, bs, d2 = k_cache.shape
    assert d2 == d and Hq % Hkv == 0
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    assert bt.shape[0] == B and cl.shape == (B,)
    out = np.empty((B, Hq, d), dtype=np.float64)
    max_ctx = int(cl.max()) if (return_weights and B > 0) else 0
    w = np.empty((B, Hq, max(max_ctx, 1)), dtype=np.float64) if return_weights else None
    _load().orc_paged_attention(_ptr(np.ascontiguousarray(q)), _ptr(k_cache), _ptr(v_cache),
                                _ptr(bt), _ptr(cl), float(scale), _ptr(out), B, Hq, Hkv, d, bs,
                                bt.shape[1], code, _ptr(w) if w is not None else None,
                                max_ctx)
    return (out, w[:, :, :max_ctx]) if return_weights else out


def paged_attention_prefill(q, token_seq, positions, k_cache, v_cache, block_tables, scale):
    """Causal prefill attention: query token t (sequence token_seq[t], position
    positions[t]) attends to its sequence's tokens 0 .. positions[t] -- the
    decode definition with that token's own context length."""
    rows = np.ascontiguousarray(np.asarray(block_tables)[np.asarray(token_seq, np.int64)], np.int32)
    ctx = np.asarray(positions, np.int32) + 1
    return paged_attention(q, k_cache, v_cache, rows, ctx, scale)


def paged_attention_split(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                          block_tables: np.ndarray, context_lens: np.ndarray, scale: float,
                          partition_size: int) -> np.ndarray:
    """Split-K + log-sum-exp form of paged_attention, fp64 result [B, H_q, d]."""
    code = _dtype_code(k_cache)
    B, Hq, d = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.empty((B, Hq, d), dtype=np.float64)
    _load().orc_paged_attention_split(_ptr(np.ascontiguousarray(q)), _ptr(k_cache),
                                      _ptr(v_cache), _ptr(bt), _ptr(cl), float(scale),
                                      _ptr(out), B, Hq, Hkv, d, bs, bt.shape[1], code,
                                      int(partition_size))
    return out


def decode_step(q, k, v, positions, slot_mapping_, k_cache, v_cache, block_tables,
                context_lens, scale, rope_theta, rope_style=ROPE_NEOX):
    """The whole step on host copies: write first, then attend over the context
    that now holds the new tokens.  Mutates k_cache / v_cache."""
    kv_cache_write(k, v, positions, slot_mapping_, k_cache, v_cache, rope_theta, rope_style)
    return paged_attention(q, k_cache, v_cache, block_tables, context_lens, scale)
