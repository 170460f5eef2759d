"""Thin Python binding of the GB300 paged-KV decode library (libphoton_gb300.so).

Argument marshalling only: every step of the write and the attention runs in
the library's CUDA kernels.  PyTorch supplies device memory and streams.  The
functions carry the C ABI's names (include/photon.h) and take torch tensors
(device) or numpy arrays (host metadata); sizes are read off the shapes.

If the shared library has not been built, every call raises: there is no
fallback implementation.  Build it with ``python -c "import __graft_entry__ as
g; g.build()"`` (or ``python paged_kv_decode_write_gb300/_build.py``).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "PhotonError", "F32", "BF16", "ROPE_NEOX", "ROPE_GPTJ", "ROPE_NONE",
    "DEVERR_SLOT_RANGE", "DEVERR_BLOCK_RANGE", "DEVERR_CONTEXT_RANGE", "DEVERR_WAIT_TIMEOUT",
    "lib", "lib_path", "photon_version", "photon_status_string",
    "photon_kv_cache_write", "photon_rope_q_kv_cache_write", "photon_kv_cache_write_fp8",
    "photon_paged_attention_decode_fp8", "photon_paged_attention_partial_fp8",
    "photon_paged_attention_prefill",
    "photon_paged_attention_workspace_size",
    "photon_paged_attention_decode", "photon_paged_attention_partial",
    "photon_paged_attention_reduce", "photon_paged_attention_decode_static",
    "STATIC_SCRATCH_BYTES", "photon_device_errors", "photon_selftest_wait_timeout", "photon_slot_mapping",
    "photon_build_step_metadata", "BlockPool", "Scheduler",
    "REQ_WAITING", "REQ_RUNNING", "REQ_FINISHED", "REQ_PREEMPTED",
]

F32, BF16 = 0, 1
ROPE_NEOX, ROPE_GPTJ, ROPE_NONE = 0, 1, 2
DEVERR_SLOT_RANGE, DEVERR_BLOCK_RANGE, DEVERR_CONTEXT_RANGE, DEVERR_WAIT_TIMEOUT = 1, 2, 4, 8
_ROPE = {"neox": ROPE_NEOX, "gptj": ROPE_GPTJ, "none": ROPE_NONE}
STATIC_SCRATCH_BYTES = 32 * 1024 * 1024  # PHOTON_STATIC_SCRATCH_BYTES

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libphoton_gb300.so")
_lib = None


class PhotonError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {photon_status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(lib_path):
        raise RuntimeError(f"{lib_path} is missing: build the CUDA library first "
                           "(paged_kv_decode_write_gb300/_build.py); there is no fallback")
    L = ctypes.CDLL(lib_path)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    E = ctypes.c_int
    L.photon_status_string.argtypes = [E]
    L.photon_status_string.restype = ctypes.c_char_p
    L.photon_version.argtypes = []
    L.photon_version.restype = E
    L.photon_kv_cache_write.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i64, E, f32, E, P]
    L.photon_kv_cache_write.restype = E
    L.photon_rope_q_kv_cache_write.argtypes = [P, P, i32, i32, P, P, P, P, P, P, i32, i32, i32,
                                               i32, i64, E, f32, E, P]
    L.photon_rope_q_kv_cache_write.restype = E
    L.photon_paged_attention_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.photon_paged_attention_workspace_size.restype = sz
    dec = [P, P, P, P, P, f32, P, i32, i32, i32, i32, i32, i64, i32, i32, i32, E, E, P, sz, P]
    for name in ("photon_paged_attention_decode", "photon_paged_attention_partial"):
        getattr(L, name).argtypes = dec
        getattr(L, name).restype = E
    L.photon_paged_attention_decode_static.argtypes = dec[:-3] + [P]
    L.photon_paged_attention_decode_static.restype = E
    L.photon_kv_cache_write_fp8.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i64, E,
                                            f32, E, P]
    L.photon_kv_cache_write_fp8.restype = E
    for name in ("photon_paged_attention_decode_fp8", "photon_paged_attention_partial_fp8"):
        getattr(L, name).argtypes = [P, P, P, P, P, P, P, f32, P, i32, i32, i32, i32, i32, i64, i32,
                                     i32, i32, E, P, sz, P]
        getattr(L, name).restype = E
    L.photon_paged_attention_prefill.argtypes = [P, P, P, P, P, P, f32, P, i32, i32, i32, i32, i32,
                                                 i32, i64, i32, i32, i32, E, E, P, sz, P]
    L.photon_paged_attention_prefill.restype = E
    L.photon_paged_attention_reduce.argtypes = [P, P, i32, i32, i32, i32, i32, E, P, sz, P]
    L.photon_paged_attention_reduce.restype = E
    L.photon_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32), E]
    L.photon_device_errors.restype = E
    L.photon_selftest_wait_timeout.argtypes = [ctypes.c_uint32, P]
    L.photon_selftest_wait_timeout.restype = E
    L.photon_block_pool_create.argtypes = [i64, ctypes.c_uint64, ctypes.POINTER(P)]
    L.photon_block_pool_create.restype = E
    L.photon_block_pool_destroy.argtypes = [P]
    L.photon_block_pool_destroy.restype = None
    L.photon_block_pool_num_free.argtypes = [P]
    L.photon_block_pool_num_free.restype = i64
    L.photon_block_pool_alloc.argtypes = [P, i32, P]
    L.photon_block_pool_alloc.restype = E
    L.photon_block_pool_free.argtypes = [P, P, i32]
    L.photon_block_pool_free.restype = E
    L.photon_slot_mapping.argtypes = [P, i32, i32, P, P, i32, i32, P]
    L.photon_slot_mapping.restype = E
    L.photon_build_step_metadata.argtypes = [i32, P, P, i32, P, i32, P, i32, P, P, P, P,
                                             ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.photon_build_step_metadata.restype = E
    _lib = L
    return L


def photon_status_string(status: int) -> str:
    return lib().photon_status_string(int(status)).decode()


def photon_version() -> int:
    return int(lib().photon_version())


def _check(status: int, what: str):
    if status != 0:
        raise PhotonError(status, what)


# ---- device-tensor marshalling ---------------------------------------------

def _dt(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"storage dtype must be float32 or bfloat16, got {t.dtype}")


def _p(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def photon_kv_cache_write(k, v, positions, slot_mapping, k_cache, v_cache, rope_theta,
                          rope_style="neox", stream=None):
    """k, v [T, H_kv, d]; positions int32 [T]; slot_mapping int64 [T];
    k_cache, v_cache [num_blocks, H_kv, block_size, d] -- all on the device."""
    T, H, d = k.shape
    nb, H2, bs, d2 = k_cache.shape
    if (H2, d2) != (H, d) or tuple(v.shape) != tuple(k.shape) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch between k/v and the caches")
    style = _ROPE[rope_style] if isinstance(rope_style, str) else int(rope_style)
    _check(lib().photon_kv_cache_write(_p(k), _p(v), _p(positions), _p(slot_mapping), _p(k_cache),
                                       _p(v_cache), T, H, d, bs, nb, _dt(k_cache), float(rope_theta),
                                       style, _stream(stream)), "photon_kv_cache_write")


def photon_rope_q_kv_cache_write(q, q_positions, k, v, positions, slot_mapping, k_cache, v_cache,
                                 rope_theta, rope_style="neox", stream=None):
    """photon_kv_cache_write plus the in-place rotation of q [Tq, H_q, d] at
    q_positions (int32 [Tq]) in the same launch."""
    Tq, Hq, dq = q.shape
    T, H, d = k.shape
    nb, H2, bs, d2 = k_cache.shape
    if dq != d or (H2, d2) != (H, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch between q, k/v and the caches")
    style = _ROPE[rope_style] if isinstance(rope_style, str) else int(rope_style)
    _check(lib().photon_rope_q_kv_cache_write(_p(q), _p(q_positions), Tq, Hq, _p(k), _p(v),
                                              _p(positions), _p(slot_mapping), _p(k_cache),
                                              _p(v_cache), T, H, d, bs, nb, _dt(k_cache),
                                              float(rope_theta), style, _stream(stream)),
           "photon_rope_q_kv_cache_write")


def photon_kv_cache_write_fp8(k, v, positions, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                              rope_theta, rope_style="neox", stream=None):
    """FP8 (E4M3) write: k, v [T, H_kv, d] (float32 or bfloat16); k_cache uint8
    [num_blocks, H_kv, bs, d]; v_cache uint8 [num_blocks, H_kv, d, bs];
    k_scale, v_scale float32 [H_kv]."""
    T, H, d = k.shape
    nb, H2, bs, d2 = k_cache.shape
    if (H2, d2) != (H, d) or tuple(v_cache.shape) != (nb, H, d, bs) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch between k/v and the FP8 pools")
    style = _ROPE[rope_style] if isinstance(rope_style, str) else int(rope_style)
    _check(lib().photon_kv_cache_write_fp8(_p(k), _p(v), _p(positions), _p(slot_mapping),
                                           _p(k_cache), _p(v_cache), _p(k_scale), _p(v_scale), T,
                                           H, d, bs, nb, _dt(k), float(rope_theta), style,
                                           _stream(stream)), "photon_kv_cache_write_fp8")


def _decode_fp8_args(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale,
                     out, max_context_len, partition_size, workspace, stream):
    B, Hq, d = q.shape
    nb, Hkv, bs, d2 = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return (_p(q), _p(k_cache), _p(v_cache), _p(k_scale), _p(v_scale), _p(block_tables),
            _p(context_lens), float(scale), _p(out), B, Hq, Hkv, d, bs, nb, block_tables.shape[1],
            int(max_context_len), int(partition_size), _dt(out), _p(workspace), ws_bytes,
            _stream(stream))


def photon_paged_attention_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                      context_lens, scale, out, max_context_len,
                                      partition_size=512, workspace=None, stream=None):
    """Decode attention over FP8 pools (see photon_kv_cache_write_fp8); q bf16."""
    _check(lib().photon_paged_attention_decode_fp8(*_decode_fp8_args(
        q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale, out,
        max_context_len, partition_size, workspace, stream)), "photon_paged_attention_decode_fp8")


def photon_paged_attention_partial_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                       context_lens, scale, out, max_context_len,
                                       partition_size=512, workspace=None, stream=None):
    """The partial half of photon_paged_attention_decode_fp8; merge with
    photon_paged_attention_reduce."""
    _check(lib().photon_paged_attention_partial_fp8(*_decode_fp8_args(
        q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale, out,
        max_context_len, partition_size, workspace, stream)), "photon_paged_attention_partial_fp8")


def photon_paged_attention_workspace_size(num_seqs, num_q_heads, head_dim, max_context_len,
                                          partition_size) -> int:
    return int(lib().photon_paged_attention_workspace_size(int(num_seqs), int(num_q_heads),
                                                          int(head_dim), int(max_context_len),
                                                          int(partition_size)))


def _decode_args(q, k_cache, v_cache, block_tables, context_lens, scale, out, max_context_len,
                 partition_size, workspace, stream):
    B, Hq, d = q.shape
    nb, Hkv, bs, d2 = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return (_p(q), _p(k_cache), _p(v_cache), _p(block_tables), _p(context_lens), float(scale),
            _p(out), B, Hq, Hkv, d, bs, nb, block_tables.shape[1], int(max_context_len),
            int(partition_size), _dt(k_cache), _dt(out), _p(workspace), ws_bytes, _stream(stream))


def photon_paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                                  max_context_len, partition_size=512, workspace=None,
                                  stream=None):
    """q [B, H_q, d]; caches [num_blocks, H_kv, bs, d]; block_tables int32
    [B, max_blocks]; context_lens int32 [B]; out [B, H_q, d] (float32 or
    bfloat16); workspace a device tensor of at least
    photon_paged_attention_workspace_size(...) bytes (None if that is 0)."""
    _check(lib().photon_paged_attention_decode(*_decode_args(
        q, k_cache, v_cache, block_tables, context_lens, scale, out, max_context_len,
        partition_size, workspace, stream)), "photon_paged_attention_decode")


def photon_paged_attention_partial(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                                   max_context_len, partition_size=512, workspace=None,
                                   stream=None):
    _check(lib().photon_paged_attention_partial(*_decode_args(
        q, k_cache, v_cache, block_tables, context_lens, scale, out, max_context_len,
        partition_size, workspace, stream)), "photon_paged_attention_partial")


def photon_paged_attention_decode_static(q, k_cache, v_cache, block_tables, context_lens, scale,
                                         out, max_context_len, partition_size=512, stream=None):
    """photon_paged_attention_decode without a workspace: for callers that may
    not allocate device memory.  The split-K partials live in a scratch array
    inside the library (STATIC_SCRATCH_BYTES, shared by every call on a
    device: calls that overlap on the GPU race)."""
    args = _decode_args(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                        max_context_len, partition_size, None, stream)
    _check(lib().photon_paged_attention_decode_static(*(args[:-3] + (args[-1],))),
           "photon_paged_attention_decode_static")


def photon_paged_attention_prefill(q, token_seq, positions, k_cache, v_cache, block_tables, scale,
                                   out, max_position, partition_size=512, workspace=None,
                                   stream=None):
    """Causal attention of query tokens q [T, H_q, d] (sequence token_seq[t],
    position positions[t]) over their sequences' pages; out [T, H_q, d]."""
    T, Hq, d = q.shape
    nb, Hkv, bs, d2 = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().photon_paged_attention_prefill(
        _p(q), _p(token_seq), _p(positions), _p(k_cache), _p(v_cache), _p(block_tables),
        float(scale), _p(out), T, block_tables.shape[0], Hq, Hkv, d, bs, nb, block_tables.shape[1],
        int(max_position), int(partition_size), _dt(k_cache), _dt(out), _p(workspace), ws_bytes,
        _stream(stream)), "photon_paged_attention_prefill")


def photon_paged_attention_reduce(context_lens, out, max_context_len, partition_size=512,
                                  workspace=None, stream=None):
    B, Hq, d = out.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().photon_paged_attention_reduce(_p(context_lens), _p(out), B, Hq, d,
                                               int(max_context_len), int(partition_size), _dt(out),
                                               _p(workspace), ws_bytes, _stream(stream)),
           "photon_paged_attention_reduce")


def photon_selftest_wait_timeout(budget_cycles: int, stream=None):
    """Launches a warp whose bounded wait on a never-completed mbarrier phase
    gives up (sets DEVERR_WAIT_TIMEOUT; read it with photon_device_errors)."""
    _check(lib().photon_selftest_wait_timeout(int(budget_cycles), _stream(stream)),
           "photon_selftest_wait_timeout")


def photon_device_errors(clear: bool = True) -> int:
    """Sticky DEVERR_* bits of the current device (synchronises the device)."""
    v = ctypes.c_uint32(0)
    _check(lib().photon_device_errors(ctypes.byref(v), int(bool(clear))), "photon_device_errors")
    return int(v.value)


# ---- host metadata ------------------------------------------------------------

def _np(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def photon_slot_mapping(block_tables, token_seq, positions, block_size=16) -> np.ndarray:
    bt, btp = _np(block_tables, np.int32)
    ts, tsp = _np(token_seq, np.int32)
    pos, posp = _np(positions, np.int32)
    out = np.empty(len(pos), np.int64)
    _check(lib().photon_slot_mapping(btp, bt.shape[0], bt.shape[1], tsp, posp, len(pos), block_size,
                                     out.ctypes.data_as(ctypes.c_void_p)), "photon_slot_mapping")
    return out


class BlockPool:
    """Physical block ids 0..num_blocks-1 from a seeded shuffled free list."""

    def __init__(self, num_blocks: int, seed: int = 0):
        h = ctypes.c_void_p()
        _check(lib().photon_block_pool_create(int(num_blocks), int(seed) & (2 ** 64 - 1),
                                              ctypes.byref(h)), "photon_block_pool_create")
        self._h = h

    @property
    def handle(self):
        return self._h

    def num_free(self) -> int:
        return int(lib().photon_block_pool_num_free(self._h))

    def alloc(self, n: int) -> np.ndarray:
        out = np.empty(int(n), np.int32)
        _check(lib().photon_block_pool_alloc(self._h, int(n), out.ctypes.data_as(ctypes.c_void_p)),
               "photon_block_pool_alloc")
        return out

    def free(self, ids) -> None:
        a, p = _np(ids, np.int32)
        _check(lib().photon_block_pool_free(self._h, p, len(a)), "photon_block_pool_free")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.photon_block_pool_destroy(h)
            self._h = None


def photon_build_step_metadata(num_computed_tokens, num_new_tokens, block_tables, pool=None,
                               block_size=16, max_tokens=None):
    """Host-side step metadata.  block_tables (int32 [B, max_blocks], -1
    padded) is grown in place.  Returns dict(token_seq, positions,
    slot_mapping, context_lens, max_context_len)."""
    nc, ncp = _np(num_computed_tokens, np.int32)
    nn, nnp = _np(num_new_tokens, np.int32)
    if not (isinstance(block_tables, np.ndarray) and block_tables.dtype == np.int32
            and block_tables.flags["C_CONTIGUOUS"]):
        raise TypeError("block_tables must be a C-contiguous int32 numpy array (updated in place)")
    B, W = block_tables.shape
    T = int(nn.sum()) if max_tokens is None else int(max_tokens)
    ts, pos = np.empty(max(T, 1), np.int32), np.empty(max(T, 1), np.int32)
    sm, cl = np.empty(max(T, 1), np.int64), np.empty(B, np.int32)
    nt, mc = ctypes.c_int32(0), ctypes.c_int32(0)
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(lib().photon_build_step_metadata(B, ncp, nnp, block_size, vp(block_tables), W,
                                            pool.handle if pool is not None else None, T, vp(ts),
                                            vp(pos), vp(sm), vp(cl), ctypes.byref(nt),
                                            ctypes.byref(mc)), "photon_build_step_metadata")
    n = nt.value
    return {"token_seq": ts[:n], "positions": pos[:n], "slot_mapping": sm[:n],
            "context_lens": cl, "max_context_len": mc.value}


# ---- two-phase scheduler ---------------------------------------------------------

REQ_WAITING, REQ_RUNNING, REQ_FINISHED, REQ_PREEMPTED = 0, 1, 2, 3


class _SchedConfig(ctypes.Structure):
    _fields_ = [("max_running", ctypes.c_int32), ("max_step_tokens", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("block_size", ctypes.c_int32)]


class _StepBatch(ctypes.Structure):
    _fields_ = [("max_seqs", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("request_ids", ctypes.c_void_p), ("num_new_tokens", ctypes.c_void_p),
                ("context_lens", ctypes.c_void_p), ("block_tables", ctypes.c_void_p),
                ("token_seq", ctypes.c_void_p), ("positions", ctypes.c_void_p),
                ("slot_mapping", ctypes.c_void_p), ("num_seqs", ctypes.c_int32),
                ("num_tokens", ctypes.c_int32), ("max_context_len", ctypes.c_int32),
                ("num_preempted", ctypes.c_int32), ("num_admitted", ctypes.c_int32)]


def _sched_lib():
    L = lib()
    if not getattr(L, "_sched_ready", False):
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.photon_scheduler_create.argtypes = [ctypes.POINTER(_SchedConfig), P, ctypes.POINTER(P)]
        L.photon_scheduler_create.restype = ctypes.c_int
        L.photon_scheduler_destroy.argtypes = [P]
        L.photon_scheduler_destroy.restype = None
        L.photon_scheduler_add_request.argtypes = [P, i64, i32, i32]
        L.photon_scheduler_add_request.restype = ctypes.c_int
        L.photon_scheduler_schedule.argtypes = [P, ctypes.POINTER(_StepBatch)]
        L.photon_scheduler_schedule.restype = ctypes.c_int
        L.photon_scheduler_complete_step.argtypes = [P]
        L.photon_scheduler_complete_step.restype = ctypes.c_int
        ip = ctypes.POINTER(i32)
        L.photon_scheduler_request_state.argtypes = [P, i64, ip, ip, ip]
        L.photon_scheduler_request_state.restype = ctypes.c_int
        L.photon_scheduler_counts.argtypes = [P, ip, ip, ip]
        L.photon_scheduler_counts.restype = ctypes.c_int
        L._sched_ready = True
    return L


class Scheduler:
    """Two-phase continuous-batching scheduler over a BlockPool (host C++)."""

    def __init__(self, pool: BlockPool, max_running: int, max_step_tokens: int,
                 max_blocks_per_seq: int, block_size: int = 16):
        L = _sched_lib()
        self.pool = pool  # keeps the pool alive
        self.cfg = _SchedConfig(max_running, max_step_tokens, max_blocks_per_seq, block_size)
        h = ctypes.c_void_p()
        _check(L.photon_scheduler_create(ctypes.byref(self.cfg), pool.handle, ctypes.byref(h)),
               "photon_scheduler_create")
        self._h = h
        self._ids = np.empty(max_running, np.int64)
        self._new = np.empty(max_running, np.int32)
        self._ctx = np.empty(max_running, np.int32)
        self._bt = np.empty((max_running, max_blocks_per_seq), np.int32)
        self._ts = np.empty(max_step_tokens, np.int32)
        self._pos = np.empty(max_step_tokens, np.int32)
        self._sm = np.empty(max_step_tokens, np.int64)
        vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)
        self._batch = _StepBatch(max_running, max_step_tokens, vp(self._ids), vp(self._new),
                                 vp(self._ctx), vp(self._bt), vp(self._ts), vp(self._pos),
                                 vp(self._sm), 0, 0, 0, 0, 0)

    def add_request(self, request_id: int, prompt_len: int, max_new_tokens: int) -> None:
        _check(_sched_lib().photon_scheduler_add_request(self._h, int(request_id), int(prompt_len),
                                                         int(max_new_tokens)),
               "photon_scheduler_add_request")

    def schedule(self, copy: bool = True) -> dict:
        """Plans one step; returns the batch arrays (copies, or views of the
        scheduler's buffers, valid until the next call, with copy=False)."""
        b = self._batch
        _check(_sched_lib().photon_scheduler_schedule(self._h, ctypes.byref(b)),
               "photon_scheduler_schedule")
        n, t = b.num_seqs, b.num_tokens
        c = (lambda a: a.copy()) if copy else (lambda a: a)
        return {"request_ids": c(self._ids[:n]), "num_new_tokens": c(self._new[:n]),
                "context_lens": c(self._ctx[:n]), "block_tables": c(self._bt[:n]),
                "token_seq": c(self._ts[:t]), "positions": c(self._pos[:t]),
                "slot_mapping": c(self._sm[:t]), "max_context_len": b.max_context_len,
                "num_preempted": b.num_preempted, "num_admitted": b.num_admitted}

    def complete_step(self) -> None:
        _check(_sched_lib().photon_scheduler_complete_step(self._h), "photon_scheduler_complete_step")

    def request_state(self, request_id: int):
        st, nc, ng = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(_sched_lib().photon_scheduler_request_state(self._h, int(request_id), ctypes.byref(st),
                                                           ctypes.byref(nc), ctypes.byref(ng)),
               "photon_scheduler_request_state")
        return st.value, nc.value, ng.value

    def counts(self):
        w, r, f = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(_sched_lib().photon_scheduler_counts(self._h, ctypes.byref(w), ctypes.byref(r),
                                                    ctypes.byref(f)), "photon_scheduler_counts")
        return w.value, r.value, f.value

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.photon_scheduler_destroy(h)
            self._h = None
