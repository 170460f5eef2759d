"""Host-side checks of the C ABI (no GPU needed): the library loads and
exports every symbol the header declares; arguments the host can check are
rejected before any launch; workspace sizing; and the ragged-batch metadata
builder (block pool, slot numbers, step metadata) against the oracle's slot
definition and the allocation invariants."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import synth
from tests.helpers import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pk():
    return ensure_built()


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "photon.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(photon_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(pk):
    names = _declared_symbols()
    assert "photon_kv_cache_write" in names and "photon_paged_attention_decode" in names
    L = ctypes.CDLL(pk.lib_path)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings_and_version(pk):
    assert pk.photon_status_string(0) == "ok"
    assert "invalid" in pk.photon_status_string(-1)
    assert pk.photon_status_string(12345) == "unknown status"
    assert pk.photon_version() >= 100


def _write(L, **kw):
    a = dict(k=1, v=1, pos=1, sm=1, kc=16, vc=16, T=4, H=2, d=64, bs=16, nb=8, dt=1, theta=1e4,
             style=0)
    a.update(kw)
    P = ctypes.c_void_p
    return L.photon_kv_cache_write(P(a["k"] * 16), P(a["v"] * 16), P(a["pos"] * 16), P(a["sm"] * 16),
                                   P(a["kc"] * 16), P(a["vc"] * 16), a["T"], a["H"], a["d"], a["bs"],
                                   a["nb"], a["dt"], a["theta"], a["style"], None)


def test_write_argument_validation_happens_before_launch(pk):
    L = pk.lib()
    assert _write(L, H=0) == -1
    assert _write(L, nb=0) == -1
    assert _write(L, T=-1) == -1
    assert _write(L, dt=7) == -1
    assert _write(L, style=9) == -1
    assert _write(L, theta=-1.0) == -1
    assert _write(L, theta=float("nan")) == -1
    assert _write(L, bs=32) == -2
    assert _write(L, d=48) == -2
    assert _write(L, k=0) == -1          # null pointer
    assert _write(L, T=0, k=0) == 0      # nothing to do is fine
    assert _write(L, style=2, theta=-1.0, T=0) == 0  # theta unused without rotation


def _decode(L, **kw):
    a = dict(q=16, kc=16, vc=16, bt=16, cl=16, scale=0.125, out=16, B=2, Hq=8, Hkv=2, d=64, bs=16,
             nb=100, mbps=4, maxctx=64, part=512, dt=1, odt=0, ws=0, wsb=0)
    a.update(kw)
    P = ctypes.c_void_p
    return L.photon_paged_attention_decode(
        P(a["q"]), P(a["kc"]), P(a["vc"]), P(a["bt"]), P(a["cl"]), a["scale"], P(a["out"]), a["B"],
        a["Hq"], a["Hkv"], a["d"], a["bs"], a["nb"], a["mbps"], a["maxctx"], a["part"], a["dt"],
        a["odt"], P(a["ws"]), a["wsb"], None)


def test_decode_argument_validation_happens_before_launch(pk):
    L = pk.lib()
    assert _decode(L, Hq=6, Hkv=4) == -1          # heads do not group
    assert _decode(L, Hq=32, Hkv=2) == -2         # group of 16 not compiled
    assert _decode(L, d=96) == -2
    assert _decode(L, dt=0, d=256) == -2          # fp32 storage stops at 128
    assert _decode(L, bs=8) == -2
    assert _decode(L, part=100) == -1             # not a multiple of the block size
    assert _decode(L, mbps=3) == -1               # table cannot hold max_context_len
    assert _decode(L, scale=float("inf")) == -1
    assert _decode(L, q=0) == -1
    assert _decode(L, q=8) == -1                  # misaligned for 16-byte loads
    assert _decode(L, kc=24) == -1                # misaligned for bulk copies
    assert _decode(L, out=20) == -1               # output rows are stored as 16-byte vectors
    assert _decode(L, maxctx=1024, mbps=64) == -3 # split needed, no workspace
    assert _decode(L, B=0) == 0


def test_workspace_size(pk):
    assert pk.photon_paged_attention_workspace_size(4, 8, 64, 512, 512) == 0
    assert pk.photon_paged_attention_workspace_size(4, 8, 64, 0, 512) == 0
    # 1025 tokens in 512-token partitions: 3 partitions, one more piece slot per
    # row (a page-balanced run may split one), plus one piece count per row
    # and the mode word (rounded up to 16 bytes), then the 16-byte control
    # block of the dynamic item order
    rows = 4 * 8
    n = rows * (3 + 1)
    al = lambda x: (x + 255) // 256 * 256
    a16 = lambda x: (x + 15) // 16 * 16
    assert pk.photon_paged_attention_workspace_size(4, 8, 64, 1025, 512) == (
        2 * al(n * 4) + al(n * 64 * 4) + al(a16((rows + 1) * 4) + 16))
    assert pk.photon_paged_attention_workspace_size(8, 8, 64, 1025, 512) == (
        2 * al(2 * n * 4) + al(2 * n * 64 * 4) + al(a16((2 * rows + 1) * 4) + 16))
    # a row count whose counts end on a 256-byte boundary: the control block
    # needs one more 256-byte unit
    assert pk.photon_paged_attention_workspace_size(1, 63, 64, 1025, 512) == (
        2 * al(63 * 4 * 4) + al(63 * 4 * 64 * 4) + al(a16(64 * 4) + 16))


# ---------------------------------------------------------------- metadata (host C++)

@pytest.mark.parametrize("name", synth.WORKLOADS)
def test_native_slot_mapping_is_bit_exact_against_oracle(pk, name):
    wl = synth.make(name)
    got = pk.photon_slot_mapping(wl.block_tables, wl.token_seq, wl.positions, wl.block_size)
    ref = oracle.slot_mapping(wl.block_tables, wl.token_seq, wl.positions, wl.block_size)
    assert got.dtype == np.int64 and np.array_equal(got, ref)


def test_native_slot_mapping_edge_cases(pk):
    rng = np.random.default_rng(0)
    bt = rng.integers(-1, 50, size=(5, 7)).astype(np.int32)
    ts = rng.integers(0, 5, size=400).astype(np.int32)
    pos = rng.integers(-3, 7 * 16 + 5, size=400).astype(np.int32)
    assert np.array_equal(pk.photon_slot_mapping(bt, ts, pos), oracle.slot_mapping(bt, ts, pos, 16))
    with pytest.raises(pk.PhotonError):
        pk.photon_slot_mapping(bt, np.array([5], np.int32), np.array([0], np.int32))


def test_block_pool_invariants(pk):
    pool = pk.BlockPool(1000, seed=3)
    assert pool.num_free() == 1000
    a = pool.alloc(300)
    b = pool.alloc(700)
    ids = np.concatenate([a, b])
    assert sorted(ids.tolist()) == list(range(1000))           # a permutation of the pool
    assert not np.array_equal(ids, np.arange(1000))            # shuffled
    with pytest.raises(pk.PhotonError) as e:
        pool.alloc(1)
    assert e.value.status == -5
    pool.free(a[:10])
    with pytest.raises(pk.PhotonError):
        pool.free(a[:1])                                       # double free
    with pytest.raises(pk.PhotonError):
        pool.free(np.array([b[0], b[0]], np.int32))            # repeat inside one call
    with pytest.raises(pk.PhotonError):
        pool.free(np.array([1000], np.int32))                  # out of range
    assert pool.num_free() == 10
    pool.free(b[:5])                                           # earlier failures changed nothing
    assert pool.num_free() == 15
    # same seed, same order
    assert np.array_equal(pk.BlockPool(50, 9).alloc(50), pk.BlockPool(50, 9).alloc(50))
    assert not np.array_equal(pk.BlockPool(50, 9).alloc(50), pk.BlockPool(50, 10).alloc(50))


def test_step_metadata_two_phase_step(pk):
    # 3 running requests continue (one token each), 2 waiting requests are
    # admitted with 100-token prompts (100 + 1 tokens), 1 idle row
    pool = pk.BlockPool(200, seed=1)
    computed = np.array([5, 16, 31, 0, 0, 9], np.int32)
    new = np.array([1, 1, 1, 101, 101, 0], np.int32)
    bt = np.full((6, 8), -1, np.int32)
    for s, c in enumerate(computed):
        n = -(-int(c) // 16)
        bt[s, :n] = pool.alloc(n)
    before = bt.copy()
    md = pk.photon_build_step_metadata(computed, new, bt, pool)
    assert md["context_lens"].tolist() == (computed + new).tolist()
    assert md["max_context_len"] == 101
    assert md["token_seq"].tolist() == [0, 1, 2] + [3] * 101 + [4] * 101
    assert md["positions"].tolist() == [5, 16, 31] + list(range(101)) * 2
    # previously allocated entries stay; rows grow to cover their context
    assert np.array_equal(bt[before >= 0], before[before >= 0])
    for s, c in enumerate(md["context_lens"]):
        n = -(-int(c) // 16)
        assert (bt[s, :n] >= 0).all() and (bt[s, n:] == -1).all()
    used = bt[bt >= 0]
    assert len(set(used.tolist())) == len(used)                # no block shared
    assert pool.num_free() == 200 - len(used)
    ref = oracle.slot_mapping(bt, md["token_seq"], md["positions"], 16)
    assert np.array_equal(md["slot_mapping"], ref)
    assert len(set(md["slot_mapping"].tolist())) == len(ref)


def test_step_metadata_fails_without_side_effects(pk):
    pool = pk.BlockPool(3, seed=0)
    bt = np.full((2, 4), -1, np.int32)
    with pytest.raises(pk.PhotonError) as e:
        pk.photon_build_step_metadata([0, 0], [40, 40], bt, pool)  # needs 6 blocks
    assert e.value.status == -5
    assert pool.num_free() == 3 and (bt == -1).all()
    with pytest.raises(pk.PhotonError):
        pk.photon_build_step_metadata([0], [65], np.full((1, 4), -1, np.int32), pool)  # row overflow
    with pytest.raises(pk.PhotonError):
        pk.photon_build_step_metadata([0], [1], np.full((1, 4), -1, np.int32), None)  # needs a pool


def test_selftest_rejects_a_zero_budget(pk):
    # checked on the host before any launch (no device needed)
    assert pk.lib().photon_selftest_wait_timeout(0, None) == -1  # PHOTON_ERR_INVALID_ARG
