"""Pins for the fp64 CPU oracle: each check ties an oracle function to
something other than itself -- IEEE-754 facts, closed forms, invariants, a
library routine on a special case, or a brute-force loop on tiny inputs --
chosen so that a plausible slip (a dropped term, a flipped sign, a swapped
index, a transposed head grouping, double rounding) fails at least one.

The method is the one in the PhotonInfer README, "Technical details > Paged
attention" and "Key features > GPU-optimised kernels" (batched RoPE,
numerically stable softmax)."""
import cmath
import math

import numpy as np
import pytest

import oracle
import synth


# ---------------------------------------------------------------- bf16 rounding

def _bf16_bits_of_f32(x32: np.ndarray) -> np.ndarray:
    import torch
    return torch.from_numpy(x32.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_round_bf16_matches_single_rounding_of_floats():
    # For float-representable inputs a float->bf16 RNE conversion (torch) is a
    # single correct rounding: the oracle must agree bit for bit.
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(4000), rng.standard_normal(2000) * 1e-3,
                        rng.standard_normal(2000) * 1e4]).astype(np.float32)
    ref = _bf16_bits_of_f32(x)
    got = np.array([oracle.round_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(ref, got)


def test_round_bf16_ties_go_to_even_and_no_double_rounding():
    rng = np.random.default_rng(2)
    for _ in range(500):
        # two adjacent bf16 numbers b < b' and their exact midpoint
        bits = int(rng.integers(0x3000, 0x4F00)) & ~1  # even mantissa
        lo = oracle.bf16_to_f64(np.array([bits], np.uint16))[0]
        hi = oracle.bf16_to_f64(np.array([bits + 1], np.uint16))[0]
        mid = (lo + hi) / 2
        assert oracle.round_bf16(mid) == bits                # tie -> even (lower here)
        assert oracle.round_bf16(-mid) == (bits | 0x8000)
        # a hair above the midpoint must round up.  Going through float first
        # would collapse mid*(1+2^-40) onto mid and then round to even: wrong.
        assert oracle.round_bf16(mid * (1 + 2.0 ** -40)) == bits + 1
        assert oracle.round_bf16(mid * (1 - 2.0 ** -40)) == bits
        # odd lower neighbour: the tie goes up to the even one
        lo2 = oracle.bf16_to_f64(np.array([bits + 1], np.uint16))[0]
        hi2 = oracle.bf16_to_f64(np.array([bits + 2], np.uint16))[0]
        assert oracle.round_bf16((lo2 + hi2) / 2) == bits + 2


def test_round_bf16_edges():
    assert oracle.round_bf16(0.0) == 0
    assert oracle.round_bf16(-0.0) == 0x8000
    assert oracle.round_bf16(1.0) == 0x3F80
    assert oracle.round_bf16(-2.0) == 0xC000
    assert oracle.round_bf16(float("inf")) == 0x7F80
    # largest finite bf16 is (2 - 2^-7) * 2^127; half a step above overflows
    assert oracle.round_bf16((2 - 2 ** -7) * 2.0 ** 127) == 0x7F7F
    assert oracle.round_bf16((2 - 2 ** -8) * 2.0 ** 127) == 0x7F80
    # subnormal spacing is 2^-133: 1.5 * 2^-133 ties to the even code 2
    assert oracle.round_bf16(1.5 * 2.0 ** -133) == 0x0002
    assert oracle.round_bf16(2.0 ** -133) == 0x0001
    assert oracle.round_bf16(0.4 * 2.0 ** -133) == 0x0000


# ---------------------------------------------------------------- RoPE

def _rope_complex(x, pos, theta, style):
    """RoPE as multiplication of each pair, seen as a complex number, by
    exp(i * pos * theta^(-2i/d)) -- the rotary form, written with cmath."""
    d = len(x)
    y = np.array(x, dtype=np.float64)
    for i in range(d // 2):
        a, b = (i, i + d // 2) if style == oracle.ROPE_NEOX else (2 * i, 2 * i + 1)
        w = math.exp(-2.0 * i / d * math.log(theta))
        z = complex(x[a], x[b]) * cmath.exp(1j * pos * w)
        y[a], y[b] = z.real, z.imag
    return y


@pytest.mark.parametrize("style", [oracle.ROPE_NEOX, oracle.ROPE_GPTJ])
@pytest.mark.parametrize("d", [8, 32, 64, 128])
def test_rope_equals_complex_rotation(style, d):
    rng = np.random.default_rng(d + 10 * style)
    for pos in [0, 1, 2, 17, 1023, 32767]:
        for theta in [1e4, 5e5, 1e6]:
            x = rng.standard_normal(d)
            got = oracle.rope(x, pos, theta, style)
            ref = _rope_complex(x, pos, theta, style)
            # the two differ only by fp64 rounding of the angle (|angle| < 4e4)
            np.testing.assert_allclose(got, ref, rtol=0, atol=1e-10)


def test_rope_position_zero_is_identity_and_none_style():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(64)
    assert np.array_equal(oracle.rope(x, 0, 1e4, oracle.ROPE_NEOX), x)
    assert np.array_equal(oracle.rope(x, 0, 1e4, oracle.ROPE_GPTJ), x)
    assert np.array_equal(oracle.rope(x, 777, 1e4, oracle.ROPE_NONE), x)


def test_rope_pairs_keep_norm_and_first_pair_turns_one_radian_per_step():
    rng = np.random.default_rng(4)
    d = 64
    x = rng.standard_normal(d)
    y = oracle.rope(x, 5, 1e4, oracle.ROPE_NEOX)
    for i in range(d // 2):
        assert math.isclose(math.hypot(x[i], x[i + d // 2]), math.hypot(y[i], y[i + d // 2]),
                            rel_tol=1e-14)
    # pair 0 has frequency theta^0 = 1: unit vector e_0 at position 1 -> (cos 1, sin 1)
    e = np.zeros(d)
    e[0] = 1.0
    r = oracle.rope(e, 1, 1e4, oracle.ROPE_NEOX)
    assert math.isclose(r[0], math.cos(1.0), abs_tol=1e-15)
    assert math.isclose(r[d // 2], math.sin(1.0), abs_tol=1e-15)
    # last pair: frequency theta^(-(d-2)/d)
    e = np.zeros(d)
    e[d // 2 - 1] = 1.0
    r = oracle.rope(e, 1, 1e4, oracle.ROPE_NEOX)
    ang = math.atan2(r[d - 1], r[d // 2 - 1])
    assert math.isclose(ang, 1e4 ** (-(d - 2) / d), rel_tol=1e-12)


def test_rope_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(5)
    d = 64
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    for m, n in [(3, 11), (100, 40), (5000, 5001)]:
        base = oracle.rope(q, m, 5e5) @ oracle.rope(k, n, 5e5)
        for c in [1, 77, 9000]:
            shifted = oracle.rope(q, m + c, 5e5) @ oracle.rope(k, n + c, 5e5)
            assert math.isclose(base, shifted, rel_tol=1e-9, abs_tol=1e-9)


def test_rope_neox_and_gptj_are_a_fixed_permutation_apart():
    rng = np.random.default_rng(6)
    d = 32
    perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])  # interleaved -> halves
    x = rng.standard_normal(d)
    a = oracle.rope(x, 123, 1e4, oracle.ROPE_GPTJ)
    b = oracle.rope(x[perm], 123, 1e4, oracle.ROPE_NEOX)
    np.testing.assert_array_equal(a[perm], b)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rope_rows_is_one_rounding_of_the_complex_rotation(dtype):
    rng = np.random.default_rng(16)
    n, h, d = 5, 3, 64
    x = rng.standard_normal((n, h, d))
    if dtype == "f32":
        xs = x.astype(np.float32)
    else:
        xs = np.vectorize(oracle.round_bf16, otypes=[np.uint16])(x)
    pos = np.array([0, 1, 77, 4096, 32767], np.int32)
    y = oracle.rope_rows(xs, pos, 5e5)
    assert np.array_equal(y[0], xs[0])                      # position 0: unchanged bits
    for r in range(n):
        for k in range(h):
            ref = _rope_complex(oracle.to_f64(xs[r, k]), int(pos[r]), 5e5, oracle.ROPE_NEOX)
            got = oracle.to_f64(y[r, k])
            ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
            if dtype == "bf16":
                ulp = ulp * 2.0 ** 16
            assert (np.abs(got - ref) <= ulp).all()


# ---------------------------------------------------------------- slot mapping

def test_slot_mapping_invariants():
    wl = synth.make_custom([1, 15, 16, 17, 33, 100], 4, 2, 32, tokens_per_seq=40, seed=7)
    bt = wl.block_tables
    bs = wl.block_size
    # every (seq, position) of every sequence
    ts = np.concatenate([np.full(c, s, np.int32) for s, c in enumerate(wl.context_lens)])
    pos = np.concatenate([np.arange(c, dtype=np.int32) for c in wl.context_lens])
    sl = oracle.slot_mapping(bt, ts, pos, bs)
    assert (sl >= 0).all()
    assert len(set(sl.tolist())) == len(sl)                   # no two tokens share a slot
    for s, p, x in zip(ts, pos, sl):
        assert x // bs in set(bt[s][bt[s] >= 0].tolist())     # slot lies in the sequence's blocks
        assert x % bs == p % bs                                # offset within the block
    # consecutive positions inside one block are consecutive slots
    same_blk = (pos[1:] // bs == pos[:-1] // bs) & (ts[1:] == ts[:-1])
    assert (np.diff(sl)[same_blk] == 1).all()
    # unmapped cases give -1
    bad = oracle.slot_mapping(bt, np.array([0, 0], np.int32), np.array([-1, bt.shape[1] * bs], np.int32), bs)
    assert bad.tolist() == [-1, -1]
    bt2 = bt.copy()
    bt2[5, 3] = -1
    assert oracle.slot_mapping(bt2, np.array([5], np.int32), np.array([3 * bs + 2], np.int32), bs)[0] == -1


# ---------------------------------------------------------------- cache write

def _tagged(shape, start):
    # values that are exact in bf16 and fp32 and unique per element (mod 2^8 steps)
    n = int(np.prod(shape))
    return (start + np.arange(n, dtype=np.float64)).reshape(shape)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("style", [oracle.ROPE_NEOX, oracle.ROPE_GPTJ, oracle.ROPE_NONE])
def test_kv_cache_write_placement_rotation_and_canaries(dtype, style):
    rng = np.random.default_rng(8)
    T, H, d, bs, nb = 7, 2, 32, 16, 6
    def store(x):
        x = np.asarray(x, np.float64)
        if dtype == "f32":
            return x.astype(np.float32)
        return np.vectorize(oracle.round_bf16, otypes=[np.uint16])(x)
    k = store(rng.standard_normal((T, H, d)))
    v = store(rng.standard_normal((T, H, d)))
    canary = store(np.full((nb, H, bs, d), -7.25))
    kc, vc = canary.copy(), canary.copy()
    slots = np.array([0, 17, 95, -1, 40, 41, 63], np.int64)
    pos = np.array([0, 3, 900, 5, 31, 32, 20000], np.int32)
    oracle.kv_cache_write(k, v, pos, slots, kc, vc, 1e4, style)
    written = np.zeros((nb, H, bs), bool)
    for t in range(T):
        if slots[t] < 0:
            continue
        b, o = slots[t] // bs, slots[t] % bs
        written[b, :, o] = True
        for h in range(H):
            assert np.array_equal(vc[b, h, o], v[t, h])        # V is a bit copy
            x = oracle.to_f64(k[t, h])
            ref = x if style == oracle.ROPE_NONE else _rope_complex(x, int(pos[t]), 1e4, style)
            got = oracle.to_f64(kc[b, h, o])
            if style == oracle.ROPE_NONE:
                assert np.array_equal(kc[b, h, o], k[t, h])
            else:
                # one rounding of nearly equal doubles: at most one step apart
                ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
                if dtype == "bf16":
                    ulp = ulp * 2.0 ** 16
                assert (np.abs(got - ref) <= ulp).all()
    assert np.array_equal(kc[~written], canary[~written])      # nothing else touched
    assert np.array_equal(vc[~written], canary[~written])


def test_kv_cache_write_rejects_slots_outside_pool():
    k = np.zeros((1, 1, 8), np.float32)
    kc = np.zeros((2, 1, 16, 8), np.float32)
    with pytest.raises(ValueError):
        oracle.kv_cache_write(k, k, np.array([0], np.int32), np.array([32], np.int64), kc, kc.copy(), 1e4)


# ---------------------------------------------------------------- attention

def _rand_case(rng, ctx, Hq, Hkv, d, bs=16, dtype="f32", pool_extra=3):
    nblk = [-(-c // bs) for c in ctx]
    nb = sum(nblk) + pool_extra
    perm = rng.permutation(nb)
    width = max(max(nblk), 1)
    bt = np.full((len(ctx), width), -1, np.int32)
    i = 0
    for s, n in enumerate(nblk):
        bt[s, :n] = perm[i:i + n]
        i += n
    q = rng.standard_normal((len(ctx), Hq, d))
    kc = rng.standard_normal((nb, Hkv, bs, d))
    vc = rng.standard_normal((nb, Hkv, bs, d))
    if dtype == "f32":
        cast = lambda a: a.astype(np.float32)
    else:
        cast = lambda a: np.vectorize(oracle.round_bf16, otypes=[np.uint16])(a)
    return cast(q), cast(kc), cast(vc), bt, np.array(ctx, np.int32)


def _gather(cache, bt, s, ctx, bs):
    """Contiguous [H_kv, ctx, d] copy of sequence s's KV, by numpy indexing."""
    j = np.arange(ctx)
    blk = bt[s, j // bs]
    return np.transpose(oracle.to_f64(cache)[blk, :, j % bs, :], (1, 0, 2))


def _bruteforce(q, kc, vc, bt, cl, scale):
    """Triple loop in pure Python floats, two-pass softmax."""
    B, Hq, d = q.shape
    Hkv, bs = kc.shape[1], kc.shape[2]
    G = Hq // Hkv
    qd, kd, vd = oracle.to_f64(q), oracle.to_f64(kc), oracle.to_f64(vc)
    out = np.zeros((B, Hq, d))
    for s in range(B):
        for g in range(Hq):
            h = g // G
            sc = []
            for j in range(int(cl[s])):
                b, o = int(bt[s][j // bs]), j % bs
                sc.append(scale * sum(float(qd[s, g, e]) * float(kd[b, h, o, e]) for e in range(d)))
            if not sc:
                continue
            m = max(sc)
            w = [math.exp(x - m) for x in sc]
            tot = sum(w)
            for e in range(d):
                acc = 0.0
                for j in range(int(cl[s])):
                    b, o = int(bt[s][j // bs]), j % bs
                    acc += w[j] / tot * float(vd[b, h, o, e])
                out[s, g, e] = acc
    return out


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_attention_matches_bruteforce_triple_loop(dtype):
    rng = np.random.default_rng(9)
    for ctx, Hq, Hkv, d in [([5, 19], 4, 2, 32), ([1, 40, 16, 17], 4, 1, 8), ([33, 2], 6, 3, 16)]:
        q, kc, vc, bt, cl = _rand_case(rng, ctx, Hq, Hkv, d, dtype=dtype)
        scale = 1 / math.sqrt(d)
        got = oracle.paged_attention(q, kc, vc, bt, cl, scale)
        np.testing.assert_allclose(got, _bruteforce(q, kc, vc, bt, cl, scale), rtol=0, atol=1e-12)


def test_attention_equals_library_sdpa_on_gathered_kv():
    # paged attention == textbook attention over the KV gathered contiguously
    # (torch's scaled_dot_product_attention in float64 on CPU, GQA by
    # repeating each KV head over its group of query heads)
    import torch
    rng = np.random.default_rng(10)
    ctx, Hq, Hkv, d, bs = [5, 19, 64, 130, 1], 8, 2, 64, 16
    q, kc, vc, bt, cl = _rand_case(rng, ctx, Hq, Hkv, d, bs, dtype="bf16")
    scale = 0.3
    got = oracle.paged_attention(q, kc, vc, bt, cl, scale)
    for s, c in enumerate(ctx):
        K = torch.from_numpy(_gather(kc, bt, s, c, bs)).repeat_interleave(Hq // Hkv, 0)
        V = torch.from_numpy(_gather(vc, bt, s, c, bs)).repeat_interleave(Hq // Hkv, 0)
        Q = torch.from_numpy(oracle.to_f64(q[s]))[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=scale)[:, 0, :]
        np.testing.assert_allclose(got[s], ref.numpy(), rtol=0, atol=1e-12)


def test_attention_invariant_to_relabelling_physical_blocks():
    rng = np.random.default_rng(11)
    q, kc, vc, bt, cl = _rand_case(rng, [37, 80, 3], 4, 2, 32, dtype="bf16", pool_extra=9)
    base = oracle.paged_attention(q, kc, vc, bt, cl, 0.2)
    pi = rng.permutation(kc.shape[0])
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[pi], vc2[pi] = kc, vc
    bt2 = np.where(bt >= 0, pi[np.maximum(bt, 0)], -1).astype(np.int32)
    assert np.array_equal(oracle.paged_attention(q, kc2, vc2, bt2, cl, 0.2), base)


def test_softmax_weights_are_a_distribution():
    rng = np.random.default_rng(12)
    q, kc, vc, bt, cl = _rand_case(rng, [1, 7, 300], 4, 4, 16)
    _, w = oracle.paged_attention(q, kc, vc, bt, cl, 1.0, return_weights=True)
    for s, c in enumerate(cl):
        assert (w[s, :, :c] > 0).all() and (w[s, :, c:] == 0).all()
        np.testing.assert_allclose(w[s, :, :c].sum(-1), 1.0, rtol=0, atol=1e-12)


def test_closed_forms():
    rng = np.random.default_rng(13)
    Hq, Hkv, d, bs = 4, 2, 32, 16
    q, kc, vc, bt, cl = _rand_case(rng, [1, 23, 50], Hq, Hkv, d, dtype="f32")
    # context 1: the output is that token's V, exactly
    out = oracle.paged_attention(q, kc, vc, bt, cl, 0.17)
    for g in range(Hq):
        assert np.array_equal(out[0, g], oracle.to_f64(vc[bt[0, 0], g // 2, 0]))
    # q = 0: uniform weights, the output is the mean of V over the context
    q0 = np.zeros_like(q)
    out0 = oracle.paged_attention(q0, kc, vc, bt, cl, 0.17)
    for s, c in enumerate(cl):
        for g in range(Hq):
            np.testing.assert_allclose(out0[s, g], _gather(vc, bt, s, c, bs)[g // 2].mean(0), atol=1e-13)
    # all keys equal: again the mean of V
    kc_eq = np.broadcast_to(kc[:1, :, :1, :], kc.shape).copy()
    outk = oracle.paged_attention(q, kc_eq, vc, bt, cl, 0.17)
    for s, c in enumerate(cl):
        for g in range(Hq):
            np.testing.assert_allclose(outk[s, g], _gather(vc, bt, s, c, bs)[g // 2].mean(0), atol=1e-13)
    # context 0 gives a zero row
    cl0 = cl.copy()
    cl0[1] = 0
    assert (oracle.paged_attention(q, kc, vc, bt, cl0, 0.17)[1] == 0).all()


def test_gqa_grouping_is_contiguous():
    # One token of KV head h gets a key aligned with every query and a scale
    # that makes its score dominate: query heads g with g // G == h must
    # return that token's V; the others must not.
    rng = np.random.default_rng(14)
    Hq, Hkv, d, bs = 8, 4, 16, 16
    G = Hq // Hkv
    q, kc, vc, bt, cl = _rand_case(rng, [20], Hq, Hkv, d, dtype="f32")
    q[:] = 1.0
    h_hot, j_hot = 1, 13
    b, o = bt[0, j_hot // bs], j_hot % bs
    kc[b, h_hot, o, :] = 50.0
    out = oracle.paged_attention(q, kc, vc, bt, cl, 1.0)
    for g in range(Hq):
        hit = np.allclose(out[0, g], vc[b, h_hot, o], atol=1e-9)
        assert hit == (g // G == h_hot), g


@pytest.mark.parametrize("part", [16, 32, 48, 512])
def test_split_k_lse_merge_equals_unpartitioned(part):
    rng = np.random.default_rng(15)
    q, kc, vc, bt, cl = _rand_case(rng, [1, 16, 17, 100, 513, 700], 4, 2, 32, dtype="bf16")
    a = oracle.paged_attention(q, kc, vc, bt, cl, 0.3)
    b = oracle.paged_attention_split(q, kc, vc, bt, cl, 0.3, part)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_step_composition_attends_to_the_new_token():
    # write first, then attend: a new token whose key dominates every score
    # must show up as (almost) the whole output
    wl = synth.make("tiny_fp32")
    vals = synth.make_values(wl)
    q = synth.to_storage_numpy(vals["q"][0])
    k = synth.to_storage_numpy(vals["k"][0]).copy()
    v = synth.to_storage_numpy(vals["v"][0])
    kc = synth.to_storage_numpy(vals["k_cache"][0]).copy()
    vc = synth.to_storage_numpy(vals["v_cache"][0]).copy()
    sm = oracle.slot_mapping(wl.block_tables, wl.token_seq, wl.positions, wl.block_size)
    q[:] = 1.0
    k[:] = 40.0
    out = oracle.decode_step(q, k, v, wl.positions, sm, kc, vc, wl.block_tables, wl.context_lens,
                             1.0, wl.rope_theta, oracle.ROPE_NONE)
    for t in range(wl.num_tokens):
        s = wl.token_seq[t]
        for g in range(wl.num_q_heads):
            np.testing.assert_allclose(out[s, g], v[t, g // 2], atol=1e-9)


def test_tiny_config_oracle_is_fast():
    import time
    wl = synth.make("tiny_fp32")
    vals = synth.make_values(wl)
    t0 = time.time()
    sm = oracle.slot_mapping(wl.block_tables, wl.token_seq, wl.positions, wl.block_size)
    kc = synth.to_storage_numpy(vals["k_cache"][0]).copy()
    vc = synth.to_storage_numpy(vals["v_cache"][0]).copy()
    oracle.decode_step(synth.to_storage_numpy(vals["q"][0]), synth.to_storage_numpy(vals["k"][0]),
                       synth.to_storage_numpy(vals["v"][0]), wl.positions, sm, kc, vc,
                       wl.block_tables, wl.context_lens, wl.scale, wl.rope_theta)
    assert time.time() - t0 < 1.0


# ---------------------------------------------------------------- FP8 E4M3 cache

def test_fp8_decode_all_codes_match_torch():
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.fp8_decode(c) for c in codes])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(ref[~np.isnan(ref)], got[~np.isnan(got)])
    assert oracle.fp8_decode(0x7E) == 448.0 and oracle.fp8_decode(0x01) == 2.0 ** -9


def test_fp8_encode_rounds_to_nearest_even_and_saturates():
    import torch
    rng = np.random.default_rng(17)
    x = np.concatenate([rng.standard_normal(5000) * 40, rng.standard_normal(2000) * 0.01]).astype(np.float32)
    x = x[np.abs(x) < 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(np.array([oracle.fp8_encode(float(v)) for v in x], np.uint8), ref)
    # exact midpoints between neighbours go to the even code
    for c in range(1, 0x7D):
        lo, hi = oracle.fp8_decode(c), oracle.fp8_decode(c + 1)
        even = c if c % 2 == 0 else c + 1
        assert oracle.fp8_encode((lo + hi) / 2) == even
        assert oracle.fp8_encode((lo + hi) / 2 * (1 + 1e-12)) == c + 1
    # beyond the largest finite value: saturate, keep the sign
    for v in (448.0, 464.0, 500.0, 1e30):
        assert oracle.fp8_encode(v) == 0x7E and oracle.fp8_encode(-v) == 0xFE
    assert oracle.fp8_encode(float("nan")) == 0x7F
    assert oracle.fp8_encode(2.0 ** -10) == 0x00 and oracle.fp8_encode(1.5 * 2.0 ** -10) == 0x01


def test_fp8_write_layout_and_dequant():
    rng = np.random.default_rng(18)
    T, H, d, bs, nb = 5, 2, 64, 16, 6
    k = rng.standard_normal((T, H, d)).astype(np.float32)
    v = rng.standard_normal((T, H, d)).astype(np.float32)
    ks, vs = np.array([0.01, 0.02], np.float32), np.array([0.03, 0.005], np.float32)
    kc = np.full((nb, H, bs, d), 0x55, np.uint8)
    vc = np.full((nb, H, d, bs), 0x55, np.uint8)
    slots = np.array([3, 17, -1, 90, 40], np.int64)
    pos = np.array([1, 9, 4, 1000, 0], np.int32)
    oracle.kv_cache_write_fp8(k, v, pos, slots, kc, vc, ks, vs, 1e4)
    touched_k = np.zeros(kc.shape, bool)
    touched_v = np.zeros(vc.shape, bool)
    for t in range(T):
        if slots[t] < 0:
            continue
        b, o = slots[t] // bs, slots[t] % bs
        for h in range(H):
            rot = _rope_complex(k[t, h].astype(np.float64), int(pos[t]), 1e4, oracle.ROPE_NEOX)
            got_k = np.array([oracle.fp8_decode(c) for c in kc[b, h, o]]) * ks[h]
            assert np.abs(got_k - rot).max() <= np.abs(rot).max() * 2.0 ** -4 + 2.0 ** -9 * ks[h]
            codes_v = np.array([oracle.fp8_encode(float(x) / float(vs[h])) for x in v[t, h]],
                               np.uint8)
            assert np.array_equal(vc[b, h, :, o], codes_v)         # dims outer, tokens inner
            touched_k[b, h, o, :] = True
            touched_v[b, h, :, o] = True
    assert (kc[~touched_k] == 0x55).all() and (vc[~touched_v] == 0x55).all()
    kd, vd = oracle.fp8_dequant(kc, vc, ks, vs)
    for t in (0, 1, 3, 4):
        b, o = slots[t] // bs, slots[t] % bs
        for h in range(H):
            assert np.array_equal(vd[b, h, o], np.array([oracle.fp8_decode(c) for c in vc[b, h, :, o]]) * np.float64(vs[h]))


def _e4m3_nearest_exact(q):
    """Nearest E4M3 code to the rational q by exhaustive search over the 254
    finite codes, ties to the even code, magnitudes beyond 448 saturating.
    Independent of the oracle: values come from the format's definition
    (bias 7, 3 mantissa bits, subnormal spacing 2^-9)."""
    from fractions import Fraction as Fr
    if q >= 448:
        return 0x7E
    if q <= -448:
        return 0xFE
    best = None
    for code in range(256):
        e, m = (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            continue  # NaN
        mag = Fr(m, 512) if e == 0 else Fr(8 + m, 8) * Fr(2) ** (e - 7)
        val = -mag if code & 0x80 else mag
        if val == 0 and (code & 0x80) != (0x80 if q < 0 else 0):
            continue  # keep the zero of q's sign
        key = (abs(val - q), code & 1)
        if best is None or key < best[0]:
            best = (key, code)
    return best[1]


def _fp8_tie_cases(rng, n):
    """(x, s) float32 pairs with x / s exactly a midpoint of two adjacent
    E4M3 values: s is an odd integer of 19 bits times a power of two (so 1/s
    is not exact in any binary format) and x = mid * s is exact in float."""
    vals = sorted({oracle.fp8_decode(c) for c in range(0x7E + 1)})
    cases = []
    while len(cases) < n:
        k = int(rng.integers(0, len(vals) - 1))
        mid = (vals[k] + vals[k + 1]) / 2
        s = float(int(rng.integers(2 ** 18, 2 ** 19)) | 1) * 2.0 ** int(rng.integers(-30, -20))
        x = mid * s * (1 if rng.random() < 0.5 else -1)
        if np.float32(x) == x and np.float32(s) == s:
            cases.append((np.float32(x), np.float32(s)))
    return cases


def _fp8_near_tie_cases(rng, n):
    """(x, s) with x / s within about 2^-24 (relative) of an E4M3 midpoint but
    not on it: rounding the quotient to float first would land on the
    midpoint and then round to even."""
    vals = sorted({oracle.fp8_decode(c) for c in range(0x7E + 1)})
    cases = []
    while len(cases) < n:
        k = int(rng.integers(1, len(vals) - 1))
        mid = (vals[k] + vals[k + 1]) / 2
        x = np.float32(rng.uniform(0.5, 4.0))
        s = np.float32(float(x) / mid)
        if float(x) / float(s) != mid:
            cases.append((x, s))
    return cases


def _fp8_write_one(x, s):
    """K (no rotation) and V codes the oracle writes for one token whose K row
    is all x and V row all -x, with scale s on its single KV head."""
    d, bs = 32, 16
    k = np.full((1, 1, d), x, np.float32)
    v = np.full((1, 1, d), -x, np.float32)
    kc = np.zeros((1, 1, bs, d), np.uint8)
    vc = np.zeros((1, 1, d, bs), np.uint8)
    sc = np.array([s], np.float32)
    oracle.kv_cache_write_fp8(k, v, np.array([7], np.int32), np.array([3], np.int64), kc, vc,
                              sc, sc, 1e4, oracle.ROPE_NONE)
    assert (kc[0, 0, 3] == kc[0, 0, 3, 0]).all() and (vc[0, 0, :, 3] == vc[0, 0, 0, 3]).all()
    return int(kc[0, 0, 3, 0]), int(vc[0, 0, 0, 3])


def test_fp8_write_codes_are_the_nearest_e4m3_of_the_exact_quotient():
    """The FP8 write's codes, for K (no rotation) and V, equal the nearest
    E4M3 of the exact rational x / scale (exhaustive search, ties to even).
    The cases are exact midpoints, values a hair beside a midpoint, and
    random values; the first two are where plausible slips show: multiplying
    by a rounded reciprocal (in fp64 or fp32) misses some ties, and rounding
    the quotient to float before E4M3 rounds twice."""
    from fractions import Fraction as Fr
    rng = np.random.default_rng(31)
    ties = _fp8_tie_cases(rng, 300)
    near = _fp8_near_tie_cases(rng, 100)
    rand = [(np.float32(rng.standard_normal() * 3), np.float32(rng.uniform(0.5, 1.5) * 4 / 448))
            for _ in range(100)]
    exact = lambda x, s: _e4m3_nearest_exact(Fr(float(x)) / Fr(float(s)))
    # the cases see each slip
    f32 = np.float32
    assert sum(_e4m3_nearest_exact(Fr(float(x) * (1.0 / float(s)))) != exact(x, s) for x, s in ties) >= 5
    assert sum(_e4m3_nearest_exact(Fr(float(f32(x * (f32(1) / s))))) != exact(x, s) for x, s in ties) >= 5
    assert sum(_e4m3_nearest_exact(Fr(float(f32(float(x) / float(s))))) != exact(x, s) for x, s in near) >= 20
    for x, s in ties + near + rand:
        assert _fp8_write_one(x, s) == (exact(x, s), exact(-x, s)), (x, s)


def test_fp8_write_codes_equal_torch_on_exact_quotients():
    """Where x / scale is exact in float, torch's float8_e4m3fn conversion of
    that quotient is a single correct rounding: the write's codes agree."""
    import torch
    rng = np.random.default_rng(32)
    n, d, bs = 64, 32, 16
    qv = (rng.integers(-2 ** 11, 2 ** 11, size=(n, d)) * 2.0 ** rng.integers(-14, -2, size=(n, 1)))
    s = (rng.integers(1, 2 ** 11, size=n) * 2.0 ** rng.integers(-16, -6, size=n))
    x = qv * s[:, None]
    assert (x.astype(np.float32) == x).all() and (s.astype(np.float32) == s).all()
    k = x.astype(np.float32).reshape(n, 1, d)
    kc = np.zeros((n, 1, bs, d), np.uint8)
    vc = np.zeros((n, 1, d, bs), np.uint8)
    for t in range(n):
        kt = k[t:t + 1]
        kct, vct = kc[t:t + 1].copy(), vc[t:t + 1].copy()
        sc = np.array([s[t]], np.float32)
        oracle.kv_cache_write_fp8(kt, kt, np.array([0], np.int32), np.array([0], np.int64), kct, vct,
                                  sc, sc, 1e4, oracle.ROPE_NONE)
        ref = torch.from_numpy(qv[t]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(kct[0, 0, 0], ref) and np.array_equal(vct[0, 0, :, 0], ref), t


def test_fp8_attention_is_attention_on_dequantised_values():
    rng = np.random.default_rng(19)
    nb, H, bs, d = 8, 2, 16, 64
    kc = rng.integers(0, 0x7E, size=(nb, H, bs, d)).astype(np.uint8)   # finite positive codes
    kc |= (rng.integers(0, 2, size=kc.shape) << 7).astype(np.uint8)    # random signs
    vc = rng.integers(0, 0x7E, size=(nb, H, d, bs)).astype(np.uint8)
    ks, vs = np.array([0.003, 0.004], np.float32), np.array([0.01, 0.02], np.float32)
    q = np.vectorize(oracle.round_bf16, otypes=[np.uint16])(rng.standard_normal((2, 4, d)))
    bt = np.array([[5, 2, -1], [0, 7, 1]], np.int32)
    cl = np.array([20, 40], np.int32)
    got = oracle.paged_attention_fp8(q, kc, vc, ks, vs, bt, cl, 0.125)
    kd, vd = oracle.fp8_dequant(kc, vc, ks, vs)
    ref = _bruteforce(oracle.to_f64(q), kd, vd, bt, cl, 0.125)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- prefill (causal)

def test_prefill_is_causal_sdpa_on_the_gathered_prompt():
    """A whole prompt (positions 0..P-1) equals torch's causal
    scaled_dot_product_attention on the contiguously gathered K/V; a chunk at
    positions c..P-1 equals the same with the prefix visible."""
    import torch
    rng = np.random.default_rng(20)
    P, Hq, Hkv, d, bs = 45, 4, 2, 32, 16
    q, kc, vc, bt, cl = _rand_case(rng, [P, 20], Hq, Hkv, d, bs, dtype="f32")
    qtok = np.vectorize(lambda x: x, otypes=[np.float32])(rng.standard_normal((P, Hq, d)))
    pos = np.arange(P, dtype=np.int32)
    seq = np.zeros(P, np.int32)
    got = oracle.paged_attention_prefill(qtok, seq, pos, kc, vc, bt, 0.3)
    K = torch.from_numpy(_gather(kc, bt, 0, P, bs)).repeat_interleave(Hq // Hkv, 0)
    V = torch.from_numpy(_gather(vc, bt, 0, P, bs)).repeat_interleave(Hq // Hkv, 0)
    Q = torch.from_numpy(qtok.astype(np.float64)).transpose(0, 1)             # [Hq, P, d]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=0.3)
    np.testing.assert_allclose(got, ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
    c0 = 30  # chunk of the last 15 tokens
    got_c = oracle.paged_attention_prefill(qtok[c0:].copy(), seq[c0:], pos[c0:], kc, vc, bt, 0.3)
    mask = torch.from_numpy(np.arange(P)[None, :] <= pos[c0:, None])
    ref_c = torch.nn.functional.scaled_dot_product_attention(Q[:, c0:], K, V, attn_mask=mask, scale=0.3)
    np.testing.assert_allclose(got_c, ref_c.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
