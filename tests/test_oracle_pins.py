"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks one oracle function against something other than itself: a value
worked out by hand, a closed form, an invariant, a special case that reduces to a
textbook result, or a brute-force loop on a tiny input.  Each is chosen so that a
plausible slip (a dropped term, a wrong sign, a transposed operand, the wrong block
axis, interleaved instead of rotate-half RoPE, modulo instead of contiguous GQA
grouping) fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
import synth

RNG = np.random.default_rng(20261202)


def fp16_bits(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


# ----------------------------------------------------------------------------- dequantisation

def test_dequant_hand_values():
    q = np.zeros((2, 64), dtype=np.int8)
    q[0, :4] = [3, -7, 127, -127]
    q[0, 32:34] = [1, -1]
    q[1, 0] = 127
    q[1, 63] = -5
    s = np.array([[0x3400, 0x4000], [0x0001, 0x3C00]], dtype=np.uint16)  # 0.25, 2.0 | 2^-24, 1.0
    w = oracle.dequant(q, s)
    assert w[0, 0] == 0.75 and w[0, 1] == -1.75 and w[0, 2] == 31.75 and w[0, 3] == -31.75
    assert w[0, 32] == 2.0 and w[0, 33] == -2.0          # block 1 of row 0 uses scale 2.0
    assert w[1, 0] == 127 * 2.0 ** -24                   # subnormal fp16 scale
    assert w[1, 63] == -5.0
    assert np.count_nonzero(w) == 8


def test_dequant_block_axis_is_input_axis():
    q = np.ones((3, 96), dtype=np.int8)
    s = fp16_bits([[1, 2, 4], [1, 1, 1], [0.5, 0.5, 0.5]])
    w = oracle.dequant(q, s)
    assert (w[0, :32] == 1).all() and (w[0, 32:64] == 2).all() and (w[0, 64:] == 4).all()
    assert (w[1] == 1).all() and (w[2] == 0.5).all()


def test_dequant_exact_in_float32():
    q, s = synth.q8(synth.key(7, 7), 64, 256)
    w = oracle.dequant(q, s)
    assert np.array_equal(w.astype(np.float32).astype(np.float64), w)


# ----------------------------------------------------------------------------- quantiser (input side)

def test_quantiser_invariants():
    w = (RNG.standard_normal((50, 128)) * 0.02).astype(np.float32)
    w[3, 32:64] = 0.0
    q, s = synth.quantize(w)
    assert np.abs(q.astype(int)).max() <= 127
    deq = oracle.dequant(q, s)
    scale = s.view(np.float16).astype(np.float64)
    err = np.abs(deq - w.astype(np.float64)).reshape(50, 4, 32)
    assert (err <= scale[:, :, None] / 2 * (1 + 1e-6)).all()
    blocks = np.abs(w.reshape(50, 4, 32))
    qa = np.abs(q.reshape(50, 4, 32).astype(int))
    am = blocks.argmax(axis=-1)
    nz = blocks.max(axis=-1) > 0
    assert (np.take_along_axis(qa, am[..., None], -1)[..., 0][nz] == 127).all()
    assert s[3, 1] == 0 and (q[3, 32:64] == 0).all()


def test_quantiser_generated_rows_are_addressable():
    k = synth.key(1, 2, 3)
    q, s = synth.q8(k, 40, 96)
    q2, s2 = synth.q8(k, 40, 96, row0=17, nrows=5, n_threads=1)
    assert np.array_equal(q[17:22], q2) and np.array_equal(s[17:22], s2)
    w = synth.normal_f32(k, 17 * 96, 5 * 96, synth.WEIGHT_SIGMA)
    q3, s3 = synth.quantize(w.reshape(5, 96))
    assert np.array_equal(q3, q2) and np.array_equal(s3, s2)


def test_generator_moments():
    w = synth.normal_f32(synth.key(99), 0, 1 << 18, 1.0)
    assert abs(w.mean()) < 0.01 and abs(w.std() - 1) < 0.01
    kurt = ((w - w.mean()) ** 4).mean() / w.var() ** 2
    assert abs(kurt - 3.0) < 0.05


# ----------------------------------------------------------------------------- rounding helpers

def test_bf16_rounding_ties_to_even():
    assert oracle.bf16(1 + 2 ** -8) == 1.0                 # halfway, even neighbour is 1.0
    assert oracle.bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6     # halfway, even neighbour is above
    assert oracle.bf16(1 + 2 ** -8 + 2 ** -20) == 1 + 2 ** -7
    assert oracle.bf16(-3.0) == -3.0


# ----------------------------------------------------------------------------- matmul

def test_matvec_bruteforce():
    w = RNG.standard_normal((5, 7))
    x = RNG.standard_normal((3, 7))
    got = oracle.matvec(w, x)
    for i in range(3):
        for r in range(5):
            ref = math.fsum(w[r, c] * x[i, c] for c in range(7))
            assert abs(got[i, r] - ref) <= 1e-12 * (1 + abs(ref))


# ----------------------------------------------------------------------------- RMSNorm

def test_rmsnorm_mean_square_closed_form():
    x = RNG.standard_normal((4, 64)) * 3
    eps = 1e-5
    h = oracle.rmsnorm(x, np.ones(64), eps)
    ms_x = (x * x).mean(axis=1)
    assert np.allclose((h * h).mean(axis=1), 1.0 / (1.0 + eps / ms_x), rtol=1e-12)


def test_rmsnorm_constant_vector_and_gain():
    h = oracle.rmsnorm(np.full((1, 8), 2.0), np.ones(8), 0.0)
    assert np.allclose(h, 1.0, rtol=1e-15)
    g = np.zeros(8)
    g[5] = 3.0
    h = oracle.rmsnorm(np.full((1, 8), -2.0), g, 0.0)
    assert np.allclose(h[0], [0, 0, 0, 0, 0, -3.0, 0, 0], rtol=1e-15)
    h = oracle.rmsnorm(np.full((1, 4), 1.0), np.ones(4), 1.0)      # 1/sqrt(1 + 1)
    assert np.allclose(h, 2 ** -0.5, rtol=1e-15)


# ----------------------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    v = RNG.standard_normal((3, 2, 16))
    assert np.array_equal(oracle.rope_rotate(v, np.zeros(3), 10000.0), v)


def test_rope_rotate_half_closed_form():
    p = 3.0
    e0 = np.array([[[1.0, 0, 0, 0]]])
    e1 = np.array([[[0, 1.0, 0, 0]]])
    r0 = oracle.rope_rotate(e0, np.array([p]), 10000.0)[0, 0]
    r1 = oracle.rope_rotate(e1, np.array([p]), 10000.0)[0, 0]
    # pair (0, 2) turns at angle p; pair (1, 3) at p * 10000^(-2/4) = p / 100
    assert np.allclose(r0, [math.cos(p), 0, math.sin(p), 0], atol=1e-15)
    assert np.allclose(r1, [0, math.cos(p / 100), 0, math.sin(p / 100)], atol=1e-15)


def test_rope_preserves_pair_norms_and_is_relative():
    d = 32
    q = RNG.standard_normal((1, 1, d))
    k = RNG.standard_normal((1, 1, d))
    rq = oracle.rope_rotate(q, np.array([17]), 10000.0)
    pn = lambda v: v[..., : d // 2] ** 2 + v[..., d // 2:] ** 2
    assert np.allclose(pn(rq), pn(q), rtol=1e-12)
    dots = []
    for m, n in [(5, 2), (13, 10), (103, 100)]:
        a = oracle.rope_rotate(q, np.array([m]), 10000.0)
        b = oracle.rope_rotate(k, np.array([n]), 10000.0)
        dots.append(float((a * b).sum()))
    assert np.allclose(dots, dots[0], rtol=1e-9)


# ----------------------------------------------------------------------------- attention

def naive_attention(q, keys, vals, scale):
    scores = [scale * sum(q[d] * kk[d] for d in range(len(q))) for kk in keys]
    m = max(scores)
    e = [math.exp(s - m) for s in scores]
    z = sum(e)
    return [sum(e[i] * vals[i][d] for i in range(len(keys))) / z for d in range(len(vals[0]))]


def test_attention_partial_bruteforce():
    q = RNG.standard_normal((3, 4))
    k = RNG.standard_normal((5, 4))
    v = RNG.standard_normal((5, 4))
    q_pos, k_pos = np.array([1, 3, 4]), np.arange(5)
    out, lse = oracle.attention_partial(q, k, v, q_pos, k_pos, 0.5)
    for i in range(3):
        p = q_pos[i]
        ref = naive_attention(q[i], k[: p + 1], v[: p + 1], 0.5)
        assert np.allclose(out[i], ref, rtol=1e-12, atol=1e-14)
        sc = [0.5 * float(q[i] @ k[j]) for j in range(p + 1)]
        assert abs(lse[i] - math.log(sum(math.exp(s) for s in sc))) < 1e-12


def test_attention_partial_masked_row():
    out, lse = oracle.attention_partial(np.ones((1, 2)), np.ones((2, 2)), np.ones((2, 2)),
                                        np.array([0]), np.array([1, 2]), 1.0)
    assert np.isneginf(lse[0]) and (out == 0).all()


def make_cache(seqs, hkv, length, d, rng):
    k = rng.standard_normal((seqs, hkv, length, d)).astype(np.float16)
    v = rng.standard_normal((seqs, hkv, length, d)).astype(np.float16)
    return k, v


def test_attention_single_token_returns_v():
    k, v = make_cache(1, 2, 4, 8, RNG)
    q = RNG.standard_normal((1, 4, 8))
    out = oracle.attention(q, k, v, np.array([0]), np.array([0]), 2)
    assert np.allclose(out[0, 0], v[0, 0, 0]) and np.allclose(out[0, 1], v[0, 0, 0])
    assert np.allclose(out[0, 2], v[0, 1, 0]) and np.allclose(out[0, 3], v[0, 1, 0])


def test_attention_gqa_groups_are_contiguous():
    hq, hkv, d, L = 8, 2, 4, 6
    k = np.zeros((1, hkv, L, d), np.float16)
    v = np.zeros((1, hkv, L, d), np.float16)
    v[0, 0], v[0, 1] = 1.0, 2.0
    out = oracle.attention(RNG.standard_normal((1, hq, d)), k, v, np.array([0]), np.array([L - 1]), hkv)
    assert np.allclose(out[0, :4], 1.0) and np.allclose(out[0, 4:], 2.0)


def test_attention_causal_and_per_sequence():
    k, v = make_cache(2, 1, 8, 4, RNG)
    q = RNG.standard_normal((2, 2, 4))
    out = oracle.attention(q, k, v, np.array([0, 1]), np.array([3, 5]), 1)
    k2, v2 = k.copy(), v.copy()
    k2[0, :, 4:] = 9.0
    v2[0, :, 4:] = 9.0        # future rows of sequence 0
    k2[1, :, 6:] = 9.0
    out2 = oracle.attention(q, k2, v2, np.array([0, 1]), np.array([3, 5]), 1)
    assert np.array_equal(out, out2)
    ref = naive_attention(q[1, 1], k[1, 0, :6].astype(float), v[1, 0, :6].astype(float), 0.5)
    assert np.allclose(out[1, 1], ref, rtol=1e-12)


def test_attention_equal_keys_average_values():
    k = np.ones((1, 1, 5, 4), np.float16)
    v = RNG.standard_normal((1, 1, 5, 4)).astype(np.float16)
    out = oracle.attention(RNG.standard_normal((1, 1, 4)), k, v, np.array([0]), np.array([4]), 1)
    assert np.allclose(out[0, 0], v[0, 0].astype(float).mean(axis=0), rtol=1e-12)


def test_merge_equals_unsplit_softmax():
    q = RNG.standard_normal((4, 8))
    k = RNG.standard_normal((20, 8))
    v = RNG.standard_normal((20, 8))
    q_pos = np.array([19, 19, 7, 12])
    k_pos = np.arange(20)
    full, full_lse = oracle.attention_partial(q, k, v, q_pos, k_pos, 8 ** -0.5)
    cuts = [0, 3, 9, 10, 20]
    parts = [oracle.attention_partial(q, k[a:b], v[a:b], q_pos, k_pos[a:b], 8 ** -0.5)
             for a, b in zip(cuts, cuts[1:])]
    merged, lse = oracle.merge_partials([p[0] for p in parts], [p[1] for p in parts])
    assert np.allclose(merged, full, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, full_lse, rtol=1e-12)
    # the chunk [10, 20) is fully masked for q_pos = 7: its partial is (-inf, 0)
    assert np.isneginf(parts[3][1][2])


# ----------------------------------------------------------------------------- SwiGLU / MoE

def test_silu_values():
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert abs(oracle.silu(np.array([1.0]))[0] - 0.7310585786300049) < 1e-15
    assert abs(oracle.silu(np.array([-1.0]))[0] + 0.2689414213699951) < 1e-15
    assert abs(oracle.silu(np.array([40.0]))[0] - 40.0) < 1e-12


def test_swiglu_bruteforce():
    h = RNG.standard_normal((2, 6))
    wg, wu, wd = RNG.standard_normal((4, 6)), RNG.standard_normal((4, 6)), RNG.standard_normal((6, 4))
    got = oracle.swiglu(h, wg, wu, wd)
    for t in range(2):
        g = [sum(wg[i, c] * h[t, c] for c in range(6)) for i in range(4)]
        u = [sum(wu[i, c] * h[t, c] for c in range(6)) for i in range(4)]
        a = [float(np.float32(g[i] / (1 + math.exp(-g[i])) * u[i])) for i in range(4)]
        ref = [sum(wd[r, i] * a[i] for i in range(4)) for r in range(6)]
        assert np.allclose(got[t], ref, rtol=1e-12)


def test_moe_route_matches_full_sort_and_ties():
    z = RNG.standard_normal(16)
    idx, w = oracle.moe_route(z, 4)
    brute = sorted(range(16), key=lambda e: (-z[e], e))[:4]
    assert list(idx) == brute
    assert abs(w.sum() - 1) < 1e-15
    ex = [math.exp(z[e]) for e in brute]
    assert np.allclose(w, [e / sum(ex) for e in ex], rtol=1e-12)
    idx, w = oracle.moe_route(np.array([0.0, 1.0, 1.0, 0.5, 1.0]), 2)
    assert list(idx) == [1, 2] and np.allclose(w, 0.5)


def test_moe_top1_single_expert_is_dense_swiglu():
    h = RNG.standard_normal((3, 8))
    wg, wu, wd = RNG.standard_normal((5, 8)), RNG.standard_normal((5, 8)), RNG.standard_normal((8, 5))
    out, ids, ws = oracle.moe_ffn(h, RNG.standard_normal((1, 8)), [wg], [wu], [wd], 1)
    assert (ids == 0).all() and (ws == 1).all()
    assert np.allclose(out, oracle.swiglu(h, wg, wu, wd), rtol=1e-12)


def test_moe_all_experts_equal_logits_is_average():
    E = 4
    h = RNG.standard_normal((2, 8))
    ex = [(RNG.standard_normal((5, 8)), RNG.standard_normal((5, 8)), RNG.standard_normal((8, 5))) for _ in range(E)]
    out, ids, ws = oracle.moe_ffn(h, np.zeros((E, 8)), [e[0] for e in ex], [e[1] for e in ex],
                                  [e[2] for e in ex], E)
    assert list(ids[0]) == [0, 1, 2, 3]
    avg = sum(oracle.swiglu(h, *e) for e in ex) / E
    assert np.allclose(out, avg, rtol=1e-12)


# ----------------------------------------------------------------------------- greedy readout

def test_greedy_is_the_lowest_index_of_the_maximum():
    """Brute force over rows full of ties (small integers): the greedy token is the first
    index holding the row's maximum, also when the tie sits at the ends of the row, and a
    single maximum wins wherever it is."""
    rows = RNG.integers(-3, 4, (400, 17)).astype(np.float32)
    rows[0] = 5.0            # all equal: index 0
    rows[1, [3, 16]] = 9.0   # a tie with the last index
    rows[2, [0, 16]] = 9.0   # a tie between the two ends
    rows[3, 11] = 9.0        # a single maximum
    want = []
    for r in rows:
        m = max(r)
        want.append(next(i for i, v in enumerate(r) if v == m))
    got = oracle.greedy(rows)
    assert got.tolist() == want
    assert got[0] == 0 and got[1] == 3 and got[2] == 0 and got[3] == 11
