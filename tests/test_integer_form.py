"""The integer form in which the persistent decode stages its projection input, checked on the
host against exact arithmetic (a numpy restatement of the scheme, not the CUDA code).

A chunk of 16 inputs h_j becomes an exponent e with every |h_j| < 2^e and integers
N_j = rint(h_j / u), u = (128/127) 2^(e - 23); N_j + 0x808080 written in base 256 gives three
digits, each a signed byte plus 128.  For 16 weights q_j in [-127, 127] stored as b_j = q_j + 128,
  D_i = sum_j b_j l_ij - 128 sum_j l_ij   (exact integers), and
  sum_j q_j h_j = u (2^16 D0 + 2^8 D1 + D2) + sum_j q_j (h_j - u N_j).
N_j is rint of the float32 product h_j * (1/u), so two roundings meet: the product's (relative
2^-24 of h_j, what float32 keeps anyway) and rint's (half a unit), and where the first lands on
a half-integer the second can add to it (up to 0.75 u).  Checked here: the three bytes rebuild
N_j exactly and stay signed bytes; each input is off by at most u/2 + 2^-24 |h_j|, below
(128/127 + 1/2) 2^-23 of the chunk's largest input; the dot's only error is those roundings;
and D_i fits the 2^22 window of the float trick the kernel uses to read it back.
"""
import numpy as np


def encode(h):
    """(N, limbs [3][16] as signed ints, unit u) of one chunk, float32 arithmetic as on the GPU."""
    h = np.asarray(h, np.float32)
    m = np.float32(np.max(np.abs(h)))
    e = max(int((m.view(np.uint32) >> 23) & 0xFF) - 126, -100)
    sc = np.float32(np.uint32((127 + 23 - e) << 23).view(np.float32) * np.float32(0.9921875))
    n = np.rint((h * sc).astype(np.float64)).astype(np.int64)  # rint of the float32 product
    biased = n + 0x808080
    assert np.all(biased >= 0) and np.all(biased < (1 << 24))
    digits = np.stack([(biased >> 16) & 255, (biased >> 8) & 255, biased & 255]) - 128
    u = float(np.uint32((127 + e - 23) << 23).view(np.float32)) * 128.0 / 127.0
    return n, digits, u, e


def chunks(rng, count):
    for t in range(count):
        scale = 10.0 ** rng.uniform(-20, 20)
        h = (rng.standard_normal(16) * scale).astype(np.float32)
        if t % 5 == 0:
            h[rng.integers(0, 16, 6)] = 0.0
        if t % 7 == 0:  # one dominant input
            h[rng.integers(0, 16)] = np.float32(np.max(np.abs(h)) * 100.0)
        if t % 11 == 0:
            h[:] = 0.0
        yield h


def test_limbs_rebuild_the_integers_and_stay_signed_bytes():
    rng = np.random.default_rng(7)
    for h in chunks(rng, 4000):
        n, l, u, e = encode(h)
        assert np.array_equal((l[0] << 16) + (l[1] << 8) + l[2], n)
        assert l.min() >= -128 and l.max() <= 127
        assert np.all(np.abs(n) < (127 * (1 << 23)) // 128 + 1)


def test_dot_error_is_the_rounding_of_the_inputs_only():
    rng = np.random.default_rng(8)
    for h in chunks(rng, 4000):
        n, l, u, e = encode(h)
        q = rng.integers(-127, 128, 16)
        b = q + 128
        d = [int(np.dot(b, l[i]) - 128 * l[i].sum()) for i in range(3)]
        assert all(abs(x) < (1 << 22) for x in d)  # the float trick's window (1.5 * 2^23 +- 2^22)
        h64 = h.astype(np.float64)
        per_input = u / 2.0 + 2.0 ** -24 * np.abs(h64)
        assert np.all(np.abs(h64 - u * n) <= per_input * (1.0 + 1e-12))
        got = u * ((d[0] << 16) + (d[1] << 8) + d[2])
        exact = float(np.dot(q.astype(np.float64), h64))
        assert abs(got - exact) <= float(np.dot(np.abs(q), per_input)) * (1.0 + 1e-12) + 1e-300
        # relative to the chunk's largest input (at least 2^(e - 1)): u/2 is at most
        # (128/127) 2^-23 of it and 2^-24 |h_j| at most 2^-24 of it
        mh = float(np.max(np.abs(h64)))
        if mh > 0:
            assert np.abs(h64 - u * n).max() <= (128.0 / 127.0 + 0.5) * 2.0 ** -23 * mh * (1.0 + 1e-12)


def test_zero_chunk_encodes_to_zero():
    n, l, u, e = encode(np.zeros(16, np.float32))
    assert not n.any() and not l.any() and e == -100
