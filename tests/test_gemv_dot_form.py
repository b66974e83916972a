"""The float form of the decode GEMV's dot product, checked on the host in exact arithmetic
(a restatement of the scheme with Python fractions, not the CUDA code).

A weight is stored biased, b = q + 128 in [1, 255]; the byte alone in a float32 word is the
denormal b * 2^-149.  Inputs enter scaled by 2^64, so one fused multiply-add per weight
accumulates b_j * x_j * 2^-85 over a 16-weight chunk; the chunk sum is scaled by 2^85 and the
bias removed with -128 * X (X = sum of the chunk's inputs), then the block scale s applies:
    s * (2^85 * acc - 128 X) = s * sum_j q_j x_j   up to float32 rounding.
Checked here: the constants give that identity; the error stays within the float32 bound of a
17-step fused chain measured against the biased magnitudes (sum_j b_j |x_j| + 128 |X|, the
price of removing the bias after the sum); inputs down to 2^-41 keep every product normal and
smaller ones lose only an absolute 2^-65 s per product; |x| >= 2^64 overflows the scaled input
(the entry points normalise or bound every input far below that).
"""
from fractions import Fraction

import numpy as np

F32_MIN_EXP = -126
F32_MANT = 23


def round_f32(v: Fraction) -> Fraction:
    """v rounded to the nearest float32 (ties to even, subnormals kept); inf as None."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    quantum = Fraction(2) ** (max(e, F32_MIN_EXP) - F32_MANT)
    n = a / quantum
    m = n.numerator // n.denominator
    rem = n - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    r = m * quantum
    if r >= Fraction(2) ** 128:
        return None
    return sign * r


def fma(a, b, c):
    return round_f32(a * b + c)


def f32(x) -> Fraction:
    return Fraction(float(np.float32(x)))


def gemv_chunk(b, x, s):
    """The scheme for one chunk: 16 biased bytes b, 16 float32 inputs x, block scale s."""
    den = [Fraction(int(bj), 2 ** 149) for bj in b]  # the byte alone in a float32 word
    xs = [round_f32(f32(xj) * 2 ** 64) for xj in x]
    if any(v is None for v in xs):
        return None
    acc = round_f32(den[0] * xs[0])
    for j in range(1, 16):
        acc = fma(den[j], xs[j], acc)
    big_x = Fraction(0)
    for xj in x:  # the chunk sum of the inputs, in float32
        big_x = round_f32(big_x + f32(xj))
    t = fma(acc, Fraction(2) ** 85, -128 * big_x)
    return round_f32(t * f32(s))


def chunks(rng, count):
    for t in range(count):
        q = rng.integers(-127, 128, 16)
        if t % 4 == 0:
            q[:] = rng.choice([-127, 127], 16)  # extreme weights: the bias cancellation at its worst
        x = (rng.standard_normal(16) * 10.0 ** rng.uniform(-8, 8)).astype(np.float32)
        if t % 5 == 0:
            x = np.abs(x)  # one-signed inputs: 128 X at its largest
        s = np.float32(np.float16(rng.uniform(1e-4, 1e-2)))
        yield q, x, s


def test_constants_give_the_dot_product():
    """With small integer inputs every step is exact: the scheme returns sum_j q_j x_j s exactly."""
    rng = np.random.default_rng(3)
    for _ in range(200):
        q = rng.integers(-127, 128, 16)
        x = rng.integers(-64, 65, 16).astype(np.float32)
        s = np.float32(0.5)
        got = gemv_chunk(q + 128, x, s)
        assert got == Fraction(int(np.dot(q, x.astype(np.int64)))) * Fraction(1, 2)


def test_error_within_the_float32_bound_of_the_biased_sum():
    rng = np.random.default_rng(4)
    u = Fraction(1, 2 ** 24)
    for q, x, s in chunks(rng, 400):
        got = gemv_chunk(q + 128, x, s)
        exact = sum(int(qj) * f32(xj) for qj, xj in zip(q, x)) * f32(s)
        mag = (sum((int(qj) + 128) * abs(f32(xj)) for qj, xj in zip(q, x))
               + 128 * sum(abs(f32(xj)) for xj in x)) * f32(s)
        assert abs(got - exact) <= 18 * u * mag, (q, x, s)


def test_small_inputs_lose_only_an_absolute_amount():
    """Inputs of 2^-41 and above keep every product b x 2^-85 normal; below, a product is a
    denormal and carries an absolute error of at most half its spacing, 2^-150, i.e. 2^-65 s
    after the 2^85 rescale."""
    b = np.full(16, 1)  # the smallest biased byte: the first to fall below the normal range
    x = np.full(16, 2.0 ** -41, dtype=np.float32)
    den = Fraction(1, 2 ** 149)
    assert den * round_f32(f32(x[0]) * 2 ** 64) == Fraction(2) ** -126  # still normal
    rng = np.random.default_rng(5)
    for _ in range(200):
        q = rng.integers(-127, 128, 16)
        x = (rng.standard_normal(16) * 2.0 ** rng.uniform(-70, -40)).astype(np.float32)
        s = np.float32(np.float16(rng.uniform(1e-4, 1e-2)))
        got = gemv_chunk(q + 128, x, s)
        exact = sum(int(qj) * f32(xj) for qj, xj in zip(q, x)) * f32(s)
        mag = (sum((int(qj) + 128) * abs(f32(xj)) for qj, xj in zip(q, x))
               + 128 * sum(abs(f32(xj)) for xj in x)) * f32(s)
        assert abs(got - exact) <= 18 * Fraction(1, 2 ** 24) * mag + 17 * Fraction(2) ** -65 * f32(s)


def test_inputs_of_two_to_the_64_overflow():
    q = np.zeros(16, dtype=np.int64)
    x = np.zeros(16, dtype=np.float32)
    x[3] = np.float32(2.0 ** 64)
    assert gemv_chunk(q + 128, x, np.float32(1.0)) is None
    x[3] = np.float32(2.0 ** 63)
    assert gemv_chunk(q + 128, x, np.float32(1.0)) is not None
