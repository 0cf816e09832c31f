"""Pins of the oracle to facts that do not come from the oracle itself:
brute-force sums, closed forms derived from the schedule, exact rational
rounding, library conversions, invariants the pages state."""
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

rng = np.random.default_rng(12345)


# ------------------------------------------------------------- partition

def test_chunk_bounds_first_chunks_longer():
    """"Ring All-Reduce, in depth", "An implementation": the first N mod p
    chunks get one extra element; 4099 over 4 gives 1025/1025/1025/1024."""
    b = oracle.chunk_bounds(4099, 4)
    assert [e - s for s, e in b] == [1025, 1025, 1025, 1024]
    for n in range(0, 70):
        for p in range(1, 18):
            b = oracle.chunk_bounds(n, p)
            sizes = [e - s for s, e in b]
            # same sizes as numpy.array_split, a library partition of the
            # same rule
            assert sizes == [len(a) for a in np.array_split(np.arange(n), p)]
            assert b[0][0] == 0 and b[-1][1] == n
            assert all(b[i][1] == b[i + 1][0] for i in range(p - 1))


# ------------------------------------------------------------- int32 brute force

def _rand_i32(p, n):
    return [rng.integers(-(2 ** 31), 2 ** 31, size=n, dtype=np.int64).astype(np.int32) for _ in range(p)]


def _naive_sum_i32(bufs):
    s = np.zeros(bufs[0].shape, dtype=np.int64)
    for b in bufs:
        s += b.astype(np.int64)
    return (s & 0xFFFFFFFF).astype(np.uint32).view(np.int32)


def test_int32_sum_brute_force_small():
    """"Ring All-Reduce, in depth", "What to do next" item 1: the simulator
    against a plain sum, for many p and N including N not divisible by p.
    int32 addition is exact modulo 2^32 in any order, so the ring must equal
    the naive sum bit for bit; a dropped or doubled hop cannot."""
    for p in range(1, 18):
        for n in list(range(0, 40)) + [63, 64, 65]:
            bufs = _rand_i32(p, n)
            expect = _naive_sum_i32(bufs)
            oracle.simulate(bufs, "int32", "sum")
            for b in bufs:
                np.testing.assert_array_equal(b, expect)


def test_int32_sum_brute_force_random_sizes():
    r = random.Random(7)
    for _ in range(40):
        p, n = r.randint(1, 33), r.randint(0, 2000)
        bufs = _rand_i32(p, n)
        expect = _naive_sum_i32(bufs)
        oracle.simulate(bufs, "int32", "sum")
        for b in bufs:
            np.testing.assert_array_equal(b, expect)


def test_bidir_int32_brute_force():
    """The bidirectional variant computes the same all-reduce."""
    for p in range(1, 12):
        for n in [0, 1, 2, 3, 7, 8, 31, 100, 257]:
            bufs = _rand_i32(p, n)
            expect = _naive_sum_i32(bufs)
            oracle.simulate_bidir(bufs, "int32", "sum")
            for b in bufs:
                np.testing.assert_array_equal(b, expect)


# ------------------------------------------------------------- ownership / steps

@pytest.mark.parametrize("direction", ["forward", "mirrored"])
def test_ownership_after_reduce_scatter(direction):
    """"Ring All-Reduce, in depth", "The schedule": after the p - 1
    reduce-scatter steps rank r holds the complete sum of chunk (r + 1) mod p
    (mirrored ring: chunk (r - 1) mod p)."""
    for p in range(2, 11):
        for n in [p, 3 * p + 1, 50]:
            bufs = _rand_i32(p, n)
            full = _naive_sum_i32(bufs)
            oracle.simulate(bufs, "int32", "sum", direction=direction, first_step=0, n_steps=p - 1)
            bounds = oracle.chunk_bounds(n, p)
            for r in range(p):
                c = (r + 1) % p if direction == "forward" else (r - 1) % p
                s, e = bounds[c]
                np.testing.assert_array_equal(bufs[r][s:e], full[s:e])


def test_step_count_is_two_p_minus_two():
    """"Ring All-Reduce, in depth", "The schedule": two phases of p - 1 steps;
    running reduce-scatter then all-gather separately equals the whole."""
    for p in [2, 3, 5, 8]:
        n = 23
        a = _rand_i32(p, n)
        b = [x.copy() for x in a]
        oracle.simulate(a, "int32", "sum")
        oracle.simulate(b, "int32", "sum", first_step=0, n_steps=p - 1)
        oracle.simulate(b, "int32", "sum", first_step=p - 1, n_steps=p - 1)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)
        with pytest.raises(ValueError):
            oracle.simulate([x.copy() for x in a], "int32", "sum", first_step=0, n_steps=2 * p - 1)


# ------------------------------------------------------------- send counts

def test_send_counts_law():
    """Each rank sends every chunk but one in each phase ("The schedule"): in
    the reduce-scatter all but chunk (r + 1), in the all-gather all but chunk
    (r + 2), so sends_r = 2N - |C_(r+1)| - |C_(r+2)|, the total is
    2(p - 1) N, and each rank sends exactly 2(p - 1)/p x N when p | N."""
    for p in range(1, 14):
        for n in [0, 1, 5, p, 4 * p, 4 * p + 3, 101]:
            bufs = _rand_i32(p, n)
            sends = oracle.simulate(bufs, "int32", "sum")
            if p == 1:
                assert list(sends) == [0]
                continue
            sizes = [e - s for s, e in oracle.chunk_bounds(n, p)]
            for r in range(p):
                assert sends[r] == 2 * n - sizes[(r + 1) % p] - sizes[(r + 2) % p]
            assert sends.sum() == 2 * (p - 1) * n
            if n % p == 0:
                assert all(s * p == 2 * (p - 1) * n for s in sends)


def test_send_counts_config_p4_n4099():
    sends = oracle.simulate(_rand_i32(4, 4099), "int32", "sum")
    assert list(sends) == [6148, 6149, 6149, 6148]


def test_bidir_send_counts():
    """Bidirectional: forward ring on the first half plus the mirrored ring
    (sends all but chunks r - 1 and r - 2) on the second half."""
    for p in range(2, 10):
        for n in [1, 2, 9, 64, 99]:
            bufs = _rand_i32(p, n)
            sends = oracle.simulate_bidir(bufs, "int32", "sum")
            h = oracle.chunk_bounds(n, 2)[0][1]
            f = [e - s for s, e in oracle.chunk_bounds(h, p)]
            m = [e - s for s, e in oracle.chunk_bounds(n - h, p)]
            for r in range(p):
                expect = (2 * h - f[(r + 1) % p] - f[(r + 2) % p]) + \
                         (2 * (n - h) - m[(r - 1) % p] - m[(r - 2) % p])
                assert sends[r] == expect


# ------------------------------------------------------------- hop order

def _order_detector(p, n, big, last, dtype, direction="forward"):
    """Per chunk c: the chunk's starting rank c holds `big`, the last rank the
    chunk visits holds `last`, every other rank 1."""
    st = np.float32
    bufs = [np.ones(n, dtype=st) for _ in range(p)]
    for c, (s, e) in enumerate(oracle.chunk_bounds(n, p)):
        last_rank = (c - 1) % p if direction == "forward" else (c + 1) % p
        bufs[c][s:e] = big
        bufs[last_rank][s:e] = last
    if dtype == "bfloat16":
        bufs = [np.array([oracle.f32_to_bf16(float(v)) for v in b], dtype=np.uint16) for b in bufs]
    return bufs


@pytest.mark.parametrize("direction", ["forward", "mirrored"])
def test_fp32_hop_order_closed_form(direction):
    """Chunk c starts at rank c and visits c+1, c+2, ... ("Tracing four GPUs":
    chunk 0 goes 0 -> 1 -> 2 -> 3).  With 2^24 at the start, ones in the
    middle and 2 at the last rank: each +1 is exactly half a unit in the last
    place at 2^24 and rounds to the even neighbour 2^24, and the final +2 is
    exact, so every element ends at 2^24 + 2.  Starting one rank early or
    late, or folding in reverse, gives 2^24 + 4 or 2^24 + p instead."""
    for p in [3, 4, 5, 8, 13]:
        for n in [p, 2 * p + 1, 37]:
            bufs = _order_detector(p, n, 2.0 ** 24, 2.0, "float32", direction)
            oracle.simulate(bufs, "float32", "sum", direction=direction)
            for b in bufs:
                assert np.all(b == np.float32(2.0 ** 24 + 2.0))


def test_bf16_hop_order_closed_form():
    """The same detector in bf16: spacing at 256 is 2, so 256 + 1 ties back to
    256 and the final + 2 gives 258."""
    for p in [3, 4, 8]:
        n = 3 * p + 2
        bufs = _order_detector(p, n, 256.0, 2.0, "bfloat16")
        oracle.simulate(bufs, "bfloat16", "sum")
        for b in bufs:
            assert np.all(b == oracle.f32_to_bf16(258.0))


def test_max_tie_rule_pm_zero():
    """max keeps the running value unless the receiver's element is strictly
    greater: +0 starting at rank c meets -0 at rank c + 1 and stays +0; the
    opposite start keeps -0.  (IEEE: +0 == -0, so neither is greater.)"""
    p, n = 4, 8
    bufs = [np.full(n, -1.0, dtype=np.float32) for _ in range(p)]
    for c, (s, e) in enumerate(oracle.chunk_bounds(n, p)):
        bufs[c][s:e] = 0.0
        bufs[(c + 1) % p][s:e] = -0.0
    oracle.simulate(bufs, "float32", "max")
    for b in bufs:
        assert np.all(b.view(np.uint32) == 0x00000000)
    bufs = [np.full(n, -1.0, dtype=np.float32) for _ in range(p)]
    for c, (s, e) in enumerate(oracle.chunk_bounds(n, p)):
        bufs[c][s:e] = -0.0
        bufs[(c + 1) % p][s:e] = 0.0
    oracle.simulate(bufs, "float32", "max")
    for b in bufs:
        assert np.all(b.view(np.uint32) == 0x80000000)


# ------------------------------------------------------------- max / avg

def test_max_equals_library_max():
    """max is order-independent on finite inputs without +-0 ties: the ring
    must equal numpy's maximum over the ranks."""
    for p in [1, 2, 3, 7, 16]:
        n = 301
        bufs = [rng.uniform(-1e3, 1e3, size=n).astype(np.float32) for _ in range(p)]
        expect = np.max(np.stack(bufs), axis=0)
        oracle.simulate(bufs, "float32", "max")
        for b in bufs:
            np.testing.assert_array_equal(b, expect)
        ibufs = _rand_i32(p, n)
        iexp = np.max(np.stack(ibufs), axis=0)
        oracle.simulate(ibufs, "int32", "max")
        for b in ibufs:
            np.testing.assert_array_equal(b, iexp)


def test_avg_power_of_two_is_scaled_sum():
    """For p = 2^k, 1/p is exact in binary32, so avg is exactly the ring sum
    times 2^-k (no underflow at these magnitudes), on every rank."""
    for p in [2, 4, 8, 16]:
        n = 257
        base = [rng.normal(0, 1, size=n).astype(np.float32) for _ in range(p)]
        s = [b.copy() for b in base]
        a = [b.copy() for b in base]
        oracle.simulate(s, "float32", "sum")
        oracle.simulate(a, "float32", "avg")
        for x in a:
            np.testing.assert_array_equal(x, s[0] * np.float32(1.0 / p))


def test_avg_close_to_mean_any_p():
    """avg within a few ulps of the exact mean (ring sum error bound plus one
    rounding of the scale and one of the product)."""
    for p in [3, 5, 6, 7]:
        n = 200
        bufs = [rng.normal(0, 1, size=n).astype(np.float32) for _ in range(p)]
        exact = np.sum(np.stack(bufs).astype(np.float64), axis=0) / p
        mag = np.sum(np.abs(np.stack(bufs).astype(np.float64)), axis=0) / p
        oracle.simulate(bufs, "float32", "avg")
        err = np.abs(bufs[0].astype(np.float64) - exact)
        assert np.all(err <= (p + 2) * 2.0 ** -24 * mag + 1e-30)


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_avg_any_p_exact_rational(dtype):
    """avg = (ring sum) x (1/p rounded to binary32), the product rounded once
    to binary32 (then to bf16).  With small integer inputs the ring sum S is
    exact, so the expected value is computed here from exact rationals:
    round32(S * round32(1/p))."""
    for p in [3, 5, 6, 7, 11, 12]:
        n = 40
        ints = [rng.integers(-20, 21, size=n).astype(np.float32) for _ in range(p)]
        S = np.sum(np.stack(ints).astype(np.int64), axis=0)
        inv = _exact_rne(Fraction(1, p), 23, -126, 127)
        if dtype == "float32":
            bufs = [v.copy() for v in ints]
        else:
            bufs = [np.array([oracle.f32_to_bf16(float(x)) for x in v], dtype=np.uint16) for v in ints]
        oracle.simulate(bufs, dtype, "avg")
        for i in range(n):
            e = _exact_rne(Fraction(int(S[i])) * inv, 23, -126, 127)
            if dtype == "bfloat16":
                e = _exact_rne(e, 7, -126, 127)
                got = Fraction(oracle.bf16_to_f32(int(bufs[p - 1][i])))
            else:
                got = Fraction(float(bufs[p - 1][i]))
            assert got == e, (p, i)


def test_prediv_avoids_fp16_overflow():
    """"Ring All-Reduce, in depth", "Failure modes": summing fp16 from many
    ranks can overflow; pre-dividing avoids it.  16 ranks of 4096: the sum
    65536 exceeds the largest fp16 value (65504) and rounds to inf, so the
    post-divided average is inf; pre-divided, each contribution is 256
    (exact) and the sum is exactly 4096, the true mean."""
    p, n = 16, 10
    h4096 = oracle.f32_to_f16(4096.0)
    post = [np.full(n, h4096, dtype=np.uint16) for _ in range(p)]
    oracle.simulate(post, "float16", "avg")
    assert all(oracle.f16_to_f32(int(v)) == float("inf") for v in post[0])
    pre = [np.full(n, h4096, dtype=np.uint16) for _ in range(p)]
    oracle.simulate(pre, "float16", "avg_prediv")
    for b in pre:
        assert all(oracle.f16_to_f32(int(v)) == 4096.0 for v in b)


def test_prediv_exact_mean_when_division_is_exact():
    """For p a power of two and inputs that are multiples of p, every
    pre-divided contribution and every partial sum is exact: the result is
    the exact mean."""
    for p in [2, 4, 8, 16]:
        n = 50
        ints = [rng.integers(-40, 41, size=n) for _ in range(p)]
        bufs = [(v * p).astype(np.float32) for v in ints]
        oracle.simulate(bufs, "float32", "avg_prediv")
        mean = np.sum(np.stack(ints), axis=0).astype(np.float32)
        for b in bufs:
            np.testing.assert_array_equal(b, mean)


def test_avg_rejected_for_int32():
    with pytest.raises(ValueError):
        oracle.simulate(_rand_i32(4, 8), "int32", "avg")
    with pytest.raises(ValueError):
        oracle.simulate(_rand_i32(4, 8), "int32", "avg_prediv")


# ------------------------------------------------------------- float sums

@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_integer_valued_floats_equal_naive_sum(dtype):
    """Small integers sum exactly in any order, so the ring equals the plain
    sum; exercises the float path without rounding."""
    for p in [2, 3, 4, 8, 16]:
        n = 77
        vals = [rng.integers(-8, 9, size=n).astype(np.float32) for _ in range(p)]
        expect = np.sum(np.stack(vals), axis=0)
        if dtype == "bfloat16":
            bufs = [np.array([oracle.f32_to_bf16(float(v)) for v in b], dtype=np.uint16) for b in vals]
        else:
            bufs = [v.copy() for v in vals]
        oracle.simulate(bufs, dtype, "sum")
        for b in bufs:
            got = b if dtype == "float32" else np.array([oracle.bf16_to_f32(int(h)) for h in b], dtype=np.float32)
            np.testing.assert_array_equal(got, expect)


def test_fp32_ring_sum_within_bound():
    """Any order of p - 1 binary32 additions is within (p - 1) u sum|x| of the
    exact sum (u = 2^-24)."""
    for p in [2, 4, 8, 33]:
        n = 500
        bufs = [rng.normal(0, 1, size=n).astype(np.float32) for _ in range(p)]
        ref, mag = oracle.f64_sum(bufs, "float32")
        oracle.simulate(bufs, "float32", "sum")
        assert np.all(np.abs(bufs[0] - ref) <= (p - 1) * 2.0 ** -24 * mag * 1.0001 + 1e-38)


# ------------------------------------------------------------- rounding pins

def _exact_rne(x: Fraction, man_bits: int, emin: int, emax: int):
    """Round an exact rational to a binary format with `man_bits` stored
    fraction bits, minimum normal exponent emin and maximum exponent emax;
    returns a Fraction or +-inf (float)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = max(e, emin) - man_bits
    scaled = a / Fraction(2) ** q
    lo = scaled.numerator // scaled.denominator
    rem = scaled - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    r = Fraction(lo) * Fraction(2) ** q
    if r >= Fraction(2) ** (emax + 1):
        return sign * float("inf")
    return sign * r


def _random_f32_patterns(k, seed):
    g = np.random.default_rng(seed)
    pats = g.integers(0, 2 ** 32, size=k, dtype=np.uint64).astype(np.uint32)
    # include ties and near-overflow / subnormal patterns
    extra = [0x3F808000, 0x3F818000, 0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0x00000001,
             0x00008000, 0x00018000, 0x80008000, 0x477FF000, 0x477FEFFF, 0x33000000,
             0x33000001, 0x387FC000, 0x38800000, 0x00000000, 0x80000000]
    return np.concatenate([pats, np.array(extra, dtype=np.uint32)])


def test_bf16_conversion_against_exact_rounding():
    pats = _random_f32_patterns(3000, 1)
    for u in pats:
        f = np.array([u], dtype=np.uint32).view(np.float32)[0]
        if not np.isfinite(f):
            continue
        exact = _exact_rne(Fraction(float(f)), 7, -126, 127)
        got = oracle.bf16_to_f32(oracle.f32_to_bf16(float(f)))
        if isinstance(exact, float):
            assert got == exact
        else:
            assert Fraction(got) == exact, hex(int(u))


def test_bf16_conversion_against_torch():
    f = _random_f32_patterns(20000, 2).view(np.float32)
    f = f[np.isfinite(f)]
    t = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(float(v)) for v in f], dtype=np.uint16)
    np.testing.assert_array_equal(got, t)


def test_f16_conversion_against_exact_and_numpy():
    f = _random_f32_patterns(20000, 3).view(np.float32)
    f = f[np.isfinite(f)]
    got = np.array([oracle.f32_to_f16(float(v)) for v in f], dtype=np.uint16)
    np.testing.assert_array_equal(got, f.astype(np.float16).view(np.uint16))
    for v in f[:500]:
        exact = _exact_rne(Fraction(float(v)), 10, -14, 15)
        back = oracle.f16_to_f32(oracle.f32_to_f16(float(v)))
        if isinstance(exact, float):
            assert back == exact
        else:
            assert Fraction(back) == exact
    # widening every binary16 pattern agrees with numpy
    allp = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = allp.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(h)) for h in allp], dtype=np.float32)
    ok = np.isfinite(ref)
    np.testing.assert_array_equal(got[ok].view(np.uint32), ref[ok].view(np.uint32))


def test_bf16_add_is_correctly_rounded():
    """One bf16 hop equals the exact sum rounded once to bf16 (including wide
    exponent gaps, ties and subnormals)."""
    g = np.random.default_rng(4)
    for _ in range(4000):
        ea, eb = g.integers(-133, 127, size=2)
        if g.random() < 0.5:
            eb = ea - g.integers(0, 20)
        ma, mb = g.integers(0, 128, size=2)
        sa, sb = g.choice([-1, 1], size=2)
        def mk(s, e, m):
            v = s * (1 + m / 128.0) * 2.0 ** int(e)
            return oracle.f32_to_bf16(float(np.float32(v)))
        a, b = mk(sa, ea, ma), mk(sb, max(eb, -133), mb)
        fa, fb = oracle.bf16_to_f32(a), oracle.bf16_to_f32(b)
        exact = _exact_rne(Fraction(fa) + Fraction(fb), 7, -126, 127)
        got = oracle.bf16_to_f32(int(oracle.combine("bfloat16", "sum", a, b)))
        if isinstance(exact, float):
            assert got == exact
        else:
            assert Fraction(got) == exact


def test_f16_add_is_correctly_rounded():
    g = np.random.default_rng(5)
    for _ in range(3000):
        a, b = g.integers(0, 1 << 16, size=2)
        fa, fb = oracle.f16_to_f32(int(a)), oracle.f16_to_f32(int(b))
        if not (np.isfinite(fa) and np.isfinite(fb)):
            continue
        exact = _exact_rne(Fraction(fa) + Fraction(fb), 10, -14, 15)
        got = oracle.f16_to_f32(int(oracle.combine("float16", "sum", np.uint16(a), np.uint16(b))))
        if isinstance(exact, float):
            assert got == exact
        else:
            assert Fraction(got) == exact


def test_fp32_add_is_ieee():
    """The fp32 hop is the platform's IEEE binary32 addition: it matches
    numpy's float32 addition bit for bit."""
    a = rng.normal(0, 1, size=2000).astype(np.float32)
    b = (rng.normal(0, 1, size=2000) * 10.0 ** rng.integers(-8, 8, size=2000)).astype(np.float32)
    for x, y in zip(a[:300], b[:300]):
        assert oracle.combine("float32", "sum", x, y) == np.float32(x + y)


# ------------------------------------------------------------- closed form

CASES = [
    ("int32", "sum"), ("int32", "max"), ("float32", "sum"), ("float32", "max"),
    ("float32", "avg"), ("bfloat16", "sum"), ("bfloat16", "max"), ("bfloat16", "avg"),
    ("float16", "sum"), ("float16", "avg"), ("float32", "avg_prediv"), ("bfloat16", "avg_prediv"),
    ("float16", "avg_prediv"),
]


def _rand_bufs(p, n, dtype, seed):
    g = np.random.default_rng(seed)
    if dtype == "int32":
        return [g.integers(-(2 ** 20), 2 ** 20, size=n).astype(np.int32) for _ in range(p)]
    vals = [g.normal(0, 1, size=n).astype(np.float32) for _ in range(p)]
    if dtype == "float32":
        return vals
    t = torch.bfloat16 if dtype == "bfloat16" else torch.float16
    return [torch.from_numpy(v).to(t).view(torch.int16).numpy().view(np.uint16).copy() for v in vals]


@pytest.mark.parametrize("dtype,op", CASES)
@pytest.mark.parametrize("mode", ["ring", "bidir"])
def test_closed_form_equals_simulator(dtype, op, mode):
    """The per-element fold read off the schedule equals the step-by-step
    simulator bit for bit, for every element."""
    for p, n in [(2, 5), (3, 10), (4, 4099), (5, 64), (8, 1000), (16, 333), (1, 9)]:
        bufs = _rand_bufs(p, n, dtype, p * 1000 + n)
        vals = np.stack(bufs)
        idx = np.arange(n, dtype=np.int64)
        folded = oracle.fold_sampled(vals, idx, n, dtype, op, mode)
        if mode == "ring":
            oracle.simulate(bufs, dtype, op)
        else:
            oracle.simulate_bidir(bufs, dtype, op)
        for b in bufs:
            np.testing.assert_array_equal(b, folded)


# ------------------------------------------------------------- tree order

def test_tree_order_closed_form():
    """Tree order over 4 ranks is (x0 + x1) + (x2 + x3): with [2^24, 1, 1, 1]
    that is 2^24 + 2, where the ring order from rank 0 gives 2^24."""
    bufs = [np.array([v], dtype=np.float32) for v in [2.0 ** 24, 1.0, 1.0, 1.0]]
    oracle.tree_fold(bufs, "float32", "sum")
    assert bufs[0][0] == np.float32(2.0 ** 24 + 2)
    # odd count: ((x0 + x1) + x2) with the third entry carried one level
    bufs = [np.array([v], dtype=np.float32) for v in [2.0 ** 24, 1.0, 1.0]]
    oracle.tree_fold(bufs, "float32", "sum")
    assert bufs[0][0] == np.float32(2.0 ** 24)


def test_tree_order_fp32_error_bound():
    """|tree - exact| <= 4 p 2^-24 sum|x| elementwise."""
    for p in [2, 3, 8, 16, 64]:
        n = 300
        bufs = [rng.normal(0, 1, size=n).astype(np.float32) for _ in range(p)]
        ref, mag = oracle.f64_sum(bufs, "float32")
        oracle.tree_fold(bufs, "float32", "sum")
        assert np.all(np.abs(bufs[0] - ref) <= 4 * p * 2.0 ** -24 * mag)


@pytest.mark.parametrize("dtype,op", [("float32", "sum"), ("bfloat16", "sum"), ("float32", "max"),
                                      ("bfloat16", "avg"), ("int32", "sum")])
def test_tree_sampled_equals_full(dtype, op):
    """The per-element tree fold (used for the full-size checks of the tree
    executor) equals the whole-buffer tree fold on every rank, for odd, even
    and large p."""
    for p, n in [(2, 33), (7, 50), (8, 257), (64, 130)]:
        bufs = _rand_bufs(p, n, dtype, 99 + p)
        folded = oracle.fold_sampled(np.stack(bufs), np.arange(n), n, dtype, op, "tree")
        oracle.tree_fold(bufs, dtype, op)
        for b in bufs:
            np.testing.assert_array_equal(b, folded)


# ------------------------------------------------------------- trivial cases

def test_trivial_cases():
    """p == 1 leaves the buffer untouched ("An implementation": the torch ring
    returns t when p == 1); N == 0 is a no-op."""
    b = [np.arange(5, dtype=np.float32)]
    assert list(oracle.simulate(b, "float32", "sum")) == [0]
    np.testing.assert_array_equal(b[0], np.arange(5, dtype=np.float32))
    e = [np.zeros(0, dtype=np.float32) for _ in range(4)]
    assert list(oracle.simulate(e, "float32", "sum")) == [0, 0, 0, 0]


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "float16"])
def test_f64_sum_against_fsum(dtype):
    """orc_f64_sum, the fp64 reference behind the tree-order error bound:
    per element, the sum over ranks and the sum of magnitudes, accumulated
    in binary64.  Pinned against math.fsum (the correctly rounded sum) on
    mixed-sign inputs spanning many binades: a sequential binary64 sum is
    within (p - 1) 2^-53 sum|x| of it, which a binary32 accumulation, a
    dropped rank or a missing abs in the magnitudes would all exceed."""
    import math
    rng = np.random.default_rng(20261202)
    for p, n in [(2, 64), (7, 333), (64, 256)]:
        # magnitudes from 2^-10 to 2^10, random signs
        vals = rng.uniform(-1.0, 1.0, size=(p, n)) * np.exp2(rng.integers(-10, 11, size=(p, n)))
        if dtype == "float32":
            bufs = [v.astype(np.float32) for v in vals]
            as64 = np.stack([b.astype(np.float64) for b in bufs])
        else:
            conv = oracle.f32_to_bf16 if dtype == "bfloat16" else oracle.f32_to_f16
            back = oracle.bf16_to_f32 if dtype == "bfloat16" else oracle.f16_to_f32
            bufs = [np.array([conv(float(x)) for x in v], dtype=np.uint16) for v in vals]
            as64 = np.stack([[back(int(h)) for h in b] for b in bufs]).astype(np.float64)
        ref, mag = oracle.f64_sum(bufs, dtype)
        for i in range(n):
            exact = math.fsum(as64[:, i])
            exact_mag = math.fsum(np.abs(as64[:, i]))
            bound = (p - 1) * 2.0 ** -53 * exact_mag
            assert abs(ref[i] - exact) <= bound, (p, i)
            assert abs(mag[i] - exact_mag) <= bound, (p, i)
        # at least one element where binary32 accumulation is off by more
        # than the bound (so the check above can tell the two apart)
        f32 = np.zeros(n, dtype=np.float32)
        for r in range(p):
            f32 = (f32 + as64[r].astype(np.float32)).astype(np.float32)
        exact_all = np.array([math.fsum(as64[:, i]) for i in range(n)])
        mag_all = np.array([math.fsum(np.abs(as64[:, i])) for i in range(n)])
        if p > 2:
            assert np.any(np.abs(f32.astype(np.float64) - exact_all) > (p - 1) * 2.0 ** -53 * mag_all)


def test_f64_sum_exact_cases():
    """Integer-valued inputs: every partial sum is exact in binary64, so the
    sum and the magnitudes equal the integer sums; a rank with value 0
    everywhere and p = 1 included."""
    for p in (1, 3, 16):
        vals = [np.arange(-50, 50, dtype=np.float32) * (r - 1) for r in range(p)]
        ref, mag = oracle.f64_sum([v.copy() for v in vals], "float32")
        np.testing.assert_array_equal(ref, np.sum(np.stack(vals).astype(np.int64), axis=0).astype(np.float64))
        np.testing.assert_array_equal(mag, np.sum(np.abs(np.stack(vals).astype(np.int64)), axis=0).astype(np.float64))
