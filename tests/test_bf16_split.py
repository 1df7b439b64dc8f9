"""The arithmetic the tensor-core multi-vector kernel rests on, checked on the host with
numpy: an fp32 value splits into three bfloat16 terms, each rounded to nearest (ties to
even), with both residuals exact in fp32, so x = x1 + x2 + x3 exactly; and the sum of the
nine products x_a * y_b of two split values equals x * y exactly (every bfloat16 product is
exact in fp32, and their sum is exact in fp64), i.e. no error beyond the fp32 sums that
accumulate the products. Rounding to bfloat16 is written from its definition (round the
fp32 bit pattern to its top 16 bits, to nearest, ties to even)."""
import numpy as np
import pytest


def bf16_rn(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bfloat16 (ties to even), returned as fp32; non-finite values pass."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    return np.where(np.isfinite(x), out, x).astype(np.float32)


def split3(x: np.ndarray):
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(invalid="ignore", over="ignore"):  # inf - inf beyond the largest bfloat16
        x1 = bf16_rn(x)
        r1 = (x - x1).astype(np.float32)  # exact in fp32
        x2 = bf16_rn(r1)
        x3 = bf16_rn((r1 - x2).astype(np.float32))
    return x1, x2, x3


def is_bf16(v: np.ndarray) -> bool:
    return bool(np.all((np.asarray(v, dtype=np.float32).view(np.uint32) & 0xFFFF) == 0))


def samples(seed=0, n=200_000):
    rng = np.random.default_rng(seed)
    parts = [
        rng.standard_normal(n).astype(np.float32),
        (rng.standard_normal(n) * 10.0 ** rng.uniform(-30, 30, n)).astype(np.float32),
        rng.uniform(-1, 1, n).astype(np.float32),
        # every mantissa pattern near 1, and halfway cases of the bfloat16 rounding
        (1.0 + np.arange(n, dtype=np.float32) * np.float32(2.0 ** -23)).astype(np.float32),
        np.float32(1.0) + np.float32(2.0 ** -8) * (np.arange(n) % 2).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0, 1.0 + 2.0 ** -23, 2.0 ** -100, 2.0 ** 100, 65504.0, 1e-30, 3.4e38],
                 dtype=np.float32),
    ]
    return np.concatenate(parts)


def test_bf16_rounding_against_a_direct_definition():
    """bf16_rn against a slow definition on a sample: the nearest of the two bfloat16
    neighbours, ties to the even one."""
    x = samples(1, 2000)
    x = x[np.isfinite(x) & (np.abs(x) < 3e38)]
    got = bf16_rn(x)
    for xi, gi in zip(x[:3000], got[:3000]):
        bits = np.float32(xi).view(np.uint32)
        lo = np.uint32(bits & 0xFFFF0000).view(np.float32)
        hi_bits = (int(bits) & 0xFFFF0000) + 0x10000
        hi = np.uint32(hi_bits & 0xFFFFFFFF).view(np.float32)
        dlo, dhi = abs(float(xi) - float(lo)), abs(float(hi) - float(xi))
        if dlo < dhi:
            want = lo
        elif dhi < dlo:
            want = hi
        else:
            want = lo if ((int(bits) >> 16) & 1) == 0 else hi
        assert np.float32(gi) == np.float32(want), (xi, gi, want)


def test_split_is_exact_and_each_term_is_bfloat16():
    x = samples()
    x = x[np.isfinite(x) & (np.abs(x) < 3.39e38)]
    x1, x2, x3 = split3(x)
    assert is_bf16(x1) and is_bf16(x2) and is_bf16(x3)
    # exact: summed in fp64 (no rounding there), the three terms give x back
    assert np.array_equal(x1.astype(np.float64) + x2.astype(np.float64) + x3.astype(np.float64), x.astype(np.float64))
    # sizes: |x2| <= 2^-8 |x|, |x3| <= 2^-16 |x| (up to the rounding of each step)
    nz = x != 0
    assert np.all(np.abs(x2[nz]) <= np.abs(x[nz]) * 2.0 ** -8 * (1 + 2.0 ** -7))
    assert np.all(np.abs(x3[nz]) <= np.abs(x[nz]) * 2.0 ** -16 * (1 + 2.0 ** -6))


def test_nine_products_give_the_exact_product():
    """Every product of two bfloat16 terms is exact in fp32 (8 + 8 significant bits), and the
    nine of them sum, in fp64, to x * y exactly: the split loses nothing; only the fp32
    accumulation of the products rounds."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(50_000) * 10.0 ** rng.uniform(-10, 10, 50_000)).astype(np.float32)
    y = (rng.standard_normal(50_000) * 10.0 ** rng.uniform(-10, 10, 50_000)).astype(np.float32)
    xs, ys = split3(x), split3(y)
    total = np.zeros(x.size, dtype=np.float64)
    for xa in xs:
        for yb in ys:
            p32 = (xa * yb).astype(np.float32)
            assert np.array_equal(p32.astype(np.float64), xa.astype(np.float64) * yb.astype(np.float64))
            total += p32.astype(np.float64)
    assert np.array_equal(total, x.astype(np.float64) * y.astype(np.float64))


@pytest.mark.parametrize("m", [128, 512])
def test_tile_sums_stay_within_the_fp32_bound(m):
    """The scatter's sums as the tensor cores form them: per step of K = 16 rows the products
    of the split terms summed (here in fp64) and added once, rounded to fp32, into
    the accumulator; 512 rows (32 steps) are what the kernel sums before folding them into
    its compensated column sums. The result stays within the fp32 entry points' 2e-5 S of the
    exact sum, S_j = sum_i |t_i| |x_ij|: 32 roundings cost at most 32 * 2^-24 S."""
    rng = np.random.default_rng(m)
    X = rng.standard_normal((m, 32)).astype(np.float32)
    t = rng.standard_normal(m).astype(np.float32)
    xs, ts = split3(X), split3(t)
    W = np.zeros(32, dtype=np.float32)
    for i0 in range(0, m, 16):
        step = np.zeros(32, dtype=np.float64)
        for xa in xs:
            for tb in ts:
                step += (tb[i0:i0 + 16, None].astype(np.float64) * xa[i0:i0 + 16].astype(np.float64)).sum(axis=0)
        W = (W.astype(np.float64) + step).astype(np.float32)
    exact = (t.astype(np.float64)[:, None] * X.astype(np.float64)).sum(axis=0)
    S = (np.abs(t.astype(np.float64))[:, None] * np.abs(X.astype(np.float64))).sum(axis=0)
    err = np.abs(W.astype(np.float64) - exact)
    assert np.all(err <= (m // 16) * 2.0 ** -24 * S * 1.01)
    assert np.all(err <= 2e-5 * S)


def test_values_beyond_the_largest_bfloat16_do_not_split():
    """The split's one limit: fp32 values within half a bfloat16 step of the fp32 maximum
    (|x| > 3.3961e38) round to infinity as bfloat16, so their terms are not finite."""
    big = np.array([3.39e38, 3.396e38, 3.4e38], dtype=np.float32)
    x1, _, _ = split3(big)
    assert np.isfinite(x1[0]) and not np.isfinite(x1[2])
