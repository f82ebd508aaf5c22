"""The fixed-point rounding the dq kernel uses for its dT bins, checked as IEEE
float32 arithmetic on the host (numpy rounds every float32 add to nearest even,
as the kernel's packed adds do).

For |v| < 2^29: h = v + 1.5 * 2^30 has a unit in the last place of 128, so h =
1.5 * 2^30 + a with a a multiple of 128 within 64 of v; u = (1.5 * 2^30 + 1.5 *
2^23) - h = 1.5 * 2^23 - a is exact; b = v + u rounds once, to 1.5 * 2^23 +
round(v - a).  Then bits(h) * 128 + bits(b) - (bits(1.5 * 2^30) * 128 +
bits(1.5 * 2^23)) = a + round(v - a) = round(v), modulo 2^32."""
import numpy as np

C1 = np.float32(1.5 * 2 ** 30)
C12 = np.float32(1.5 * 2 ** 30 + 1.5 * 2 ** 23)
BIAS = ((0x4EC00000 << 7) + 0x4B400000) & 0xFFFFFFFF


def round_fixed(v: np.ndarray) -> np.ndarray:
    h = v + C1
    u = C12 - h
    b = v + u
    w = ((h.view(np.uint32).astype(np.uint64) << 7) + b.view(np.uint32) - BIAS) & 0xFFFFFFFF
    return w.astype(np.uint32).view(np.int32).astype(np.int64)


def test_constants_are_exact_floats():
    assert float(C12) == 1.5 * 2 ** 30 + 1.5 * 2 ** 23
    assert int(np.float32(1.5 * 2 ** 30).view(np.uint32)) == 0x4EC00000
    assert int(np.float32(1.5 * 2 ** 23).view(np.uint32)) == 0x4B400000


def test_matches_round_half_even_over_the_range():
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.uniform(-2 ** 29 + 64, 2 ** 29 - 64, 1_000_000),
        rng.normal(0.0, 200.0, 500_000),
        rng.integers(-2 ** 27, 2 ** 27, 300_000) + 0.5,      # ties at every scale
        rng.integers(-4096, 4096, 100_000) * 128.0 + 64.0,   # ties on the 128 grid
        np.array([0.0, -0.0, 0.5, -0.5, 1.5, 2.5, 63.5, 64.0, 64.5, -64.5, 127.5, 128.5,
                  2 ** 29 - 128.0, -(2 ** 29 - 128.0), 2 ** 29 - 0.5]),
    ]).astype(np.float32)
    v = v[np.abs(v) < 2 ** 29]
    assert np.array_equal(round_fixed(v), np.rint(v.astype(np.float64)).astype(np.int64))


def test_a_planted_mistake_is_caught():
    # dropping the 1.5 * 2^23 part of the second constant breaks every value
    v = np.array([1.0, 2.5, -3.25, 1000.75], np.float32)
    h = v + C1
    b = v + (C1 - h)
    w = ((h.view(np.uint32).astype(np.uint64) << 7) + b.view(np.uint32) - BIAS) & 0xFFFFFFFF
    assert not np.array_equal(w.astype(np.uint32).view(np.int32), np.rint(v).astype(np.int32))
