"""The fixed-point rounding the dq kernel uses for its dT bins, checked as IEEE
float32 arithmetic on the host (numpy rounds every float32 add to nearest even,
as the kernel's packed adds do).

For |v| < 2^29: h = v + C1, C1 = bits 0x4FDA7FFF in [2^32, 2^33), has a unit in
the last place of 512, so h = C1 + a with a a multiple of 512 within 256 of v;
u = (C1 + C2) - h = C2 - a is exact for C2 = 2^23 + 512; b = v + u rounds once, to
C2 + round(v - a).  512 bits(h) + bits(b) = 512 bits(C1) + bits(C2) + a + round(v -
a) = round(v) modulo 2^32, since 512 bits(C1) + bits(C2) = 0 mod 2^32."""
import numpy as np

C1 = np.array([0x4FDA7FFF], np.uint32).view(np.float32)[0]
C2 = np.array([0x4B000200], np.uint32).view(np.float32)[0]
C12 = np.float32(7340032000.0)


def round_fixed(v: np.ndarray, c1=C1, c12=C12) -> np.ndarray:
    h = v + c1
    u = c12 - h
    b = v + u
    w = ((h.view(np.uint32).astype(np.uint64) << 9) + b.view(np.uint32)) & 0xFFFFFFFF
    return w.astype(np.uint32).view(np.int32).astype(np.int64)


def test_constants():
    # the decimal literals the kernel writes are these floats, exactly
    assert float(C1) == 7331642880.0 and float(C2) == 2.0 ** 23 + 512
    assert float(C12) == float(C1) + float(C2)
    # the offset cancels modulo 2^32, and v + C1 stays in C1's binade for |v| < 2^29
    assert (512 * 0x4FDA7FFF + 0x4B000200) % 2 ** 32 == 0
    assert 2.0 ** 32 < float(C1) - 2 ** 29 and float(C1) + 2 ** 29 < 2.0 ** 33


def test_matches_round_half_even_over_the_range():
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.uniform(-2 ** 29 + 512, 2 ** 29 - 512, 1_000_000),
        rng.normal(0.0, 300.0, 500_000),
        rng.integers(-2 ** 27, 2 ** 27, 300_000) + 0.5,       # ties at every scale
        rng.integers(-4096, 4096, 100_000) * 512.0 + 256.0,   # ties on the 512 grid
        np.array([0.0, -0.0, 0.5, -0.5, 1.5, 2.5, 255.5, 256.0, 256.5, -256.5, 511.5, 512.5,
                  2 ** 29 - 512.0, -(2 ** 29 - 512.0), 2 ** 29 - 1.0]),
    ]).astype(np.float32)
    v = v[np.abs(v) < 2 ** 29]
    assert np.array_equal(round_fixed(v), np.rint(v.astype(np.float64)).astype(np.int64))


def test_a_planted_mistake_is_caught():
    # a second constant that misses the 2^23 + 512 part breaks every value
    v = np.array([1.0, 2.5, -3.25, 1000.75], np.float32)
    assert not np.array_equal(round_fixed(v, c12=np.float32(float(C1))), np.rint(v).astype(np.int64))
