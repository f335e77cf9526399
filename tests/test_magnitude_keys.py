"""The signed 16-bit magnitude keys that the per-(token, head) write and the
scale calibration use to find the largest finite |x| of bf16 values.

A bf16 half h becomes key(h) = (h & 0x7FFF) + 0x80, read as a signed 16-bit
value: the finite magnitudes (bits 0 .. 0x7F7F) map onto 0x80 .. 0x7FFF in
their order and +-inf / NaN (bits 0x7F80 .. 0x7FFF) onto negative values, so
a signed max that starts at key(0) skips the non-finite values and
key - 0x80 of the result is the largest finite magnitude.  These checks are
exhaustive over the 65536 bf16 bit patterns; the GPU parity tests check the
kernels' scales bit for bit against the oracle's definition.
"""
import numpy as np

BITS = np.arange(1 << 16, dtype=np.int64)
MAG = BITS & 0x7FFF
FINITE = MAG < 0x7F80


def key_s16(bits):
    k = (bits & 0x7FFF) + 0x80
    return np.where(k >= 0x8000, k - 0x10000, k)


def test_no_carry_between_halves():
    # the largest key fits in 16 bits, so the 32-bit add of 0x00800080 to a
    # word of two halves never carries from the low half into the high one
    assert ((MAG + 0x80) < (1 << 16)).all()


def test_finite_keys_positive_and_ordered():
    k = key_s16(BITS)
    assert (k[FINITE] > 0).all()
    order = np.argsort(MAG[FINITE], kind="stable")
    assert (np.diff(k[FINITE][order]) >= 0).all()
    # equal magnitudes (x and -x) give equal keys
    assert (k[BITS[:0x8000]] == k[BITS[0x8000:]]).all()


def test_nonfinite_keys_negative():
    k = key_s16(BITS)
    assert (k[~FINITE] < 0).all()
    assert k[0x7F80] < 0 and k[0xFF80] < 0  # +-inf
    assert k[0x7FC0] < 0 and k[0xFFFF] < 0  # NaNs


def test_running_max_gives_largest_finite_magnitude():
    rng = np.random.default_rng(7)
    specials = np.array([0x0000, 0x8000, 0x0001, 0x7F7F, 0xFF7F, 0x7F80, 0xFF80, 0x7FC0, 0xFFFF,
                         0x3F80, 0xBF80], dtype=np.int64)
    for trial in range(4000):
        if trial % 3 == 0:
            vals = rng.choice(specials, 16)
        else:
            vals = rng.integers(0, 1 << 16, 16)
        want = int(np.where(FINITE[vals], MAG[vals], 0).max())
        got = max(0x80, int(key_s16(vals).max())) - 0x80
        assert got == want, (vals, want, got)


def test_all_nonfinite_row_gives_zero():
    vals = np.array([0x7F80, 0xFF80, 0x7FC0, 0xFFC1] * 4, dtype=np.int64)
    assert max(0x80, int(key_s16(vals).max())) - 0x80 == 0
