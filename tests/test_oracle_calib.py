"""Pins of the oracle's scale calibration (scale = amax / format max):
hand-worked values, the defining property that the largest magnitude lands
exactly on the format's largest finite code, and the ignored specials."""
import numpy as np
import pytest

import oracle
import workloads

E4, E5 = oracle.E4M3, oracle.E5M2


def bits(x):
    return workloads.f32_to_bf16_bits(np.asarray(x, np.float32))


def test_worked_values_per_head():
    # 3 tokens x 4 heads x 16 dims; head amax 896, 0 (all zero), 1.5, 57344
    x = np.zeros((3, 4, 16), np.float32)
    x[1, 0, 3] = -896.0
    x[0, 2, 7] = 1.5
    x[2, 2, 0] = -0.75
    x[2, 3, 15] = 57344.0
    s4 = oracle.calibrate(bits(x), oracle.PER_HEAD, E4)
    np.testing.assert_array_equal(s4, np.array([2.0, 1.0, np.float32(1.5) / np.float32(448),
                                                128.0], np.float32))
    s5 = oracle.calibrate(bits(x), oracle.PER_HEAD, E5)
    np.testing.assert_array_equal(s5, np.array([np.float32(896) / np.float32(57344), 1.0,
                                                np.float32(1.5) / np.float32(57344), 1.0],
                                               np.float32))
    st = oracle.calibrate(bits(x), oracle.PER_TENSOR, E4)
    np.testing.assert_array_equal(st, np.array([128.0], np.float32))


def test_specials_are_ignored_and_empty_gives_one():
    x = np.ones((2, 1, 16), np.float32)
    x[0, 0, 0] = np.nan
    x[1, 0, 1] = np.inf
    x[1, 0, 2] = -np.inf
    x[0, 0, 3] = -7.0
    np.testing.assert_array_equal(oracle.calibrate(bits(x), oracle.PER_TENSOR, E4),
                                  np.array([np.float32(7) / np.float32(448)], np.float32))
    empty = np.zeros((0, 3, 16), np.uint16)
    np.testing.assert_array_equal(oracle.calibrate(empty, oracle.PER_HEAD, E4), np.ones(3, np.float32))
    # the smallest bf16 subnormal (2^-133) still gives a (subnormal) quotient
    tiny = np.zeros((1, 1, 16), np.uint16)
    tiny[0, 0, 0] = 1
    for fmt, m in ((E4, 448), (E5, 57344)):
        got = oracle.calibrate(tiny, oracle.PER_TENSOR, fmt)
        assert got[0] == np.float32(2.0 ** -133) / np.float32(m) and 0 < got[0] < 2.0 ** -126


@pytest.mark.parametrize("fmt", [E4, E5])
def test_amax_lands_on_the_largest_code(fmt):
    r = np.random.default_rng(5)
    x = (r.standard_normal((200, 8, 64)) * 10.0 ** r.uniform(-3, 3, (1, 8, 1))).astype(np.float32)
    b = bits(x)
    s = oracle.calibrate(b, oracle.PER_HEAD, fmt)
    vals = (b.astype(np.uint32) << 16).view(np.float32)
    top = 0x7E if fmt == E4 else 0x7B
    for h in range(8):
        codes = oracle.quantize_bf16(fmt, b[:, h, :], float(s[h]))
        mags = np.abs(vals[:, h, :])
        i = np.unravel_index(np.argmax(mags), mags.shape)
        assert codes[i] & 0x7F == top               # amax -> the largest finite code
        assert np.all((codes & 0x7F) <= top)         # nothing beyond it
    # per tensor: the largest per-head scale
    st = oracle.calibrate(b, oracle.PER_TENSOR, fmt)
    assert st[0] == s.max()
