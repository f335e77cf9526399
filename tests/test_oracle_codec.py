"""Pins of the oracle's FP8 codec and write path against facts fixed outside it.

The pages name E4M3 / E5M2 and the write rule cast_fp8(K / sK) ("10.4 KV Cache
quantization", section 10.4.5); the bit layouts are the OCP 8-bit formats.
Each pin below is independent of the oracle's own code: code enumeration and
the formats' published constants, midpoint tie rules, torch's CPU float8
casts (RNE, non-saturating) on the domain where they do not saturate, the
KV-size worked example printed on the page, and brute force on tiny inputs.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import BF16, E4M3, E5M2, PER_HEAD, PER_TENSOR

HERE = os.path.dirname(os.path.abspath(__file__))
FMTS = [E4M3, E5M2]
MAX = {E4M3: 448.0, E5M2: 57344.0}
MAXCODE = {E4M3: 0x7E, E5M2: 0x7B}
MIN_SUB = {E4M3: 2.0 ** -9, E5M2: 2.0 ** -16}
# torch's casts are not saturating: above these magnitudes they give NaN / inf
TORCH_LIMIT = {E4M3: 464.0, E5M2: 61440.0}
TORCH_DT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def torch_codes(fmt, x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(TORCH_DT[fmt]).view(torch.uint8).numpy()


def f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


# ---------------------------------------------------------------- enumeration

@pytest.mark.parametrize("fmt", FMTS)
def test_all_256_codes(fmt):
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode(fmt, codes)
    nan = np.isnan(vals)
    inf = np.isinf(vals)
    finite = ~nan & ~inf
    if fmt == E4M3:
        assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
        assert not inf.any()
        assert finite.sum() == 254
    else:
        assert set(np.flatnonzero(nan)) == {0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF}
        assert set(np.flatnonzero(inf)) == {0x7C, 0xFC}
        assert finite.sum() == 248
    assert np.nanmax(vals[finite]) == MAX[fmt]
    assert vals[MAXCODE[fmt]] == MAX[fmt]
    assert vals[0x01] == MIN_SUB[fmt]
    assert vals[0x00] == 0.0 and not math.copysign(1.0, vals[0x00]) < 0
    assert vals[0x80] == 0.0 and math.copysign(1.0, vals[0x80]) < 0
    # sign symmetry and strict monotonicity of the positive half
    pos = vals[: MAXCODE[fmt] + 1]
    assert np.all(np.diff(pos) > 0)
    np.testing.assert_array_equal(vals[0x80: 0x80 + MAXCODE[fmt] + 1], -pos)
    # encode(decode(c)) is the identity on every finite code, signed zeros included
    fc = codes[finite]
    back = oracle.encode(fmt, vals[finite].astype(np.float32))
    np.testing.assert_array_equal(back, fc)
    # every finite code matches torch's float8 interpretation of the same byte
    tv = torch.from_numpy(fc.copy()).view(TORCH_DT[fmt]).to(torch.float64).numpy()
    np.testing.assert_array_equal(tv, vals[finite])


@pytest.mark.parametrize("fmt", FMTS)
def test_midpoints_round_to_even(fmt):
    codes = np.arange(0, MAXCODE[fmt], dtype=np.uint8)  # c and c+1 both finite
    lo = oracle.decode(fmt, codes)
    hi = oracle.decode(fmt, codes + 1)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.all(mid.astype(np.float64) == (lo + hi) / 2)  # midpoints are exact in fp32
    even = np.where(codes % 2 == 0, codes, codes + 1).astype(np.uint8)
    for sign, off in ((1, 0), (-1, 0x80)):
        m = (sign * mid).astype(np.float32)
        np.testing.assert_array_equal(oracle.encode(fmt, m), even + off)
        below = np.nextafter(m, np.float32(0))
        above = np.nextafter(m, np.float32(sign * np.inf))
        np.testing.assert_array_equal(oracle.encode(fmt, below), codes + off)
        np.testing.assert_array_equal(oracle.encode(fmt, above), codes + 1 + off)


@pytest.mark.parametrize("fmt", FMTS)
def test_saturation_and_specials(fmt):
    mx = MAX[fmt]
    big = np.array([mx, np.nextafter(np.float32(mx), np.float32(np.inf)), 1.5 * mx,
                    TORCH_LIMIT[fmt], 1e30, np.finfo(np.float32).max, np.inf], dtype=np.float32)
    np.testing.assert_array_equal(oracle.encode(fmt, big), MAXCODE[fmt])
    np.testing.assert_array_equal(oracle.encode(fmt, -big), 0x80 | MAXCODE[fmt])
    assert oracle.encode(fmt, [np.nan])[0] == 0x7F
    assert oracle.encode(fmt, [-np.nan])[0] == 0x7F
    # signed zero and underflow keep the sign
    tiny = np.array([0.0, 1e-30, f32(1)[()], MIN_SUB[fmt] / 2], dtype=np.float32)
    np.testing.assert_array_equal(oracle.encode(fmt, tiny), 0)
    np.testing.assert_array_equal(oracle.encode(fmt, -tiny), 0x80)


# ---------------------------------------------------------------- cross-check with torch

@pytest.mark.parametrize("fmt", FMTS)
def test_all_bf16_inputs_match_torch(fmt):
    x = f32(np.arange(65536, dtype=np.uint32) << 16)
    ok = np.isfinite(x) & (np.abs(x) < TORCH_LIMIT[fmt])
    np.testing.assert_array_equal(oracle.encode(fmt, x[ok]), torch_codes(fmt, x[ok]))
    sat = np.isfinite(x) & (np.abs(x) >= TORCH_LIMIT[fmt])
    got = oracle.encode(fmt, x[sat])
    np.testing.assert_array_equal(got & 0x7F, MAXCODE[fmt])


@pytest.mark.parametrize("fmt", FMTS)
def test_fp32_inputs_match_torch(fmt):
    r = np.random.default_rng(1234)
    # random bit patterns over the whole binary32 range, plus a dense sweep of
    # every pattern in [2^-20, 2^10) with a stride co-prime to the mantissa
    rand = r.integers(0, 2 ** 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    lo, hi = np.float32(2.0 ** -20).view(np.uint32), np.float32(2.0 ** 10).view(np.uint32)
    sweep = np.arange(lo, hi, 97, dtype=np.uint32)
    for bits in (rand, sweep, sweep | np.uint32(0x80000000)):
        x = f32(bits)
        ok = np.isfinite(x) & (np.abs(x) < TORCH_LIMIT[fmt])
        np.testing.assert_array_equal(oracle.encode(fmt, x[ok]), torch_codes(fmt, x[ok]))


# ---------------------------------------------------------------- write rule cast_fp8(x / s)

@pytest.mark.parametrize("fmt", FMTS)
def test_scale_one_is_plain_cast(fmt):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = f32(bits.astype(np.uint32) << 16)
    keep = ~np.isnan(x)
    np.testing.assert_array_equal(oracle.quantize_bf16(fmt, bits[keep], 1.0),
                                  oracle.encode(fmt, x[keep]))


@pytest.mark.parametrize("fmt", FMTS)
def test_quotient_is_binary32_division(fmt):
    """The quotient is rounded to binary32 before the FP8 rounding (two roundings)."""
    r = np.random.default_rng(7)
    bits = r.integers(0, 65536, size=200000).astype(np.uint16)
    x = f32(bits.astype(np.uint32) << 16)
    keep = np.isfinite(x)
    bits, x = bits[keep], x[keep]
    for s in (np.float32(0.0123), np.float32(3.7), np.float32(1.0 / 448.0), np.float32(0.1)):
        q32 = (torch.from_numpy(x) / torch.tensor(s, dtype=torch.float32)).numpy()
        expect = oracle.encode(fmt, q32)
        np.testing.assert_array_equal(oracle.quantize_bf16(fmt, bits, float(s)), expect)


@pytest.mark.parametrize("fmt", FMTS)
def test_round_trip_error_bound(fmt):
    """|x - dec(enc(x/s)) * s| <= 2^-(m+1) |x| in the normal range, half a
    subnormal quantum times s below it, and |x| - max*s above the range."""
    mbits = 3 if fmt == E4M3 else 2
    emin = -6 if fmt == E4M3 else -14
    r = np.random.default_rng(11)
    s = np.float32(0.37)
    x = (r.standard_normal(400000) * np.exp(r.uniform(-12, 12, 400000))).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16 inputs
    xb = f32(bits.astype(np.uint32) << 16).astype(np.float64)
    back = oracle.decode(fmt, oracle.quantize_bf16(fmt, bits, float(s))) * float(s)
    err = np.abs(xb - back)
    ratio = np.abs(xb) / float(s)
    slack = 1 + 2.0 ** -20
    normal = (ratio >= 2.0 ** emin) & (ratio <= MAX[fmt])
    assert np.all(err[normal] <= 2.0 ** -(mbits + 1) * np.abs(xb[normal]) * slack)
    sub = ratio < 2.0 ** emin
    assert np.all(err[sub] <= 2.0 ** (emin - mbits - 1) * float(s) * slack)
    over = ratio > MAX[fmt] * (1 + 2.0 ** -20)
    assert over.any()
    np.testing.assert_allclose(err[over], np.abs(xb[over]) - MAX[fmt] * float(s), rtol=1e-6)


def test_bf16_rounding_helper_matches_torch():
    r = np.random.default_rng(3)
    x = r.standard_normal(100000).astype(np.float32) * np.float32(1e3)
    x = np.concatenate([x, np.array([0.0, -0.0, np.inf, -np.inf, 1.00390625, 1.01171875], np.float32)])
    expect = torch.from_numpy(x).to(torch.bfloat16).view(torch.uint16).numpy()
    np.testing.assert_array_equal(oracle.f32_to_bf16(x), expect)


# ---------------------------------------------------------------- KV size formula

def test_kv_size_worked_example():
    rows = [ln.split() for ln in open(os.path.join(HERE, "golden", "kv_size_worked_example.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for L, B, H, S, dh, e, gib in rows:
        m = oracle.kv_bytes(int(L), int(B), int(H), int(S), int(dh), float(e))
        assert m == float(gib) * 2 ** 30


def test_kv_size_of_long_context_cache():
    """The long-context workload's paged FP8 cache (32 layers x 2048 blocks x
    8 KV heads x 16 tokens x 128 dims, K and V) is the page's 2 GiB; bf16 is 4 GiB."""
    layers, blocks, hkv, bs, dh = 32, 2048, 8, 16, 128
    for e, gib in ((1, 2), (2, 4)):
        allocated = 2 * layers * blocks * hkv * bs * dh * e
        assert allocated == oracle.kv_bytes(layers, 1, hkv, blocks * bs, dh, e) == gib * 2 ** 30


# ---------------------------------------------------------------- paged write

def _brute_force_write(k, v, slots, nb, hkv, bs, dh, ks, vs, gran, fmt, fill):
    """Pure-Python scatter, one element at a time, with the codec pinned above."""
    kc = {}
    vc = {}
    for t, slot in enumerate(slots):
        if slot < 0 or slot >= nb * bs:
            continue
        for h in range(hkv):
            for d in range(dh):
                key = (slot // bs, h, slot % bs, d)
                if fmt == BF16:
                    kc[key], vc[key] = k[t, h, d], v[t, h, d]
                else:
                    sk = ks[h if gran == PER_HEAD else 0]
                    sv = vs[h if gran == PER_HEAD else 0]
                    xk = np.float32(f32(np.uint32(k[t, h, d]) << 16)) / np.float32(sk)
                    xv = np.float32(f32(np.uint32(v[t, h, d]) << 16)) / np.float32(sv)
                    kc[key] = torch_codes(fmt, np.array([xk]))[0]
                    vc[key] = torch_codes(fmt, np.array([xv]))[0]
    K = np.full((nb, hkv, bs, dh), fill, dtype=np.uint16 if fmt == BF16 else np.uint8)
    V = K.copy()
    for key, val in kc.items():
        K[key] = val
    for key, val in vc.items():
        V[key] = val
    return K, V


@pytest.mark.parametrize("fmt,gran", [(E4M3, PER_TENSOR), (E5M2, PER_HEAD), (BF16, PER_TENSOR)])
def test_write_matches_brute_force(fmt, gran):
    r = np.random.default_rng(5)
    nb, hkv, bs, dh, n = 3, 2, 4, 8, 9
    k = (r.standard_normal((n, hkv, dh)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    v = (r.standard_normal((n, hkv, dh)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    slots = np.array([5, -1, 0, 11, 3, 12, 7, -1, 2], dtype=np.int64)  # 12 is out of range
    ks = np.array([0.013, 0.05], np.float32)[: (2 if gran == PER_HEAD else 1)]
    vs = np.array([0.02, 0.007], np.float32)[: (2 if gran == PER_HEAD else 1)]
    fill = 0x5A
    K = oracle.new_cache(nb, hkv, bs, dh, fmt, fill)
    V = oracle.new_cache(nb, hkv, bs, dh, fmt, fill)
    bad = oracle.write(k, v, slots, K, V, ks, vs, gran, fmt)
    assert bad == 1
    K2, V2 = _brute_force_write(k, v, slots, nb, hkv, bs, dh, ks, vs, gran, fmt, fill)
    np.testing.assert_array_equal(K, K2)
    np.testing.assert_array_equal(V, V2)


def test_write_token_stride():
    """K/V rows may be slices of a wider per-token row (token stride > Hkv*dh)."""
    r = np.random.default_rng(9)
    n, hkv, dh, nb, bs = 5, 2, 8, 2, 4
    wide = (r.standard_normal((n, 3 * hkv * dh)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    k = wide[:, hkv * dh: 2 * hkv * dh].reshape(n, hkv, dh)
    v = wide[:, 2 * hkv * dh:].reshape(n, hkv, dh)
    slots = np.arange(n, dtype=np.int64)
    ref_k = oracle.new_cache(nb, hkv, bs, dh, E4M3)
    ref_v = oracle.new_cache(nb, hkv, bs, dh, E4M3)
    oracle.write(k.copy(), v.copy(), slots, ref_k, ref_v, [0.01], [0.01], PER_TENSOR, E4M3)
    # strided call: pass the wide buffer with offsets through a flat view
    K = oracle.new_cache(nb, hkv, bs, dh, E4M3)
    V = oracle.new_cache(nb, hkv, bs, dh, E4M3)
    flat = np.ascontiguousarray(wide).reshape(-1)
    import ctypes
    L = oracle.lib()
    base = flat.ctypes.data
    L.kvqo_write(ctypes.c_void_p(base + 2 * hkv * dh), ctypes.c_void_p(base + 2 * 2 * hkv * dh),
                 3 * hkv * dh, slots.ctypes.data_as(ctypes.c_void_p), n, hkv, dh,
                 K.ctypes.data_as(ctypes.c_void_p), V.ctypes.data_as(ctypes.c_void_p), nb, bs,
                 np.array([0.01], np.float32).ctypes.data_as(ctypes.c_void_p),
                 np.array([0.01], np.float32).ctypes.data_as(ctypes.c_void_p), PER_TENSOR, E4M3, 1)
    np.testing.assert_array_equal(K, ref_k)
    np.testing.assert_array_equal(V, ref_v)


# ---------------------------------------------------------------- unfused dequant

@pytest.mark.parametrize("fmt", FMTS)
def test_dequant_matches_torch(fmt):
    r = np.random.default_rng(21)
    codes = r.integers(0, 256, size=(3, 2, 16, 8)).astype(np.uint8)
    codes[np.isnan(oracle.decode(fmt, codes)) | np.isinf(oracle.decode(fmt, codes))] = 0x11
    t = torch.from_numpy(codes.copy()).view(TORCH_DT[fmt])
    # scale 1: FP8 -> bf16 is exact
    np.testing.assert_array_equal(oracle.dequant(codes, [1.0], PER_TENSOR, fmt),
                                  t.to(torch.bfloat16).view(torch.uint16).numpy())
    # per-head scales: one binary32 product, then RNE to bf16
    s = np.array([0.0173, 2.5e-3], np.float32)
    prod = (t.to(torch.float32) * torch.from_numpy(s)[None, :, None, None])
    np.testing.assert_array_equal(oracle.dequant(codes, s, PER_HEAD, fmt),
                                  prod.to(torch.bfloat16).view(torch.uint16).numpy())
