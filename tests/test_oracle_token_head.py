"""Pins of the oracle's per-(token, KV head) scale mode ("10.4 KV Cache
quantization", section 10.4.3, per-token granularity; vLLM's
fp8_per_token_head): the pages' metadata arithmetic, hand-worked rows, the
scale's defining property (a row's largest finite magnitude lands on the
format's largest code), power-of-two equivariance, the reduction to the
per-head mode when every row of a head has the same amax, the round-trip
error bound, and attention against torch float64 SDPA on the rebuilt
K and V."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

HERE = os.path.dirname(os.path.abspath(__file__))
E4, E5 = oracle.E4M3, oracle.E5M2
TOP = {E4: 0x7E, E5: 0x7B}
PTH = oracle.PER_TOKEN_HEAD


def bits(x):
    return workloads.f32_to_bf16_bits(np.asarray(x, np.float32))


def test_metadata_worked_example():
    rows, ratio = [], None
    for ln in open(os.path.join(HERE, "golden", "per_token_head_metadata.txt")):
        f = ln.split()
        if not f or f[0].startswith("#"):
            continue
        if f[0] == "ratio":
            ratio = float(f[1])
            continue
        rows.append([float(x) for x in f])
    got = []
    for dh, pb, sb, want in rows:
        # bytes of one (token, head): K and V rows of one layer, one sequence, one head
        per = oracle.kv_bytes(1, 1, 1, 1, int(dh), pb, sb)
        assert per == want
        got.append(per)
    assert round(got[0] / got[1], 2) == ratio
    # the same arithmetic for this cache: FP8 codes + one binary32 scale per row
    assert oracle.kv_bytes(1, 1, 1, 1, 128, 1, 4) == 264


def _write(k, v, fmt, bs=16, nb=None, slots=None, fill=0):
    n, hkv, dh = k.shape
    nb = nb or (n + bs - 1) // bs + 1
    K = oracle.new_cache(nb, hkv, bs, dh, fmt, fill)
    V = oracle.new_cache(nb, hkv, bs, dh, fmt, fill)
    sK = oracle.new_scale_cache(nb, hkv, bs, -1.0)
    sV = oracle.new_scale_cache(nb, hkv, bs, -1.0)
    slots = np.arange(n, dtype=np.int64) if slots is None else np.asarray(slots, np.int64)
    bad = oracle.write(k, v, slots, K, V, sK, sV, PTH, fmt)
    return bad, K, V, sK, sV


def test_worked_rows():
    # one head of 16 dims; rows: amax 896 (one element), all zero, specials
    x = np.zeros((3, 1, 16), np.float32)
    x[0, 0, :4] = [896.0, 1.0, -3.5, 0.0]
    x[2, 0, :5] = [np.nan, np.inf, -np.inf, 7.0, -0.0]
    b = bits(x)
    bad, K, _, sK, _ = _write(b, b, E4)
    assert bad == 0
    assert sK[0, 0, 0] == 2.0 and sK[0, 0, 1] == 1.0 and sK[0, 0, 2] == np.float32(7) / np.float32(448)
    # 896/2 = 448 -> 0x7E; 1/2 = 0.5 -> 0x30; -3.5/2 = -1.75 -> 0xBE; 0 -> 0x00
    assert list(K[0, 0, 0, :4]) == [0x7E, 0x30, 0xBE, 0x00]
    assert not K[0, 0, 1].any()  # zero row: scale 1, zero codes
    row = K[0, 0, 2]
    assert row[0] & 0x7F == 0x7F          # NaN -> a NaN code
    assert row[1] == 0x7E and row[2] == 0xFE  # +-inf saturate
    assert row[3] == 0x7E and row[4] == 0x80  # the finite amax -> top code; -0 kept
    # E5M2: 896 / (896/57344) = 57344 -> 0x7B
    _, K5, _, sK5, _ = _write(b, b, E5)
    assert sK5[0, 0, 0] == np.float32(896) / np.float32(57344) and K5[0, 0, 0, 0] == 0x7B


@pytest.mark.parametrize("fmt", [E4, E5])
def test_amax_lands_on_top_code_and_slots(fmt):
    r = np.random.default_rng(11 + fmt)
    n, hkv, dh = 45, 4, 64
    x = r.standard_normal((n, hkv, dh)) * 10.0 ** r.uniform(-4, 4, (n, hkv, 1))
    k, v = bits(x), bits(-2 * x)
    slots = r.permutation(64)[:n].astype(np.int64)
    slots[5] = -1  # padding
    bad, K, V, sK, sV = _write(k, v, fmt, nb=4, slots=slots, fill=0x55)
    assert bad == 0
    for cache, sc, src in ((K, sK, k), (V, sV, v)):
        vals = np.abs((src.astype(np.uint32) << 16).view(np.float32))
        for t in range(n):
            if slots[t] < 0:
                continue
            blk, off = divmod(int(slots[t]), 16)
            for h in range(hkv):
                codes = cache[blk, h, off]
                i = int(np.argmax(vals[t, h]))
                assert codes[i] & 0x7F == TOP[fmt]
                assert np.all(codes & 0x7F <= TOP[fmt])
                assert sc[blk, h, off] == np.float32(vals[t, h].max()) / np.float32(oracle.FMT_MAX[fmt])
    # untouched slots keep their fill, scales included
    used = set(int(s) for s in slots if s >= 0)
    for s in range(64):
        if s not in used:
            blk, off = divmod(s, 16)
            assert np.all(K[blk, :, off] == 0x55) and np.all(sK[blk, :, off] == -1.0)


@pytest.mark.parametrize("fmt", [E4, E5])
def test_power_of_two_equivariance(fmt):
    r = np.random.default_rng(21)
    x = (r.standard_normal((20, 2, 64)) * 3).astype(np.float32)
    b1 = bits(x)
    b2 = bits(x * np.float32(2.0 ** 9))  # exact in bf16
    _, K1, _, s1, _ = _write(b1, b1, fmt)
    _, K2, _, s2, _ = _write(b2, b2, fmt)
    np.testing.assert_array_equal(K1, K2)
    w1 = s1.transpose(0, 2, 1).reshape(-1, 2)[:20]  # the 20 written rows, [token][head]
    w2 = s2.transpose(0, 2, 1).reshape(-1, 2)[:20]
    np.testing.assert_array_equal(w2, w1 * np.float32(2.0 ** 9))


@pytest.mark.parametrize("fmt", [E4, E5])
def test_equal_row_amax_reduces_to_per_head(fmt):
    """Rows of head h all with amax A_h: the per-token scales are A_h / fmt_max
    and the codes are those of the per-head mode with that scale; so is the
    attention output."""
    r = np.random.default_rng(31)
    lens = [37, 70]
    st = workloads._structure(np.array(lens), r, extra_blocks=2)
    N, hkv, hq, dh = len(st.slot_mapping), 2, 8, 64
    A = np.array([3.0, 0.25], np.float32)
    def rows():
        x = r.uniform(-1, 1, (N, hkv, dh)).astype(np.float32) * A[None, :, None] * 0.9
        j = r.integers(0, dh, N)
        x[np.arange(N), :, j] = A[None, :] * np.where(r.random((N, 1)) < 0.5, -1, 1)
        return bits(x)
    k, v = rows(), rows()
    q = bits(r.standard_normal((2, hq, dh)))
    nb = st.num_blocks
    K1 = oracle.new_cache(nb, hkv, 16, dh, fmt)
    V1 = oracle.new_cache(nb, hkv, 16, dh, fmt)
    sK = oracle.new_scale_cache(nb, hkv, 16, 1.0)
    sV = oracle.new_scale_cache(nb, hkv, 16, 1.0)
    assert oracle.write(k, v, st.slot_mapping, K1, V1, sK, sV, PTH, fmt) == 0
    s_head = (A / np.float32(oracle.FMT_MAX[fmt])).astype(np.float32)
    K2 = oracle.new_cache(nb, hkv, 16, dh, fmt)
    V2 = oracle.new_cache(nb, hkv, 16, dh, fmt)
    assert oracle.write(k, v, st.slot_mapping, K2, V2, s_head, s_head, oracle.PER_HEAD, fmt) == 0
    np.testing.assert_array_equal(K1, K2)
    np.testing.assert_array_equal(V1, V2)
    for b in range(2):
        for pos in range(lens[b]):
            blk = st.block_tables[b, pos // 16]
            np.testing.assert_array_equal(sK[blk, :, pos % 16], s_head)
    o1 = oracle.decode_attn(q, K1, V1, st.block_tables, st.seq_lens, sK, sV, PTH, fmt)
    o2 = oracle.decode_attn(q, K2, V2, st.block_tables, st.seq_lens, s_head, s_head,
                            oracle.PER_HEAD, fmt)
    np.testing.assert_array_equal(o1, o2)


@pytest.mark.parametrize("fmt,rel,sub", [(E4, 2.0 ** -4, 2.0 ** -10), (E5, 2.0 ** -3, 2.0 ** -17)])
def test_round_trip_error_bound(fmt, rel, sub):
    """|dec(code) s - x| <= max(rel |x|, sub s) (half an FP8 ulp, relative in
    the normal range, absolute in the subnormal one), widened by the binary32
    quotient's rounding."""
    r = np.random.default_rng(41)
    x = r.standard_normal((30, 3, 128)) * 10.0 ** r.uniform(-3, 3, (30, 3, 1))
    b = bits(x)
    _, K, _, sK, _ = _write(b, b, fmt, nb=3)
    xv = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for t in range(30):
        blk, off = divmod(t, 16)
        for h in range(3):
            s = float(sK[blk, h, off])
            y = oracle.decode(fmt, K[blk, h, off]) * s
            bound = np.maximum(rel * np.abs(xv[t, h]), sub * s) * (1 + 2.0 ** -20)
            assert np.all(np.abs(y - xv[t, h]) <= bound)


@pytest.mark.parametrize("fmt", [E4, E5])
def test_decode_matches_sdpa(fmt):
    r = np.random.default_rng(51 + fmt)
    lens = [45, 17, 100]
    st = workloads._structure(np.array(lens), r, extra_blocks=2)
    N, hkv, hq, dh = len(st.slot_mapping), 2, 8, 64
    x = r.standard_normal((N, hkv, dh)) * 10.0 ** r.uniform(-1, 1, (N, hkv, 1))
    k, v = bits(x), bits(r.standard_normal((N, hkv, dh)))
    q = bits(r.standard_normal((3, hq, dh)))
    nb = st.num_blocks
    K = oracle.new_cache(nb, hkv, 16, dh, fmt)
    V = oracle.new_cache(nb, hkv, 16, dh, fmt)
    sK = oracle.new_scale_cache(nb, hkv, 16)
    sV = oracle.new_scale_cache(nb, hkv, 16)
    assert oracle.write(k, v, st.slot_mapping, K, V, sK, sV, PTH, fmt) == 0
    out = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, sK, sV, PTH, fmt)
    qf = (q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    G = hq // hkv
    for b, L in enumerate(lens):
        pos = np.arange(L)
        blk = st.block_tables[b, pos // 16]
        off = pos % 16
        Kh = oracle.decode(fmt, K[blk, :, off]) * sK[blk, :, off][..., None]  # [L][Hkv][dh]
        Vh = oracle.decode(fmt, V[blk, :, off]) * sV[blk, :, off][..., None]
        Kt = torch.from_numpy(Kh.transpose(1, 0, 2)).repeat_interleave(G, 0)
        Vt = torch.from_numpy(Vh.transpose(1, 0, 2)).repeat_interleave(G, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qf[b])[:, None, :], Kt, Vt)[:, 0, :].numpy()
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


def test_dequant_uses_the_row_scale():
    r = np.random.default_rng(61)
    x = r.standard_normal((32, 2, 64)) * 10.0 ** r.uniform(-2, 2, (32, 2, 1))
    b = bits(x)
    _, K, _, sK, _ = _write(b, b, E4, nb=2)
    out = oracle.dequant(K, sK, PTH, E4)
    for blk in range(2):
        for h in range(2):
            for off in range(16):
                want = torch.from_numpy(
                    (oracle.decode(E4, K[blk, h, off]) * float(sK[blk, h, off])).astype(np.float32)
                ).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
                np.testing.assert_array_equal(out[blk, h, off], want)
