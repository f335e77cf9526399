"""Pins of the oracle's float64 decode attention over the dequantized cache.

Definition ("10.4 KV Cache quantization", section 10.4.2):
P = softmax(Q K^T / sqrt(dh) + mask), O = P V^, with K^ = cast_float(K_fp8) * sK
(section 10.4.5).  The pins: torch's float64 scaled_dot_product_attention on
the gathered K^/V^ (a library routine), a pure-Python brute force on a tiny
case, and invariants that hold whatever the values (uniform V, one token,
block-table permutation, window >= length, GQA head mapping, empty sequence).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import BF16, E4M3, E5M2, PER_HEAD, PER_TENSOR


def bits_from(x):
    return workloads.f32_to_bf16_bits(np.asarray(x, np.float32))


def _case(r, B, Hq, Hkv, dh, lens, fmt, gran, bs=16, std=1.0, spare=3):
    st = workloads._structure(np.array(lens), r, bs=bs, extra_blocks=spare)
    N = len(st.slot_mapping)
    q = bits_from(r.standard_normal((B, Hq, dh)))
    k = bits_from(r.standard_normal((N, Hkv, dh)) * std)
    v = bits_from(r.standard_normal((N, Hkv, dh)) * std)
    nsc = Hkv if gran == PER_HEAD else 1
    ks = (r.uniform(0.5, 2.0, nsc) * std / 64).astype(np.float32)
    vs = (r.uniform(0.5, 2.0, nsc) * std / 64).astype(np.float32)
    if fmt == BF16:
        ks = vs = np.ones(nsc, np.float32)
    K = oracle.new_cache(st.num_blocks, Hkv, bs, dh, fmt)
    V = oracle.new_cache(st.num_blocks, Hkv, bs, dh, fmt)
    assert oracle.write(k, v, st.slot_mapping, K, V, ks, vs, gran, fmt) == 0
    return st, q, K, V, ks, vs


def _gather(cache, st, b, fmt, scale, gran):
    """Contiguous dequantized [Hkv][L][dh] of sequence b via numpy indexing."""
    L = int(st.seq_lens[b])
    pos = np.arange(L)
    blk = st.block_tables[b, pos // cache.shape[2]]
    rows = cache[blk, :, pos % cache.shape[2], :]  # [L][Hkv][dh]
    if fmt == BF16:
        vals = oracle.bf16_to_f64(rows)
    else:
        s = np.asarray(scale, np.float64)
        s = s[None, :, None] if gran == PER_HEAD else s[0]
        vals = oracle.decode(fmt, rows) * s
    return np.transpose(vals, (1, 0, 2))


@pytest.mark.parametrize("fmt,gran", [(E4M3, PER_TENSOR), (E4M3, PER_HEAD), (E5M2, PER_HEAD),
                                      (BF16, PER_TENSOR)])
def test_matches_torch_sdpa_float64(fmt, gran):
    r = np.random.default_rng(100 + fmt)
    B, Hq, Hkv, dh = 3, 8, 2, 64
    st, q, K, V, ks, vs = _case(r, B, Hq, Hkv, dh, [37, 1, 70], fmt, gran)
    out = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, gran, fmt)
    G = Hq // Hkv
    for b in range(B):
        Kh = torch.from_numpy(_gather(K, st, b, fmt, ks, gran)).repeat_interleave(G, 0)
        Vh = torch.from_numpy(_gather(V, st, b, fmt, vs, gran)).repeat_interleave(G, 0)
        qb = torch.from_numpy(oracle.bf16_to_f64(q[b]))[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(qb, Kh, Vh)[:, 0, :].numpy()
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


def test_pure_python_brute_force():
    r = np.random.default_rng(8)
    B, Hq, Hkv, dh = 1, 2, 1, 4
    st, q, K, V, ks, vs = _case(r, B, Hq, Hkv, dh, [5], E4M3, PER_TENSOR, bs=2)
    out = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_TENSOR, E4M3)
    for h in range(Hq):
        qv = [float(oracle.bf16_to_f64(q[0, h, d])) for d in range(dh)]
        xs, vrows = [], []
        for t in range(5):
            blk, off = int(st.block_tables[0, t // 2]), t % 2
            kh = [float(oracle.decode(E4M3, K[blk, 0, off, d])) * float(ks[0]) for d in range(dh)]
            vh = [float(oracle.decode(E4M3, V[blk, 0, off, d])) * float(vs[0]) for d in range(dh)]
            xs.append(sum(a * b for a, b in zip(qv, kh)) / math.sqrt(dh))
            vrows.append(vh)
        m = max(xs)
        w = [math.exp(x - m) for x in xs]
        ref = [sum(w[t] * vrows[t][d] for t in range(5)) / sum(w) for d in range(dh)]
        np.testing.assert_allclose(out[0, h], ref, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("fmt", [E4M3, E5M2, BF16])
def test_uniform_v_gives_that_row(fmt):
    r = np.random.default_rng(31)
    B, Hq, Hkv, dh = 2, 4, 2, 64
    st, q, K, V, ks, vs = _case(r, B, Hq, Hkv, dh, [40, 17], fmt, PER_HEAD)
    V[:] = V[st.block_tables[0, 0], :, 0, :][None, :, None, :]
    out = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_HEAD, fmt)
    row = V[0, :, 0, :]
    vhat = oracle.bf16_to_f64(row) if fmt == BF16 else oracle.decode(fmt, row) * vs[:, None].astype(np.float64)
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_allclose(out[b, h], vhat[h // 2], rtol=1e-14, atol=0)


def test_one_token_gives_its_v():
    r = np.random.default_rng(32)
    st, q, K, V, ks, vs = _case(r, 2, 8, 2, 64, [1, 1], E4M3, PER_HEAD)
    out = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_HEAD, E4M3)
    for b in range(2):
        vh = _gather(V, st, b, E4M3, vs, PER_HEAD)[:, 0, :]
        for h in range(8):
            np.testing.assert_array_equal(out[b, h], vh[h // 4])


def test_block_permutation_invariance():
    r = np.random.default_rng(33)
    st, q, K, V, ks, vs = _case(r, 2, 8, 2, 64, [45, 30], E5M2, PER_HEAD)
    out = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_HEAD, E5M2)
    perm = r.permutation(st.num_blocks)
    K2 = np.empty_like(K)
    V2 = np.empty_like(V)
    K2[perm] = K
    V2[perm] = V
    bt = np.where(st.block_tables >= 0, perm[np.maximum(st.block_tables, 0)], -1).astype(np.int32)
    out2 = oracle.decode_attn(q, K2, V2, bt, st.seq_lens, ks, vs, PER_HEAD, E5M2)
    np.testing.assert_array_equal(out, out2)


def test_sliding_window():
    r = np.random.default_rng(34)
    st, q, K, V, ks, vs = _case(r, 2, 8, 2, 64, [50, 20], BF16, PER_TENSOR)
    full = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_TENSOR, BF16)
    same = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_TENSOR, BF16,
                              window=50)
    np.testing.assert_array_equal(full, same)
    W = 13
    win = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_TENSOR, BF16,
                             window=W)
    # reference: torch float64 over the newest W tokens only
    for b in range(2):
        L = int(st.seq_lens[b])
        Kh = torch.from_numpy(_gather(K, st, b, BF16, ks, PER_TENSOR)[:, L - W:]).repeat_interleave(4, 0)
        Vh = torch.from_numpy(_gather(V, st, b, BF16, vs, PER_TENSOR)[:, L - W:]).repeat_interleave(4, 0)
        qb = torch.from_numpy(oracle.bf16_to_f64(q[b]))[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(qb, Kh, Vh)[:, 0, :].numpy()
        np.testing.assert_allclose(win[b], ref, rtol=1e-12, atol=1e-12)


def test_gqa_head_mapping_and_per_head_scales():
    """Query head h reads KV head h // (Hq/Hkv) with that head's scales."""
    r = np.random.default_rng(35)
    B, Hq, Hkv, dh = 1, 8, 4, 64
    st, q, K, V, ks, vs = _case(r, B, Hq, Hkv, dh, [1], E4M3, PER_HEAD)
    vs = np.array([1.0, 2.0, 4.0, 8.0], np.float32)
    out = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_HEAD, E4M3)
    blk = st.block_tables[0, 0]
    for h in range(Hq):
        np.testing.assert_array_equal(out[0, h], oracle.decode(E4M3, V[blk, h // 2, 0]) * vs[h // 2])


def test_empty_sequence_and_pairs():
    r = np.random.default_rng(36)
    st, q, K, V, ks, vs = _case(r, 3, 8, 2, 64, [10, 1, 33], E4M3, PER_TENSOR)
    sl = st.seq_lens.copy()
    sl[1] = 0
    out = oracle.decode_attn(q, K, V, st.block_tables, sl, ks, vs, PER_TENSOR, E4M3)
    assert np.all(out[1] == 0)
    pairs = np.array([[2, 7], [0, 3], [2, 0]], np.int32)
    sub = oracle.decode_attn(q, K, V, st.block_tables, sl, ks, vs, PER_TENSOR, E4M3, pairs=pairs)
    for i, (b, h) in enumerate(pairs):
        np.testing.assert_array_equal(sub[i], out[b, h])


def test_bad_block_id_is_reported():
    r = np.random.default_rng(37)
    st, q, K, V, ks, vs = _case(r, 1, 8, 2, 64, [20], E4M3, PER_TENSOR)
    bt = st.block_tables.copy()
    bt[0, 1] = st.num_blocks + 5
    with pytest.raises(ValueError):
        oracle.decode_attn(q, K, V, bt, st.seq_lens, ks, vs, PER_TENSOR, E4M3)


# ---------------------------------------------------------------- FP8-domain query mode

def _q_hat(q_bits, q_scale, per_head, fmt):
    """dec(enc(fp32(q) / sQ)) * sQ in the cache's format with the (separately
    pinned) codec, numpy binary32 division."""
    qf = (np.asarray(q_bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
    hq = qf.shape[1]
    s = np.asarray(q_scale, np.float32)
    s = (s if per_head else np.repeat(s, hq)).reshape(1, hq, 1)
    codes = oracle.encode(fmt, (qf / s).astype(np.float32))
    return oracle.decode(fmt, codes) * s.astype(np.float64)


@pytest.mark.parametrize("fmt,per_head", [(E4M3, False), (E4M3, True), (E5M2, True)])
def test_q_fp8_matches_sdpa_on_the_quantized_query(fmt, per_head):
    r = np.random.default_rng(300 + fmt + per_head)
    B, Hq, Hkv, dh = 2, 8, 2, 64
    st, q, K, V, ks, vs = _case(r, B, Hq, Hkv, dh, [45, 17], fmt, PER_HEAD)
    qs = (r.uniform(0.5, 2.0, Hq if per_head else 1) / 200).astype(np.float32)
    out = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_HEAD, fmt,
                             q_scale=qs)
    qh = _q_hat(q, qs, per_head, fmt)
    G = Hq // Hkv
    for b in range(B):
        Kh = torch.from_numpy(_gather(K, st, b, fmt, ks, PER_HEAD)).repeat_interleave(G, 0)
        Vh = torch.from_numpy(_gather(V, st, b, fmt, vs, PER_HEAD)).repeat_interleave(G, 0)
        qb = torch.from_numpy(qh[b])[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(qb, Kh, Vh)[:, 0, :].numpy()
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)
    # the quantized query differs from the bf16 one, so the outputs do too
    plain = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_HEAD, fmt)
    assert not np.array_equal(plain, out)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_q_fp8_is_exact_for_representable_queries(fmt):
    """Queries that are codes of the cache's format times a power-of-two
    scale come back unchanged, so the FP8-domain mode equals the plain one."""
    r = np.random.default_rng(9 + fmt)
    B, Hq, Hkv, dh = 2, 4, 2, 64
    st, _, K, V, ks, vs = _case(r, B, Hq, Hkv, dh, [30, 64], fmt, PER_TENSOR)
    top = 0x7E if fmt == E4M3 else 0x7B  # largest finite code
    codes = r.integers(0, top + 1, size=(B, Hq, dh)).astype(np.uint8)
    codes |= (r.integers(0, 2, size=codes.shape) << 7).astype(np.uint8)  # both signs
    sq = np.float32(2.0 ** -7)
    q = bits_from(oracle.decode(fmt, codes) * sq)  # exact in bf16 (at most 4 significant bits)
    a = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_TENSOR, fmt)
    b = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_TENSOR, fmt,
                           q_scale=np.array([sq], np.float32))
    np.testing.assert_array_equal(a, b)


def test_q_fp8_per_head_scales_are_indexed_by_query_head():
    r = np.random.default_rng(10)
    B, Hq, Hkv, dh = 1, 4, 1, 64
    st, q, K, V, ks, vs = _case(r, B, Hq, Hkv, dh, [20], E4M3, PER_TENSOR)
    qs = np.array([0.01, 0.02, 0.003, 0.05], np.float32)
    per_head = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_TENSOR, E4M3,
                                  q_scale=qs)
    for h in range(Hq):
        one = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_TENSOR, E4M3,
                                 q_scale=qs[h:h + 1])
        np.testing.assert_array_equal(per_head[0, h], one[0, h])
