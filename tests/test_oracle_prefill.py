"""Pins of the oracle's float64 prefill / prefix-hit attention ("10.4 KV Cache
quantization", section 10.4.2: prefill, decode and prefix-hit paths read the
same quantized cache).  The last n_b tokens of sequence b are queries; query
j sits at position pos = L_b - n_b + j and attends causally to the cached
tokens [lo, pos] (lo from the sliding window).  Pins: torch float64 SDPA with
an explicit causal (and window) mask over the gathered K^/V^, the decode as
the one-query case, causality (tokens after pos do not matter), chunk-split
invariance, refusal of more queries than cached tokens, block-permutation
invariance and a uniform V (every output is that row)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import BF16, E4M3, E5M2, PER_HEAD, PER_TENSOR


def bits(x):
    return workloads.f32_to_bf16_bits(np.asarray(x, np.float32))


def _case(r, lens, Hq, Hkv, dh, fmt, gran, spare=3):
    st = workloads._structure(np.array(lens), r, extra_blocks=spare)
    N = len(st.slot_mapping)
    k = bits(r.standard_normal((N, Hkv, dh)))
    v = bits(r.standard_normal((N, Hkv, dh)))
    nsc = Hkv if gran == PER_HEAD else 1
    ks = (r.uniform(0.5, 2.0, nsc) / 64).astype(np.float32)
    vs = (r.uniform(0.5, 2.0, nsc) / 64).astype(np.float32)
    if fmt == BF16:
        ks = vs = np.ones(nsc, np.float32)
    K = oracle.new_cache(st.num_blocks, Hkv, 16, dh, fmt)
    V = oracle.new_cache(st.num_blocks, Hkv, 16, dh, fmt)
    assert oracle.write(k, v, st.slot_mapping, K, V, ks, vs, gran, fmt) == 0
    return st, K, V, ks, vs


def _gather(cache, st, b, fmt, scale, gran):
    """Dequantized [Hkv][L][dh] of sequence b via numpy indexing."""
    L = int(st.seq_lens[b])
    pos = np.arange(L)
    rows = cache[st.block_tables[b, pos // 16], :, pos % 16, :]
    if fmt == BF16:
        vals = oracle.bf16_to_f64(rows)
    else:
        s = np.asarray(scale, np.float64)
        vals = oracle.decode(fmt, rows) * (s[None, :, None] if gran == PER_HEAD else s[0])
    return np.transpose(vals, (1, 0, 2))


@pytest.mark.parametrize("fmt,gran,window", [(E4M3, PER_HEAD, 0), (E5M2, PER_TENSOR, 0),
                                             (BF16, PER_TENSOR, 0), (E4M3, PER_HEAD, 20)])
def test_matches_sdpa_with_causal_mask(fmt, gran, window):
    r = np.random.default_rng(200 + fmt + window)
    lens, nq = [70, 33, 16], [70, 5, 1]  # a full prefill, a prefix hit, one token
    Hq, Hkv, dh = 8, 2, 64
    st, K, V, ks, vs = _case(r, lens, Hq, Hkv, dh, fmt, gran)
    cu = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = bits(r.standard_normal((cu[-1], Hq, dh)))
    out = oracle.prefill_attn(q, cu, K, V, st.block_tables, st.seq_lens, ks, vs, gran, fmt,
                              window=window)
    G = Hq // Hkv
    for b, (L, n) in enumerate(zip(lens, nq)):
        Kh = torch.from_numpy(_gather(K, st, b, fmt, ks, gran)).repeat_interleave(G, 0)
        Vh = torch.from_numpy(_gather(V, st, b, fmt, vs, gran)).repeat_interleave(G, 0)
        qb = torch.from_numpy(oracle.bf16_to_f64(q[cu[b]:cu[b + 1]]).transpose(1, 0, 2))
        pos = L - n + np.arange(n)
        t = np.arange(L)
        mask = t[None, :] <= pos[:, None]
        if window:
            mask &= t[None, :] > pos[:, None] - window
        ref = torch.nn.functional.scaled_dot_product_attention(
            qb, Kh, Vh, attn_mask=torch.from_numpy(mask)).numpy().transpose(1, 0, 2)
        np.testing.assert_allclose(out[cu[b]:cu[b + 1]], ref, rtol=1e-12, atol=1e-12)


def test_one_query_is_the_decode():
    r = np.random.default_rng(210)
    lens = [45, 100, 3]
    st, K, V, ks, vs = _case(r, lens, 8, 2, 64, E4M3, PER_HEAD)
    q = bits(r.standard_normal((3, 8, 64)))
    cu = np.arange(4, dtype=np.int32)
    a = oracle.prefill_attn(q, cu, K, V, st.block_tables, st.seq_lens, ks, vs, PER_HEAD, E4M3)
    b = oracle.decode_attn(q, K, V, st.block_tables, st.seq_lens, ks, vs, PER_HEAD, E4M3)
    np.testing.assert_array_equal(a, b)


def test_causality_and_chunk_split():
    r = np.random.default_rng(220)
    L, n = 90, 40
    st, K, V, ks, vs = _case(r, [L], 4, 1, 64, E4M3, PER_TENSOR)
    q = bits(r.standard_normal((n, 4, 64)))
    cu = np.array([0, n], np.int32)
    full = oracle.prefill_attn(q, cu, K, V, st.block_tables, st.seq_lens, ks, vs, PER_TENSOR,
                               E4M3)
    # the cache after position 69 only matters to the queries at 70 and later
    K2, V2 = K.copy(), V.copy()
    for t in range(70, L):
        blk = st.block_tables[0, t // 16]
        K2[blk, :, t % 16] ^= 0x11
        V2[blk, :, t % 16] ^= 0x22
    pert = oracle.prefill_attn(q, cu, K2, V2, st.block_tables, st.seq_lens, ks, vs, PER_TENSOR,
                               E4M3)
    first = 70 - (L - n)  # query rows before position 70
    np.testing.assert_array_equal(pert[:first], full[:first])
    assert not np.array_equal(pert[first:], full[first:])
    # a chunk of 40 = a chunk of 25 (cache length 75) then one of 15 (length 90)
    a = oracle.prefill_attn(q[:25], np.array([0, 25], np.int32), K, V, st.block_tables,
                            np.array([L - 15], np.int32), ks, vs, PER_TENSOR, E4M3)
    b = oracle.prefill_attn(q[25:], np.array([0, 15], np.int32), K, V, st.block_tables,
                            st.seq_lens, ks, vs, PER_TENSOR, E4M3)
    np.testing.assert_array_equal(np.concatenate([a, b]), full)


def test_more_queries_than_tokens_is_refused():
    r = np.random.default_rng(230)
    st, K, V, ks, vs = _case(r, [10], 2, 1, 64, E4M3, PER_TENSOR)
    q = bits(r.standard_normal((11, 2, 64)))
    with pytest.raises(ValueError):
        oracle.prefill_attn(q, np.array([0, 11], np.int32), K, V, st.block_tables, st.seq_lens,
                            ks, vs, PER_TENSOR, E4M3)


def test_block_permutation_invariance():
    """Moving the physical blocks (and the block tables with them) changes
    nothing: the queries see the cache only through the tables."""
    r = np.random.default_rng(240)
    lens, nq = [60, 35], [12, 35]
    st, K, V, ks, vs = _case(r, lens, 8, 2, 64, E4M3, PER_HEAD)
    q = bits(r.standard_normal((sum(nq), 8, 64)))
    cu = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    base = oracle.prefill_attn(q, cu, K, V, st.block_tables, st.seq_lens, ks, vs, PER_HEAD, E4M3)
    perm = r.permutation(st.num_blocks)          # new position of each block
    K2, V2 = np.empty_like(K), np.empty_like(V)
    K2[perm], V2[perm] = K, V
    bt = np.where(st.block_tables >= 0, perm[np.maximum(st.block_tables, 0)], -1).astype(np.int32)
    moved = oracle.prefill_attn(q, cu, K2, V2, bt, st.seq_lens, ks, vs, PER_HEAD, E4M3)
    np.testing.assert_array_equal(moved, base)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_uniform_v_gives_that_row(fmt):
    """With every cached V row equal, each query's output is that row's
    dequantized value whatever the logits (the weights sum to one)."""
    r = np.random.default_rng(250 + fmt)
    lens, nq = [50, 20], [30, 20]
    st, K, V, ks, vs = _case(r, lens, 4, 2, 64, fmt, PER_HEAD)
    row = V[st.block_tables[0, 0], :, 0, :].copy()   # [Hkv][dh] codes of token 0
    V[...] = row[None, :, None, :]
    q = bits(r.standard_normal((sum(nq), 4, 64)) * 4)
    cu = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    out = oracle.prefill_attn(q, cu, K, V, st.block_tables, st.seq_lens, ks, vs, PER_HEAD, fmt)
    want = oracle.decode(fmt, row) * vs.astype(np.float64)[:, None]   # [Hkv][dh]
    G = 2
    np.testing.assert_allclose(out, np.broadcast_to(np.repeat(want, G, 0)[None], out.shape),
                               rtol=1e-14, atol=0)
