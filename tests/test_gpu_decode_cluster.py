"""Parity of the per-segment cluster variant of the tensor-core decode.

Batches of few (sequence, KV head) segments with long block tables take the
variant in which one cluster of CTAs splits each segment's pages evenly and
merges the parts' softmax states in the leader CTA's shared memory.  These
cases pin it against the float64 oracle: every group size, both FP8 formats,
per-tensor and per-head scales, sliding windows, the FP8-domain query,
lengths that leave some CTAs of a cluster with no page, an empty sequence, a
masked-out block, and chains of cache-ready decodes.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from kvq_testlib import DeviceLayer, bf16_out_to_f64, check_attention, oracle_caches, oracle_decode
from test_gpu_parity import _custom_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    import fp8_quantized_paged_gb300 as m
    return m


def _run(lay, flags=0, seq_lens=None, q_fp8=False):
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    sl = None if seq_lens is None else torch.as_tensor(np.asarray(seq_lens, np.int32), device="cuda")
    ref = oracle_decode(lay, K, V, seq_lens=seq_lens, q_fp8=q_fp8)
    for _ in range(2):
        got = bf16_out_to_f64(d.decode(seq_lens=sl, flags=flags))
        assert d.status_word() == 0
        check_attention(got, ref, f"lens={lay.st.seq_lens.tolist()} G={lay.Hq // lay.Hkv}")
    return got


@pytest.mark.parametrize("lens,Hq,Hkv,fmt,gran", [
    ([20000], 32, 8, workloads.E4M3, workloads.PER_HEAD),
    ([32768], 32, 8, workloads.E5M2, workloads.PER_TENSOR),
    ([9000], 8, 8, workloads.E4M3, workloads.PER_HEAD),      # G = 1
    ([7001], 16, 8, workloads.E5M2, workloads.PER_HEAD),     # G = 2, ragged last page
    ([12345], 64, 8, workloads.E4M3, workloads.PER_HEAD),    # G = 8
    ([6000, 4500], 16, 4, workloads.E4M3, workloads.PER_HEAD),
    ([8000, 300], 32, 4, workloads.E4M3, workloads.PER_HEAD),  # a short segment: parts of 0-2 pages
    ([4096, 0], 16, 4, workloads.E4M3, workloads.PER_HEAD),    # an empty sequence
])
def test_cluster_decode(kvq, lens, Hq, Hkv, fmt, gran):
    lay = _custom_layer(lens, Hq=Hq, Hkv=Hkv, dh=128, fmt=fmt, gran=gran, seed=300 + len(lens) + Hq)
    got = _run(lay)
    for b, n in enumerate(lens):
        if n == 0:
            assert np.all(got[b] == 0)


@pytest.mark.parametrize("window", [1, 100, 4096])
def test_cluster_sliding_window(kvq, window):
    lay = _custom_layer([10000], Hq=32, Hkv=8, dh=128, seed=320, window=window)
    _run(lay)


def test_cluster_short_lengths_in_long_tables(kvq):
    """Block tables sized for 9000 tokens, lengths far shorter: most CTAs of a
    cluster get no page and contribute an empty state."""
    lay = _custom_layer([9000, 9000], Hq=32, Hkv=4, dh=128, seed=330)
    _run(lay, seq_lens=[37, 1])


def test_cluster_q_fp8(kvq):
    lay = _custom_layer([15000], Hq=32, Hkv=8, dh=128, seed=340)
    lay.q_scale[:] = np.linspace(0.005, 0.02, lay.q_scale.size).astype(np.float32)
    _run(lay, flags=kvq.KVQ_Q_FP8, q_fp8=True)


def test_cluster_bad_block(kvq):
    """An out-of-range block id: its page is skipped and reported, the output
    equals attention over the other tokens."""
    lay = _custom_layer([5000], Hq=32, Hkv=8, dh=128, seed=350)
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    bt = lay.st.block_tables.copy()
    bt[0, 100] = lay.st.num_blocks + 7  # tokens 1600..1615
    got = bf16_out_to_f64(d.decode(block_tables=torch.as_tensor(bt, device="cuda")))
    assert d.status_word() == kvq.KVQ_DEV_BAD_BLOCK
    keep = np.array([t for t in range(5000) if not 1600 <= t < 1616])
    st2 = workloads._structure(np.array([len(keep)]), np.random.default_rng(1))
    K2 = oracle.new_cache(st2.num_blocks, 8, 16, 128, lay.fmt)
    V2 = oracle.new_cache(st2.num_blocks, 8, 16, 128, lay.fmt)
    old = lay.st.block_tables[0, keep // 16].astype(np.int64) * 16 + keep % 16
    for i, s_old in enumerate(old):
        b_new, o_new = divmod(int(st2.slot_mapping[i]), 16)
        b_old, o_old = divmod(int(s_old), 16)
        K2[b_new, :, o_new] = K[b_old, :, o_old]
        V2[b_new, :, o_new] = V[b_old, :, o_old]
    ref = oracle.decode_attn(lay.q, K2, V2, st2.block_tables, st2.seq_lens, lay.k_scale,
                             lay.v_scale, lay.gran, lay.fmt)
    check_attention(got, ref, "bad page masked")


def test_cluster_cache_ready_chained(kvq):
    """Long single-sequence decodes of several layers back to back, each
    allowed to start before the previous one ends."""
    lays = [_custom_layer([16000], Hq=32, Hkv=8, dh=128, seed=360 + i) for i in range(3)]
    devs = [DeviceLayer(lay) for lay in lays]
    refs = []
    for d, lay in zip(devs, lays):
        d.write()
        K, V = oracle_caches(lay)
        refs.append(oracle_decode(lay, K, V))
    torch.cuda.synchronize()
    for _ in range(4):
        for d in devs:
            d.decode(flags=kvq.KVQ_CACHE_READY)
        for d, ref in zip(devs, refs):
            assert d.status_word() == 0
            check_attention(bf16_out_to_f64(d.out), ref, "chained cluster")
