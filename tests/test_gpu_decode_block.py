"""Decode parity on the shapes of long block tables and uneven batches
(FP8 caches, head size 128, four query heads per KV head).

Few (sequence, KV head group) segments split over every CTA, and batches in
which one long sequence is split over many CTAs while the others are not,
exercise the split-segment merges of whichever kernel serves the call (the
warp-MMA kernel by default; the whole-block tensor-core kernel when the
library is built with KVQ_DECODE_BLK, whose grid merge and staged last-piece
merge these shapes were written for).  The cases pin them against the
float64 oracle: both FP8 formats, per-tensor and per-head scales, two head
groups, sliding windows, the FP8-domain query, lengths that leave CTAs with
no page, empty sequences, a masked-out block, cache-ready chains, run-to-run
identity and a workspace full of NaN bytes outside its counters.
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


def _run(lay, flags=0, seq_lens=None, q_fp8=False, poison=False, reps=2):
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    sl = None if seq_lens is None else torch.as_tensor(np.asarray(seq_lens, np.int32), device="cuda")
    ref = oracle_decode(lay, K, V, seq_lens=seq_lens, q_fp8=q_fp8)
    first = None
    for _ in range(reps):
        if poison:
            d.poison_workspace()
        got = bf16_out_to_f64(d.decode(seq_lens=sl, flags=flags))
        assert d.status_word() == 0
        check_attention(got, ref, f"lens={lay.st.seq_lens.tolist()[:4]} Hkv={lay.Hkv}")
        if first is None:
            first = got.copy()
        else:  # a fixed merge order: the same bits every run
            np.testing.assert_array_equal(got, first)
    return got


# -------------------------------------------------------------- grid merge
@pytest.mark.parametrize("lens,Hq,Hkv,fmt,gran", [
    ([20000], 32, 8, workloads.E4M3, workloads.PER_HEAD),
    ([32768], 32, 8, workloads.E5M2, workloads.PER_TENSOR),
    ([6000, 4500], 32, 8, workloads.E4M3, workloads.PER_HEAD),
    ([3000, 2001, 0], 64, 16, workloads.E4M3, workloads.PER_HEAD),  # two head groups, an empty sequence
    ([4096, 0], 32, 8, workloads.E5M2, workloads.PER_HEAD),
    ([17], 32, 8, workloads.E4M3, workloads.PER_HEAD),  # two blocks: most CTAs have nothing
])
def test_grid_merge(kvq, lens, Hq, Hkv, fmt, gran):
    lay = _custom_layer(lens, Hq=Hq, Hkv=Hkv, dh=128, fmt=fmt, gran=gran, seed=300 + len(lens) + Hq)
    got = _run(lay, poison=True)
    for b, n in enumerate(lens):
        if n == 0:
            assert np.all(got[b] == 0)


@pytest.mark.parametrize("window", [1, 100, 4096])
def test_grid_sliding_window(kvq, window):
    lay = _custom_layer([10000], Hq=32, Hkv=8, dh=128, seed=320, window=window)
    _run(lay)


def test_grid_short_lengths_in_long_tables(kvq):
    """Block tables sized for 9000 tokens, lengths far shorter."""
    lay = _custom_layer([9000, 9000], Hq=32, Hkv=8, dh=128, seed=330)
    _run(lay, seq_lens=[37, 1])


def test_all_sequences_empty(kvq):
    lay = _custom_layer([300, 200], Hq=32, Hkv=8, dh=128, seed=331)
    got = _run(lay, seq_lens=[0, 0])
    assert np.all(got == 0)


# ------------------------------------------------- merge by the last piece
def _lens_last(long_len, n_short, short_len, seed):
    r = np.random.default_rng(seed)
    return [long_len] + [int(x) for x in r.integers(short_len // 2, short_len + 1, n_short)]


@pytest.mark.parametrize("lens,fmt,gran", [
    (_lens_last(16000, 19, 1600, 1), workloads.E4M3, workloads.PER_HEAD),   # ~50 pieces staged 8 at a time
    (_lens_last(3000, 39, 900, 2), workloads.E5M2, workloads.PER_TENSOR),   # a few pieces per segment
    (_lens_last(40000, 19, 16, 3), workloads.E4M3, workloads.PER_HEAD),     # too many pieces to stage
])
def test_last_merge(kvq, lens, fmt, gran):
    lay = _custom_layer(lens, Hq=32, Hkv=8, dh=128, fmt=fmt, gran=gran, seed=400 + len(lens))
    _run(lay, poison=True)


def test_last_merge_window_and_empty(kvq):
    lens = _lens_last(9000, 23, 2000, 4)
    lens[5] = 0
    lay = _custom_layer(lens, Hq=32, Hkv=8, dh=128, seed=410, window=700)
    got = _run(lay)
    assert np.all(got[5] == 0)


@pytest.mark.parametrize("lens", [[15000], _lens_last(6000, 25, 1500, 5)])
def test_q_fp8(kvq, lens):
    lay = _custom_layer(lens, Hq=32, Hkv=8, dh=128, seed=340)
    lay.q_scale[:] = np.linspace(0.005, 0.02, lay.q_scale.size).astype(np.float32)
    _run(lay, flags=kvq.KVQ_Q_FP8, q_fp8=True)


@pytest.mark.parametrize("lens", [[5000], _lens_last(5000, 25, 800, 6)])
def test_bad_block(kvq, lens):
    """An out-of-range block id: its eight heads' tokens are skipped and
    reported, the output equals attention over the other tokens."""
    lay = _custom_layer(lens, Hq=32, Hkv=8, dh=128, seed=350)
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    bt = lay.st.block_tables.copy()
    bt[0, 100] = lay.st.num_blocks + 7  # tokens 1600..1615 of sequence 0
    got = bf16_out_to_f64(d.decode(block_tables=torch.as_tensor(bt, device="cuda")))
    assert d.status_word() == kvq.KVQ_DEV_BAD_BLOCK
    # the reference: sequence 0 without those tokens, re-packed into fresh pages
    lens2 = list(lens)
    keep = np.array([t for t in range(lens[0]) if not 1600 <= t < 1616])
    lens2[0] = len(keep)
    st2 = workloads._structure(np.array(lens2), np.random.default_rng(1))
    K2 = oracle.new_cache(st2.num_blocks, 8, 16, 128, lay.fmt)
    V2 = oracle.new_cache(st2.num_blocks, 8, 16, 128, lay.fmt)
    for b, n in enumerate(lens):
        toks = keep if b == 0 else np.arange(n)
        old = lay.st.block_tables[b, toks // 16].astype(np.int64) * 16 + toks % 16
        for i, s_old in enumerate(old):
            b_new, o_new = divmod(int(st2.block_tables[b, i // 16]) * 16 + i % 16, 16)
            b_old, o_old = divmod(int(s_old), 16)
            K2[b_new, :, o_new] = K[b_old, :, o_old]
            V2[b_new, :, o_new] = V[b_old, :, o_old]
    ref = oracle.decode_attn(lay.q, K2, V2, st2.block_tables, st2.seq_lens, lay.k_scale,
                             lay.v_scale, lay.gran, lay.fmt)
    check_attention(got, ref, "bad block masked")


@pytest.mark.parametrize("lens", [[16000], _lens_last(4000, 25, 1200, 7)])
def test_cache_ready_chained(kvq, lens):
    """Decodes of several layers back to back, each allowed to start before
    the previous one ends."""
    lays = [_custom_layer(lens, Hq=32, Hkv=8, dh=128, seed=360 + i) for i in range(3)]
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
            check_attention(bf16_out_to_f64(d.out), ref, "chained")
