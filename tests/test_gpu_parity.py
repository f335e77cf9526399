"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Cache bytes must be bit-exact; attention outputs must satisfy
|gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise against the float64 oracle over
the same dequantized cache.  Inputs are the seeded workloads of
``workloads`` (the tiny case, the Llama-3.1-8B-shaped decode layer, per-head
scales in E4M3 and E5M2, one long-context layer, a FP8 and a bf16 layer of the
mixed skip-layer batch) plus hand-made edge cases.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
from kvq_testlib import (prefill_p_bound, DeviceLayer, bf16_out_to_f64, check_attention, oracle_caches,
                         oracle_decode, to_dev, to_np)

pytestmark = pytest.mark.gpu

CASES = [  # (config, layer, fmt for config 3)
    (1, 0, workloads.E4M3),
    (2, 0, workloads.E4M3),
    (3, 0, workloads.E4M3),
    (3, 0, workloads.E5M2),
    (4, 0, workloads.E4M3),
    (5, 2, workloads.E4M3),
    (5, 3, workloads.E4M3),  # bf16 + sliding window 4096
]
IDS = ["tiny", "llama8b_layer", "perhead_e4m3", "perhead_e5m2", "longctx_layer0",
       "mixed_fp8_layer2", "mixed_bf16_window_layer3"]


@pytest.fixture(scope="module")
def kvq():
    import fp8_quantized_paged_gb300 as m
    return m


def _pairs_for(lay):
    n = lay.B * lay.Hq
    if n * int(lay.st.seq_lens.max()) <= 32 * 1024 * 1024:
        return None  # every (sequence, head) pair
    return workloads.sample_pairs(lay.B, lay.Hq, 192, seed=lay.cfg * 100 + lay.layer)


@pytest.mark.parametrize("cfg,layer,fmt3", CASES, ids=IDS)
def test_write_and_decode(kvq, cfg, layer, fmt3):
    lay = workloads.make_layer(cfg, layer, fmt3)
    d = DeviceLayer(lay)
    if cfg == 2:
        new = np.flatnonzero(lay.new_token_mask)
        old = np.flatnonzero(~lay.new_token_mask)
        d.write(old)   # prefill
        d.write(new)   # the decode step's own tokens
    else:
        d.write()
    out = d.decode()
    assert d.status_word() == 0
    K, V = oracle_caches(lay)
    np.testing.assert_array_equal(to_np(d.kc), K)
    np.testing.assert_array_equal(to_np(d.vc), V)
    pairs = _pairs_for(lay)
    ref = oracle_decode(lay, K, V, pairs=pairs)
    got = bf16_out_to_f64(out)
    if pairs is not None:
        got = got[pairs[:, 0], pairs[:, 1]]
    check_attention(got, ref, f"config {cfg} layer {layer}")
    # deterministic: a second call gives the same bits
    first = to_np(out).copy()
    d.decode()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(d.out), first)


# ---------------------------------------------------------------- write edge cases

def _custom_layer(lens, Hq=8, Hkv=2, dh=64, fmt=workloads.E4M3, gran=workloads.PER_HEAD,
                  seed=0, std=1.0, window=0, spare=2):
    r = np.random.default_rng(seed)
    st = workloads._structure(np.array(lens), r, extra_blocks=spare)
    N = len(st.slot_mapping)
    f = lambda *s: workloads.f32_to_bf16_bits((r.standard_normal(s) * std).astype(np.float32))  # noqa
    q, k, v = f(len(lens), Hq, dh), f(N, Hkv, dh), f(N, Hkv, dh)
    nsc = Hkv if gran == workloads.PER_HEAD else 1
    ks = (r.uniform(0.5, 2.0, nsc) * std / 100).astype(np.float32)
    vs = (r.uniform(0.5, 2.0, nsc) * std / 100).astype(np.float32)
    if fmt == workloads.BF16:
        ks = vs = np.ones(nsc, np.float32)
    qs = np.ones(Hq if gran == workloads.PER_HEAD else 1, np.float32)
    return workloads.Layer(0, 0, len(lens), Hq, Hkv, dh, 16, fmt, gran, window, st, q, k, v, qs,
                           ks, vs)


@pytest.mark.parametrize("fmt", [workloads.E4M3, workloads.E5M2])
def test_write_special_values(kvq, fmt):
    """Signed zeros, subnormal FP8 results, midpoints, saturation and +-inf."""
    lay = _custom_layer([40, 9], fmt=fmt, gran=workloads.PER_TENSOR, seed=3)
    s = np.float32(0.01)
    lay.k_scale[:] = s
    lay.v_scale[:] = s
    mx = 448.0 if fmt == workloads.E4M3 else 57344.0
    specials = np.array([0.0, -0.0, 1e-30, -1e-30, 2.0 ** -9 * 0.01, 2.0 ** -10 * 0.01,
                         2.0 ** -16 * 0.01, mx * 0.01, mx * 0.0105, mx * 0.02, 1e30, -1e30,
                         np.inf, -np.inf, 3.0, -2.75], np.float32)
    bits = workloads.f32_to_bf16_bits(specials)
    flat = lay.k.reshape(-1)
    flat[: len(bits) * 40: 1] = np.resize(bits, len(bits) * 40)
    lay.v.reshape(-1)[::7] = bits[np.arange(lay.v.size // 7 + (lay.v.size % 7 > 0)) % len(bits)]
    d = DeviceLayer(lay)
    d.write()
    assert d.status_word() == 0
    K, V = oracle_caches(lay)
    np.testing.assert_array_equal(to_np(d.kc), K)
    np.testing.assert_array_equal(to_np(d.vc), V)


def _fp8_is_nan(codes, fmt):
    c = codes & 0x7F
    return c == 0x7F if fmt == workloads.E4M3 else c > 0x7C


@pytest.mark.parametrize("fmt", [workloads.E4M3, workloads.E5M2])
def test_write_extreme_scales(kvq, fmt):
    """Per-head scales across the whole binary32 range (both sides of the
    reciprocal method's [2^-80, 2^80] window, and zero) against inputs of
    every magnitude, infinities and signed zeros: codes equal the oracle's,
    NaN codes compared as NaN."""
    lay = _custom_layer([300, 77], Hq=8, Hkv=8, dh=64, fmt=fmt, seed=11)
    scales = np.array([2.0 ** -80, 1e-30, 1e-20, 0.01, 3e19, 2.0 ** 80, 2.0 ** 81, 0.0], np.float32)
    lay.k_scale[:] = scales
    lay.v_scale[:] = scales[::-1]
    r = np.random.default_rng(12)
    for arr in (lay.k, lay.v):
        x = (r.standard_normal(arr.shape) * 10.0 ** r.uniform(-42, 38, arr.shape)).astype(np.float32)
        arr[...] = workloads.f32_to_bf16_bits(x)
        flat = arr.reshape(-1)
        sp = workloads.f32_to_bf16_bits(np.array([0.0, -0.0, np.inf, -np.inf, 3.3895e38, -3.3895e38,
                                                   1e-40, -1e-40], np.float32))
        flat[r.choice(flat.size, 4000, replace=False)] = np.resize(sp, 4000)
    d = DeviceLayer(lay)
    d.write()
    assert d.status_word() == 0
    K, V = oracle_caches(lay)
    for got, want in ((to_np(d.kc), K), (to_np(d.vc), V)):
        gn, wn = _fp8_is_nan(got, fmt), _fp8_is_nan(want, fmt)
        np.testing.assert_array_equal(gn, wn)
        np.testing.assert_array_equal(np.where(gn, 0, got), np.where(wn, 0, want))


def test_write_nan_gives_a_nan_code(kvq):
    lay = _custom_layer([16], gran=workloads.PER_TENSOR, seed=4)
    lay.k[0, 0, :5] = workloads.f32_to_bf16_bits(np.array([np.nan] * 5, np.float32))
    lay.k[0, 0, 5] = 0xFFC0  # negative quiet NaN
    d = DeviceLayer(lay)
    d.write()
    codes = to_np(d.kc)[lay.st.block_tables[0, 0], 0, 0, :6]
    assert np.all(np.isnan(oracle.decode(workloads.E4M3, codes)))


def test_write_padding_bad_slot_and_fill(kvq):
    lay = _custom_layer([30, 20], seed=5)
    slots = lay.st.slot_mapping.copy()
    slots[3] = -1                                   # padding token: skipped
    slots[7] = lay.st.num_blocks * 16 + 5           # past the cache: flagged
    lay.st.slot_mapping = slots
    d = DeviceLayer(lay, fill=0x33)
    d.write()
    assert d.status_word() == kvq.KVQ_DEV_BAD_SLOT
    st = lay.st
    K = oracle.new_cache(st.num_blocks, lay.Hkv, 16, lay.dh, lay.fmt, 0x33)
    V = oracle.new_cache(st.num_blocks, lay.Hkv, 16, lay.dh, lay.fmt, 0x33)
    assert oracle.write(lay.k, lay.v, slots, K, V, lay.k_scale, lay.v_scale, lay.gran,
                        lay.fmt) == 1
    np.testing.assert_array_equal(to_np(d.kc), K)
    np.testing.assert_array_equal(to_np(d.vc), V)


def test_write_token_stride(kvq):
    """K and V read as slices of a fused per-token [q | k | v] row."""
    lay = _custom_layer([33, 17], Hq=8, Hkv=2, dh=128, seed=6)
    N = lay.k.shape[0]
    fused = np.zeros((N, (8 + 2 + 2) * 128), np.uint16)
    fused[:, 8 * 128:10 * 128] = lay.k.reshape(N, -1)
    fused[:, 10 * 128:] = lay.v.reshape(N, -1)
    d = DeviceLayer(lay)
    fz = to_dev(fused).view(N, 12, 128)
    kvq.kvq_write(fz[:, 8:10], fz[:, 10:12], d.slots, d.kc, d.vc, d.ks, d.vs, lay.gran,
                  lay.fmt, dev_status=d.status)
    K, V = oracle_caches(lay)
    np.testing.assert_array_equal(to_np(d.kc), K)
    np.testing.assert_array_equal(to_np(d.vc), V)


# ---------------------------------------------------------------- decode edge cases

@pytest.mark.parametrize("fmt", [workloads.E4M3, workloads.E5M2, workloads.BF16])
@pytest.mark.parametrize("dh", [64, 128])
def test_decode_ragged_lengths(kvq, fmt, dh):
    lens = [1, 15, 16, 17, 33, 0, 250, 5, 64, 1000]
    lay = _custom_layer(lens, Hq=16, Hkv=4, dh=dh, fmt=fmt, seed=7 + dh)
    d = DeviceLayer(lay)
    d.write()
    out = d.decode()
    assert d.status_word() == 0
    K, V = oracle_caches(lay)
    ref = oracle_decode(lay, K, V)
    got = bf16_out_to_f64(out)
    check_attention(got, ref, "ragged")
    assert np.all(got[5] == 0)  # empty sequence -> zero row


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_decode_group_sizes(kvq, G):
    lay = _custom_layer([70, 300, 16], Hq=2 * G, Hkv=2, dh=128, seed=20 + G)
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    check_attention(bf16_out_to_f64(d.decode()), oracle_decode(lay, K, V), f"G={G}")


@pytest.mark.parametrize("window", [1, 7, 16, 100, 512, 5000])
def test_decode_sliding_window(kvq, window):
    lay = _custom_layer([600, 16, 1, 129], Hq=8, Hkv=2, dh=128, fmt=workloads.BF16, seed=30,
                        window=window)
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    check_attention(bf16_out_to_f64(d.decode()), oracle_decode(lay, K, V), f"window={window}")
    # FP8 layers accept a window too
    lay8 = _custom_layer([600, 40], Hq=8, Hkv=2, dh=128, seed=31, window=window)
    d8 = DeviceLayer(lay8)
    d8.write()
    K8, V8 = oracle_caches(lay8)
    check_attention(bf16_out_to_f64(d8.decode()), oracle_decode(lay8, K8, V8), "fp8 window")


def test_decode_uniform_v_and_one_token(kvq):
    lay = _custom_layer([300, 1, 45], Hq=8, Hkv=2, dh=128, seed=40)
    lay.v[:] = lay.v[0]  # every token carries the same V row
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    vhat = oracle.decode(lay.fmt, V[lay.st.block_tables[0, 0], :, 0, :]) * lay.v_scale[:, None]
    got = bf16_out_to_f64(d.decode())
    for h in range(8):
        check_attention(got[:, h, :], np.broadcast_to(vhat[h // 4], (3, 128)), "uniform V")


def test_decode_large_logits(kvq):
    """Logit spread far beyond the lazy-rescale threshold (K std 30)."""
    lay = _custom_layer([2000, 700], Hq=8, Hkv=2, dh=128, seed=41, std=30.0)
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    check_attention(bf16_out_to_f64(d.decode()), oracle_decode(lay, K, V), "large logits")


def test_decode_bad_block_and_seq_len(kvq):
    lay = _custom_layer([64, 40, 20], Hq=8, Hkv=2, dh=128, seed=42)
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    ref = oracle_decode(lay, K, V)
    bt = lay.st.block_tables.copy()
    bt[1, 1] = lay.st.num_blocks + 3  # sequence 1, tokens 16..31
    sl = lay.st.seq_lens.copy()
    sl[2] = bt.shape[1] * 16 + 1      # longer than its block table
    out = bf16_out_to_f64(d.decode(block_tables=to_dev(bt), seq_lens=to_dev(sl)))
    assert d.status_word() == kvq.KVQ_DEV_BAD_BLOCK | kvq.KVQ_DEV_BAD_SEQLEN
    check_attention(out[0], ref[0], "untouched sequence")
    assert np.all(out[2] == 0)
    # sequence 1 equals attention over its tokens outside the bad page
    keep = [t for t in range(40) if not 16 <= t < 32]
    sub = workloads.Layer(0, 0, 1, 8, 2, 128, 16, lay.fmt, lay.gran, 0,
                          workloads._structure(np.array([len(keep)]), np.random.default_rng(0)),
                          lay.q[1:2], None, None, lay.q_scale, lay.k_scale, lay.v_scale)
    pos = np.array(keep)
    blk = lay.st.block_tables[1, pos // 16] * 16 + pos % 16
    K2 = oracle.new_cache(sub.st.num_blocks, 2, 16, 128, lay.fmt)
    V2 = oracle.new_cache(sub.st.num_blocks, 2, 16, 128, lay.fmt)
    slot2 = sub.st.slot_mapping
    for i, s_old in enumerate(blk):
        b_new, o_new = divmod(int(slot2[i]), 16)
        b_old, o_old = divmod(int(s_old), 16)
        K2[b_new, :, o_new] = K[b_old, :, o_old]
        V2[b_new, :, o_new] = V[b_old, :, o_old]
    ref1 = oracle.decode_attn(sub.q, K2, V2, sub.st.block_tables, sub.st.seq_lens, lay.k_scale,
                              lay.v_scale, lay.gran, lay.fmt)
    check_attention(out[1], ref1[0], "bad page masked")


def test_decode_single_piece_segments(kvq):
    """Tiny grids where one CTA holds a whole (sequence, head) segment and the
    decode kernel writes the output itself (no reduce)."""
    for lens in ([16], [16, 16], [5], [3, 16, 9]):
        lay = _custom_layer(lens, Hq=8, Hkv=2, dh=128, seed=50 + len(lens))
        d = DeviceLayer(lay)
        d.write()
        K, V = oracle_caches(lay)
        check_attention(bf16_out_to_f64(d.decode()), oracle_decode(lay, K, V), f"lens={lens}")


def test_workspace_too_small(kvq):
    lay = _custom_layer([20], seed=60)
    d = DeviceLayer(lay)
    d.write()
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_decode_attn(d.q, d.kc, d.vc, d.bt, d.sl, None, d.ks, d.vs, lay.gran, lay.fmt, 0,
                            small, d.out)
    assert e.value.status == kvq.KVQ_ERR_WORKSPACE


# ---------------------------------------------------------------- unfused ablation

@pytest.mark.parametrize("cfg,fmt3", [(2, workloads.E4M3), (3, workloads.E5M2)])
def test_dequant_then_bf16_decode(kvq, cfg, fmt3):
    lay = workloads.make_layer(cfg, 0, fmt3)
    d = DeviceLayer(lay)
    d.write()
    kb = torch.empty(d.kc.shape, dtype=torch.bfloat16, device="cuda")
    vb = torch.empty(d.vc.shape, dtype=torch.bfloat16, device="cuda")
    kvq.kvq_dequant_cache(d.kc, kb, d.ks, lay.gran, lay.fmt)
    kvq.kvq_dequant_cache(d.vc, vb, d.vs, lay.gran, lay.fmt)
    K, V = oracle_caches(lay)
    Kb = oracle.dequant(K, lay.k_scale, lay.gran, lay.fmt)
    Vb = oracle.dequant(V, lay.v_scale, lay.gran, lay.fmt)
    np.testing.assert_array_equal(to_np(kb), Kb)
    np.testing.assert_array_equal(to_np(vb), Vb)
    kvq.kvq_decode_attn(d.q, kb, vb, d.bt, d.sl, None, None, None, 0, kvq.KVQ_FMT_BF16, 0, d.ws,
                        d.out)
    pairs = workloads.sample_pairs(lay.B, lay.Hq, 128, seed=cfg)
    ref = oracle.decode_attn(lay.q, Kb, Vb, lay.st.block_tables, lay.st.seq_lens, None, None, 0,
                             oracle.BF16, pairs=pairs)
    got = bf16_out_to_f64(d.out)[pairs[:, 0], pairs[:, 1]]
    check_attention(got, ref, "unfused bf16 path")


@pytest.mark.parametrize("lens", [[70, 33, 1], [500, 300], [16] * 7, [1] * 40, [1] * 300 + [5000],
                                  [0, 3, 0, 40000, 2, 0, 17]])
@pytest.mark.parametrize("fmt", [workloads.E4M3, workloads.BF16])
def test_decode_fewer_units_than_ctas(kvq, lens, fmt):
    """Batches with fewer KV pages than the persistent grid has CTAs: segments
    split over consecutive CTAs and the reduce must read only written slots
    (the workspace starts as NaN bytes)."""
    lay = _custom_layer(lens, Hq=8, Hkv=2, dh=128, fmt=fmt, seed=70 + len(lens))
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    for _ in range(3):
        got = bf16_out_to_f64(d.decode())
        assert d.status_word() == 0
        check_attention(got, oracle_decode(lay, K, V), f"lens={lens}")
        d.poison_workspace()


@pytest.mark.parametrize("lens,Hq,Hkv,dh,fmt", [
    ([6000], 1, 1, 64, workloads.E4M3),        # one segment over every CTA
    ([9000], 8, 1, 128, workloads.BF16),       # pieces too large to stage in shared memory
    ([20000], 32, 8, 128, workloads.E4M3),     # long-context shape: 8 segments, ~38 pieces each
    ([7000, 3], 16, 4, 64, workloads.E5M2),
    ([12000], 16, 8, 128, workloads.BF16),
    ([3000] * 4, 32, 8, 128, workloads.E4M3),  # ~10 pieces per segment
    ([1500] * 8, 32, 8, 128, workloads.E4M3),  # ~5 pieces per segment
    ([2500] * 3, 8, 4, 64, workloads.E5M2),
])
def test_decode_segments_split_over_many_ctas(kvq, lens, Hq, Hkv, dh, fmt):
    """Segments cut into many pieces: the CTA finishing a segment's last piece
    merges up to one partial state per CTA, from shared memory when they fit
    its idle ring, else from global memory."""
    lay = _custom_layer(lens, Hq=Hq, Hkv=Hkv, dh=dh, fmt=fmt, seed=90 + Hq + dh)
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    ref = oracle_decode(lay, K, V)
    for _ in range(2):
        got = bf16_out_to_f64(d.decode())
        assert d.status_word() == 0
        check_attention(got, ref, f"lens={lens} G={Hq // Hkv} dh={dh}")
        d.poison_workspace()


@pytest.mark.parametrize("fmt", [workloads.E4M3, workloads.BF16])
def test_decode_cache_ready_after_new_token_write(kvq, fmt):
    """KVQ_CACHE_READY: the decode may start while the kvq_write of each
    sequence's newest token still runs; it reads the older pages early and
    the newest token's page only after that write."""
    lens = [2048, 700, 33, 1, 16, 17, 4000, 129]
    lay = _custom_layer(lens, Hq=32, Hkv=8, dh=128, fmt=fmt, seed=130 + fmt)
    last = np.cumsum(lens) - 1
    older = np.setdiff1d(np.arange(int(np.sum(lens))), last)
    d = DeviceLayer(lay)
    K, V = oracle_caches(lay)
    ref = oracle_decode(lay, K, V)
    for _ in range(3):
        d.kc.zero_()
        d.vc.zero_()
        d.write(older)
        torch.cuda.synchronize()
        d.write(last)  # the preceding kernel writes only the newest token of each sequence
        got = bf16_out_to_f64(d.decode(flags=kvq.KVQ_CACHE_READY))
        assert d.status_word() == 0
        check_attention(got, ref, "cache ready after write")


def test_decode_cache_ready_chained_layers(kvq):
    """Decodes of different layers back to back, each allowed to start early."""
    lays = [_custom_layer([5000, 300, 64], Hq=32, Hkv=8, dh=128, seed=140 + i) for i in range(3)]
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


# ---------------------------------------------------------------- scale calibration

def _calib(kvq, k, v, gran, fmt, hkv, stride=None, status=None):
    n = hkv if gran == workloads.PER_HEAD else 1
    ks = torch.full((n,), float("nan"), device="cuda")
    vs = torch.full((n,), float("nan"), device="cuda")
    kvq.kvq_calibrate_scales(k, v, ks, vs, gran, fmt, dev_status=status, token_stride=stride)
    return to_np(ks), to_np(vs)


@pytest.mark.parametrize("cfg,layer,fmt", [(2, 0, workloads.E4M3), (3, 1, workloads.E4M3),
                                           (3, 1, workloads.E5M2), (1, 0, workloads.E4M3)])
@pytest.mark.parametrize("gran", [workloads.PER_TENSOR, workloads.PER_HEAD])
def test_calibrate_matches_oracle(kvq, cfg, layer, fmt, gran):
    lay = workloads.make_layer(cfg, layer)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ks, vs = _calib(kvq, to_dev(lay.k), to_dev(lay.v), gran, fmt, lay.Hkv, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    np.testing.assert_array_equal(ks, oracle.calibrate(lay.k, gran, fmt))
    np.testing.assert_array_equal(vs, oracle.calibrate(lay.v, gran, fmt))


def test_calibrate_specials_stride_and_empty(kvq):
    r = np.random.default_rng(21)
    n, hkv, dh = 300, 4, 64
    x = (r.standard_normal((n, hkv, dh)) * 3).astype(np.float32)
    x[5, 1, 3] = np.nan
    x[7, 2, 9] = np.inf
    x[8, 2, 10] = -np.inf
    x[:, 3, :] = 0.0          # an all-zero head -> scale 1
    x[11, 0, 0] = -250.0      # a negative maximum
    b = workloads.f32_to_bf16_bits(x)
    wide = np.zeros((n, hkv * dh + 64), np.uint16)  # token stride beyond Hkv * dh
    wide[:, : hkv * dh] = b.reshape(n, -1)
    kd = to_dev(wide)
    k = kd[:, : hkv * dh].view(n, hkv, dh)
    ks, vs = _calib(kvq, k, k, workloads.PER_HEAD, workloads.E4M3, hkv, stride=hkv * dh + 64)
    want = oracle.calibrate(b, workloads.PER_HEAD, workloads.E4M3)
    np.testing.assert_array_equal(ks, want)
    np.testing.assert_array_equal(vs, want)
    assert want[3] == 1.0 and want[0] == np.float32(250) / np.float32(448)
    e = torch.empty((0, hkv, dh), dtype=torch.bfloat16, device="cuda")
    ks, vs = _calib(kvq, e, e, workloads.PER_TENSOR, workloads.E5M2, hkv)
    assert ks[0] == 1.0 and vs[0] == 1.0


def test_calibrate_then_write_uses_the_full_range(kvq):
    """Scales from the calibration put every head's largest value on the
    format's largest finite code and nothing beyond it."""
    lay = workloads.make_layer(3, 0)
    d = DeviceLayer(lay)
    assert lay.gran == workloads.PER_HEAD
    ks, vs = _calib(kvq, d.k, d.v, workloads.PER_HEAD, lay.fmt, lay.Hkv)
    d.ks.copy_(torch.from_numpy(ks))
    d.vs.copy_(torch.from_numpy(vs))
    d.write()
    assert d.status_word() == 0
    top = 0x7E if lay.fmt == workloads.E4M3 else 0x7B
    for cache in (d.kc, d.vc):
        codes = to_np(cache)
        per_head_max = (codes & 0x7F).transpose(1, 0, 2, 3).reshape(lay.Hkv, -1).max(axis=1)
        np.testing.assert_array_equal(per_head_max, np.full(lay.Hkv, top))


# ---------------------------------------------------------------- FP8-domain query mode

def _q_fp8_layer(lay, scale=None):
    """The layer with q_scale set from the query's own amax (per tensor or per
    query head, as the layer's granularity), or to ``scale``."""
    qs = oracle.calibrate(lay.q, lay.gran, lay.fmt) if scale is None else scale
    return dataclasses.replace(lay, q_scale=np.asarray(qs, np.float32))


@pytest.mark.parametrize("cfg,layer,fmt3", [(1, 0, workloads.E4M3), (2, 0, workloads.E4M3),
                                           (3, 0, workloads.E4M3), (3, 0, workloads.E5M2),
                                           (5, 2, workloads.E4M3)],
                         ids=["tiny", "llama8b_layer", "perhead_e4m3", "perhead_e5m2",
                              "mixed_fp8_layer2"])
def test_decode_q_fp8(kvq, cfg, layer, fmt3):
    """Q quantized to the cache format with the workload's q scale, QK^T on
    FP8 codes: same output as the oracle's dec(enc(q / sQ)) sQ query."""
    lay = workloads.make_layer(cfg, layer, fmt3)
    d = DeviceLayer(lay)
    d.write()
    out = d.decode(flags=kvq.KVQ_Q_FP8)
    assert d.status_word() == 0
    K, V = oracle_caches(lay)
    pairs = _pairs_for(lay)
    ref = oracle_decode(lay, K, V, pairs=pairs, q_fp8=True)
    got = bf16_out_to_f64(out)
    if pairs is not None:
        got = got[pairs[:, 0], pairs[:, 1]]
    check_attention(got, ref, f"q fp8 config {cfg} layer {layer}")


@pytest.mark.parametrize("fmt", [workloads.E4M3, workloads.E5M2])
@pytest.mark.parametrize("G,dh", [(1, 128), (2, 64), (4, 128), (8, 64), (8, 128)])
@pytest.mark.parametrize("gran", [workloads.PER_TENSOR, workloads.PER_HEAD])
def test_decode_q_fp8_shapes(kvq, fmt, G, dh, gran):
    lay = _q_fp8_layer(_custom_layer([1, 15, 0, 250, 33, 1000], Hq=2 * G, Hkv=2, dh=dh, fmt=fmt,
                                     gran=gran, seed=110 + G + dh))
    d = DeviceLayer(lay)
    d.write()
    got = bf16_out_to_f64(d.decode(flags=kvq.KVQ_Q_FP8))
    assert d.status_word() == 0
    K, V = oracle_caches(lay)
    check_attention(got, oracle_decode(lay, K, V, q_fp8=True), f"q fp8 G={G} dh={dh}")
    assert np.all(got[2] == 0)


def test_decode_q_fp8_saturating_and_split(kvq):
    """A q scale small enough that most query codes saturate to the format's
    largest finite value, on segments split over many CTAs, with the
    cache-ready flag."""
    lay = _q_fp8_layer(_custom_layer([20000, 3], Hq=32, Hkv=8, dh=128, seed=120),
                       scale=np.full(32, 1.0 / 1024, np.float32))
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    ref = oracle_decode(lay, K, V, q_fp8=True)
    for flags in (kvq.KVQ_Q_FP8, kvq.KVQ_Q_FP8 | kvq.KVQ_CACHE_READY):
        got = bf16_out_to_f64(d.decode(flags=flags))
        assert d.status_word() == 0
        check_attention(got, ref, f"q fp8 saturating flags={flags}")
        d.poison_workspace()


def test_decode_q_fp8_rejected_without_fp8_cache_or_scale(kvq):
    lay = _custom_layer([40], Hq=4, Hkv=2, dh=64, fmt=workloads.BF16)
    d = DeviceLayer(lay)
    with pytest.raises(RuntimeError):
        d.decode(flags=kvq.KVQ_Q_FP8)
    lay8 = _custom_layer([40], Hq=4, Hkv=2, dh=64)
    d8 = DeviceLayer(lay8)
    d8.qs = None
    with pytest.raises(RuntimeError):
        d8.decode(flags=kvq.KVQ_Q_FP8)


# ---------------------------------------------------------------- per-(token, KV head) scales

def _f32_bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def _check_token_head_caches(d, K, V, sK, sV):
    np.testing.assert_array_equal(to_np(d.kc), K)
    np.testing.assert_array_equal(to_np(d.vc), V)
    np.testing.assert_array_equal(_f32_bits(to_np(d.ksc)), _f32_bits(sK))
    np.testing.assert_array_equal(_f32_bits(to_np(d.vsc)), _f32_bits(sV))


@pytest.mark.parametrize("cfg,layer,fmt3", [(1, 0, workloads.E4M3), (2, 0, workloads.E4M3),
                                           (3, 0, workloads.E4M3), (3, 0, workloads.E5M2),
                                           (5, 2, workloads.E4M3)],
                         ids=["tiny", "llama8b_layer", "perhead_e4m3", "perhead_e5m2",
                              "mixed_fp8_layer2"])
def test_token_head_write_and_decode(kvq, cfg, layer, fmt3):
    """Each row's scale from its own amax, stored beside the page; the decode
    reads the row scales: caches and scales bit-exact, attention within
    tolerance, in both query modes."""
    lay = workloads.make_layer(cfg, layer, fmt3)
    d = DeviceLayer(lay, token_head=True)
    if cfg == 2:
        new = np.flatnonzero(lay.new_token_mask)
        d.write(np.flatnonzero(~lay.new_token_mask))
        d.write(new)
    else:
        d.write()
    out = bf16_out_to_f64(d.decode())
    assert d.status_word() == 0
    K, V, sK, sV = oracle_caches(lay, token_head=True)
    _check_token_head_caches(d, K, V, sK, sV)
    pairs = _pairs_for(lay)
    ref = oracle_decode(lay, K, V, pairs=pairs, scale_caches=(sK, sV))
    got = out if pairs is None else out[pairs[:, 0], pairs[:, 1]]
    check_attention(got, ref, f"token-head config {cfg}")
    qf = bf16_out_to_f64(d.decode(flags=kvq.KVQ_Q_FP8))
    assert d.status_word() == 0
    ref8 = oracle_decode(lay, K, V, pairs=pairs, scale_caches=(sK, sV), q_fp8=True)
    check_attention(qf if pairs is None else qf[pairs[:, 0], pairs[:, 1]], ref8,
                    f"token-head q fp8 config {cfg}")


@pytest.mark.parametrize("fmt", [workloads.E4M3, workloads.E5M2])
def test_token_head_special_rows(kvq, fmt):
    """Rows of zeros, NaN / inf among finite values, subnormal-only rows, rows
    at the bf16 range's top (scales outside the fast division's range) and
    rows whose magnitudes span the whole format."""
    lay = _custom_layer([40, 17], Hq=4, Hkv=2, dh=128, fmt=fmt, seed=130)
    k = lay.k.copy()
    one = lambda x: workloads.f32_to_bf16_bits(np.asarray(x, np.float32))  # noqa: E731
    k[0] = 0                                        # zero rows -> scale 1
    k[1, 0, :3] = one([np.nan, np.inf, -np.inf])    # specials ignored by amax
    k[2, 1, :] = np.arange(1, 129, dtype=np.uint16)  # bf16 subnormals only
    k[3, 0, :] = one(np.linspace(-3e38, 3e38, 128))  # huge: s > 2^80
    k[4, 1, :] = one(np.geomspace(1e-30, 1e30, 128))
    k[5, :, :] = 0x8000                              # -0 everywhere
    lay = dataclasses.replace(lay, k=k)
    d = DeviceLayer(lay, token_head=True)
    d.write()
    assert d.status_word() == 0
    K, V, sK, sV = oracle_caches(lay, token_head=True)
    nan_k = np.isnan(oracle.decode(fmt, K))
    np.testing.assert_array_equal(np.isnan(oracle.decode(fmt, to_np(d.kc))), nan_k)
    np.testing.assert_array_equal(np.where(nan_k, 0, to_np(d.kc)), np.where(nan_k, 0, K))
    np.testing.assert_array_equal(to_np(d.vc), V)
    np.testing.assert_array_equal(_f32_bits(to_np(d.ksc)), _f32_bits(sK))
    np.testing.assert_array_equal(_f32_bits(to_np(d.vsc)), _f32_bits(sV))


@pytest.mark.parametrize("fmt", [workloads.E4M3, workloads.E5M2])
@pytest.mark.parametrize("G,dh", [(1, 64), (2, 128), (4, 64), (8, 128)])
def test_token_head_shapes(kvq, fmt, G, dh):
    """Ragged lengths (an empty sequence, partial last pages whose unwritten
    rows hold NaN scales), widely varying row magnitudes."""
    lay = _custom_layer([1, 15, 0, 250, 33, 1000], Hq=2 * G, Hkv=2, dh=dh, fmt=fmt,
                        seed=140 + G + dh)
    r = np.random.default_rng(141 + G)
    mag = 10.0 ** r.uniform(-3, 3, (lay.k.shape[0], 2, 1))
    kf = (lay.k.astype(np.uint32) << 16).view(np.float32) * mag
    vf = (lay.v.astype(np.uint32) << 16).view(np.float32) / mag
    lay = dataclasses.replace(lay, k=workloads.f32_to_bf16_bits(kf.astype(np.float32)),
                              v=workloads.f32_to_bf16_bits(vf.astype(np.float32)))
    d = DeviceLayer(lay, token_head=True)
    d.write()
    got = bf16_out_to_f64(d.decode())
    assert d.status_word() == 0
    K, V, sK, sV = oracle_caches(lay, token_head=True)
    _check_token_head_caches(d, K, V, sK, sV)
    check_attention(got, oracle_decode(lay, K, V, scale_caches=(sK, sV)), f"token-head G={G}")
    assert np.all(got[2] == 0)


@pytest.mark.parametrize("lens,Hq,Hkv,dh,fmt,window", [
    ([20000, 3], 32, 8, 128, workloads.E4M3, 0),
    ([3000] * 4, 32, 8, 128, workloads.E5M2, 0),
    ([7000, 40], 16, 4, 64, workloads.E4M3, 1000),
])
def test_token_head_split_segments_and_cache_ready(kvq, lens, Hq, Hkv, dh, fmt, window):
    lay = _custom_layer(lens, Hq=Hq, Hkv=Hkv, dh=dh, fmt=fmt, seed=150 + dh, window=window)
    d = DeviceLayer(lay, token_head=True)
    d.write()
    K, V, sK, sV = oracle_caches(lay, token_head=True)
    ref = oracle_decode(lay, K, V, scale_caches=(sK, sV))
    for flags in (0, kvq.KVQ_CACHE_READY):
        got = bf16_out_to_f64(d.decode(flags=flags))
        assert d.status_word() == 0
        check_attention(got, ref, f"token-head lens={lens} flags={flags}")
        d.poison_workspace()


@pytest.mark.parametrize("fmt", [workloads.E4M3, workloads.E5M2])
def test_token_head_dequant_then_bf16_decode(kvq, fmt):
    lay = _custom_layer([300, 77], Hq=8, Hkv=2, dh=128, fmt=fmt, seed=160)
    d = DeviceLayer(lay, token_head=True)
    d.write()
    K, V, sK, sV = oracle_caches(lay, token_head=True)
    kb = torch.empty(d.kc.shape, dtype=torch.bfloat16, device="cuda")
    kvq.kvq_dequant_cache(d.kc, kb, d.ksc, kvq.KVQ_SCALE_PER_TOKEN_HEAD, fmt)
    torch.cuda.synchronize()
    # rows nobody wrote hold NaN scales: compare the written rows
    want = oracle.dequant(K, sK, oracle.PER_TOKEN_HEAD, fmt)
    written = ~np.isnan(sK)
    np.testing.assert_array_equal(to_np(kb)[written], want[written])


# ---------------------------------------------------------------- prefill / prefix-hit attention

def _prefill_case(kvq, lay, nq, seed, window=None, repeats=1):
    """Write the layer's tokens, then attend with the last nq[b] tokens of each
    sequence as queries; returns (gpu float64 [total_q][Hq][dh], oracle inputs).
    With repeats > 1 the call runs again and must give the same bits."""
    r = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = workloads.f32_to_bf16_bits(r.standard_normal((int(cu[-1]), lay.Hq, lay.dh)).astype(np.float32))
    d = DeviceLayer(lay)
    d.write()
    out = torch.empty((int(cu[-1]), lay.Hq, lay.dh), dtype=torch.bfloat16, device="cuda")
    out.fill_(float("nan"))
    win = lay.window if window is None else window
    qd, cud = to_dev(q), to_dev(cu)
    first = None
    for _ in range(repeats):
        kvq.kvq_prefill_attn(qd, cud, int(max(nq)) if len(nq) else 0, d.kc, d.vc, d.bt, d.sl, d.ks,
                             d.vs, lay.gran, lay.fmt, win, out, dev_status=d.status)
        assert d.status_word() == 0
        bits = to_np(out).copy()
        if first is not None:
            np.testing.assert_array_equal(bits, first)  # deterministic: no race in the pipeline
        first = bits
    return bf16_out_to_f64(out), q, cu, win


def _prefill_ref(lay, q, cu, win, pairs=None):
    K, V = oracle_caches(lay)
    st = lay.st
    return oracle.prefill_attn(q, cu, K, V, st.block_tables, st.seq_lens, lay.k_scale,
                               lay.v_scale, lay.gran, lay.fmt, window=win, pairs=pairs)


@pytest.mark.parametrize("fmt", [workloads.E4M3, workloads.E5M2, workloads.BF16])
@pytest.mark.parametrize("G,dh", [(1, 64), (2, 128), (4, 128), (8, 64)])
def test_prefill_full_and_prefix_hit(kvq, fmt, G, dh):
    """Whole-sequence prefills, prefix hits of a few tokens and a single
    query (the decode) in one ragged batch."""
    lens = [70, 33, 300, 16, 129]
    nq = [70, 5, 37, 1, 0]
    lay = _custom_layer(lens, Hq=2 * G, Hkv=2, dh=dh, fmt=fmt, seed=170 + G + dh)
    got, q, cu, win = _prefill_case(kvq, lay, nq, seed=171)
    check_attention(got, _prefill_ref(lay, q, cu, win), f"prefill G={G} dh={dh}")


@pytest.mark.parametrize("window", [1, 16, 100, 1000])
def test_prefill_sliding_window(kvq, window):
    lay = _custom_layer([600, 40], Hq=8, Hkv=2, dh=128, seed=180)
    got, q, cu, win = _prefill_case(kvq, lay, [150, 40], seed=181, window=window)
    check_attention(got, _prefill_ref(lay, q, cu, win), f"prefill window={window}")
    layb = _custom_layer([600, 40], Hq=8, Hkv=2, dh=128, fmt=workloads.BF16, seed=182)
    got, q, cu, win = _prefill_case(kvq, layb, [100, 3], seed=183, window=window)
    check_attention(got, _prefill_ref(layb, q, cu, win), f"bf16 prefill window={window}")


def test_prefill_one_query_matches_decode(kvq):
    lay = _custom_layer([300, 1, 45, 1000], Hq=32, Hkv=8, dh=128, seed=190)
    got, q, cu, win = _prefill_case(kvq, lay, [1, 1, 1, 1], seed=191)
    lay_q = dataclasses.replace(lay, q=q)
    K, V = oracle_caches(lay)
    check_attention(got, oracle_decode(lay_q, K, V), "prefill n=1 vs decode")


@pytest.mark.parametrize("cfg,layer,fmt3,nq", [
    (2, 0, workloads.E4M3, 64),    # Llama-3.1-8B-shaped layer: 64-token prefix hits
    (3, 0, workloads.E5M2, 200),   # per-head scales, long prefixes
    (5, 2, workloads.E4M3, 16),    # mixed batch FP8 layer
    (5, 3, workloads.E4M3, 16),    # mixed batch bf16 layer with window 4096
])
def test_prefill_workloads(kvq, cfg, layer, fmt3, nq):
    """The workloads' caches with each sequence's last nq tokens as queries
    (all of them when shorter), on sampled (row, head) pairs."""
    lay = workloads.make_layer(cfg, layer, fmt3)
    lens = lay.st.seq_lens
    n = np.minimum(lens, nq).astype(np.int64)
    got, q, cu, win = _prefill_case(kvq, lay, list(n), seed=200 + cfg, repeats=3)
    r = np.random.default_rng(201)
    rows = r.integers(0, int(cu[-1]), 256)
    heads = r.integers(0, lay.Hq, 256)
    pairs = np.stack([rows, heads], 1).astype(np.int32)
    ref = _prefill_ref(lay, q, cu, win, pairs=pairs)
    check_attention(got[rows, heads], ref, f"prefill workload {cfg}")


def test_prefill_bad_lengths_and_empty(kvq):
    """A sequence with fewer cached tokens than queries gets zero rows and
    the length flag; the others are unaffected."""
    lay = _custom_layer([50, 40], Hq=4, Hkv=2, dh=64, seed=210)
    r = np.random.default_rng(211)
    cu = np.array([0, 10, 60], np.int32)  # sequence 1 asks for 50 queries of 40 tokens
    q = workloads.f32_to_bf16_bits(r.standard_normal((60, 4, 64)).astype(np.float32))
    d = DeviceLayer(lay)
    d.write()
    out = torch.full((60, 4, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    kvq.kvq_prefill_attn(to_dev(q), to_dev(cu), 50, d.kc, d.vc, d.bt, d.sl, d.ks, d.vs, lay.gran,
                         lay.fmt, 0, out, dev_status=d.status)
    assert d.status_word() & kvq.KVQ_DEV_BAD_SEQLEN
    got = bf16_out_to_f64(out)
    assert np.all(got[10:] == 0)
    K, V = oracle_caches(lay)
    ref = oracle.prefill_attn(q[:10], cu[:2], K, V, lay.st.block_tables[:1], lay.st.seq_lens[:1],
                              lay.k_scale, lay.v_scale, lay.gran, lay.fmt)
    check_attention(got[:10], ref, "prefill valid sequence")


@pytest.mark.parametrize("shift", [17, 40, -30])
@pytest.mark.parametrize("G,dh,fmt", [(4, 64, workloads.E4M3), (8, 128, workloads.E5M2),
                                      (2, 128, workloads.E4M3)])
def test_decode_query_outside_f16_range(kvq, shift, G, dh, fmt):
    """The query times 2^shift and the K scales times 2^-shift: the logits, and
    so the attention, are unchanged, but |q| lies beyond f16's largest value
    (shift 17, 40) or below its smallest normal (shift -30).  The FP8 decode
    scales each head's query by a power of two before its f16 conversion."""
    lay = _custom_layer([300, 77], Hq=2 * G, Hkv=2, dh=dh, fmt=fmt, seed=60 + G)
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    f = np.float32(2.0 ** shift)
    lay.q[:] = workloads.f32_to_bf16_bits(workloads.bf16_bits_to_f32(lay.q) * f)  # exact
    lay.k_scale[:] = (lay.k_scale / f).astype(np.float32)                        # exact
    d.q.copy_(to_dev(lay.q))
    d.ks.copy_(to_dev(lay.k_scale))
    got = bf16_out_to_f64(d.decode())
    assert d.status_word() == 0
    check_attention(got, oracle_decode(lay, K, V), f"q x 2^{shift}")


def test_prefill_chunk_longer_than_max_q_len(kvq):
    """max_q_len below a chunk's length: the grid covers fewer rows than the
    chunk has; the status says so, and the rows it covers are right."""
    lay = _custom_layer([300, 40], Hq=8, Hkv=2, dh=128, seed=215)
    r = np.random.default_rng(216)
    cu = np.array([0, 200, 210], np.int32)
    q = workloads.f32_to_bf16_bits(r.standard_normal((210, 8, 128)).astype(np.float32))
    d = DeviceLayer(lay)
    d.write()
    out = torch.full((210, 8, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    kvq.kvq_prefill_attn(to_dev(q), to_dev(cu), 10, d.kc, d.vc, d.bt, d.sl, d.ks, d.vs, lay.gran,
                         lay.fmt, 0, out, dev_status=d.status)
    assert d.status_word() & kvq.KVQ_DEV_BAD_QLEN
    got = bf16_out_to_f64(out)
    K, V = oracle_caches(lay)
    ref = oracle.prefill_attn(q, cu, K, V, lay.st.block_tables, lay.st.seq_lens, lay.k_scale,
                              lay.v_scale, lay.gran, lay.fmt)
    check_attention(got[200:], ref[200:], "the short chunk")
    check_attention(got[:10], ref[:10], "the long chunk's first rows")
    # with max_q_len covering every chunk: no flag
    d.status.zero_()
    kvq.kvq_prefill_attn(to_dev(q), to_dev(cu), 200, d.kc, d.vc, d.bt, d.sl, d.ks, d.vs, lay.gran,
                         lay.fmt, 0, out, dev_status=d.status)
    assert d.status_word() == 0
    check_attention(bf16_out_to_f64(out), ref, "covered")


# ---------------------------------------------------------------- prefill with per-(token, head)
# scales and the FP8-domain query

def _prefill_ex(kvq, lay, nq, seed, token_head=False, q_fp8=False, window=None):
    """Prefill with the last nq[b] tokens of each sequence as queries, over a
    cache written per tensor / per head, or per (token, head) with its scale
    caches; optionally the FP8-domain query (q_scale = lay.q_scale).  Returns
    (gpu float64, float64 oracle)."""
    r = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = workloads.f32_to_bf16_bits(r.standard_normal((int(cu[-1]), lay.Hq, lay.dh)).astype(np.float32))
    d = DeviceLayer(lay, token_head=token_head)
    d.write()
    out = torch.full((int(cu[-1]), lay.Hq, lay.dh), float("nan"), dtype=torch.bfloat16, device="cuda")
    win = lay.window if window is None else window
    ks, vs = (d.ksc, d.vsc) if token_head else (d.ks, d.vs)
    gran = kvq.KVQ_SCALE_PER_TOKEN_HEAD if token_head else lay.gran
    kvq.kvq_prefill_attn(to_dev(q), to_dev(cu), int(max(nq)), d.kc, d.vc, d.bt, d.sl, ks, vs, gran,
                         lay.fmt, win, out, dev_status=d.status,
                         q_scale=d.qs if q_fp8 else None, flags=kvq.KVQ_Q_FP8 if q_fp8 else 0)
    status = d.status_word()
    if token_head:
        K, V, sK, sV = oracle_caches(lay, token_head=True)
        ksr, vsr, granr = sK, sV, oracle.PER_TOKEN_HEAD
    else:
        K, V = oracle_caches(lay)
        ksr, vsr, granr = lay.k_scale, lay.v_scale, lay.gran
    ref = oracle.prefill_attn(q, cu, K, V, lay.st.block_tables, lay.st.seq_lens, ksr, vsr,
                              granr, lay.fmt, window=win,
                              q_scale=lay.q_scale if q_fp8 else None)
    return bf16_out_to_f64(out), ref, status


def _check_prefill(got, ref, lay, nq, what):
    """The attention tolerance plus the f16 probabilities' term (large |V|
    rows, as with per-token magnitudes over two decades, reach it)."""
    cu = np.concatenate([[0], np.cumsum(nq)])
    check_attention(got, ref, what, extra=prefill_p_bound(lay, cu))


def _per_token_magnitudes(lay, seed):
    """K and V rows scaled by factors log-uniform over 10^[-1, 1], so the
    per-(token, head) scales span two decades inside every key block (the
    probabilities reach the PV MMA as f16, within 2^-12 of their value: the
    output's error bound grows with the largest |V| a row attends to)."""
    r = np.random.default_rng(seed)
    for x in (lay.k, lay.v):
        f = 10.0 ** r.uniform(-1.0, 1.0, size=x.shape[:2] + (1,))
        x[:] = workloads.f32_to_bf16_bits((workloads.bf16_bits_to_f32(x) * f).astype(np.float32))


@pytest.mark.parametrize("fmt", [workloads.E4M3, workloads.E5M2])
@pytest.mark.parametrize("G,dh", [(1, 64), (2, 128), (4, 128), (8, 64)])
def test_prefill_token_head_scales(kvq, fmt, G, dh):
    """A prefix hit, a whole prefill and a single query over a cache written
    by kvq_write_token_head, with per-token magnitudes spanning two decades."""
    lay = _custom_layer([70, 33, 300, 16, 129], Hq=2 * G, Hkv=2, dh=dh, fmt=fmt, seed=230 + G + dh)
    _per_token_magnitudes(lay, 231)
    got, ref, st = _prefill_ex(kvq, lay, [70, 5, 37, 1, 0], seed=232, token_head=True)
    assert st == 0
    _check_prefill(got, ref, lay, [70, 5, 37, 1, 0], f"token-head prefill G={G} dh={dh}")


@pytest.mark.parametrize("mode", ["per_head", "token_head", "window", "q_fp8", "e5m2_dh64"])
def test_prefill_tile_pairs(kvq, mode):
    """Enough query tiles that the FP8 prefill runs two tiles a CTA (16
    sequences x 2 tiles of 128 rows x 8 KV heads: 256 single-tile CTAs are
    two waves on a GB300, 128 pairs one), with chunks that fill both tiles,
    part of the second, or only the first."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    waves = lambda ctas: -(-ctas // sms)  # noqa: E731
    assert 8 * waves(1 * 8 * 16) < 7 * waves(2 * 8 * 16), "the launch would not pair tiles"
    r = np.random.default_rng(270)
    nq = [256, 200, 129, 128, 64, 1, 256, 256, 130, 255, 17, 256, 192, 256, 100, 256]
    lens = [q + int(r.integers(0, 300)) for q in nq]
    fmt = workloads.E5M2 if mode == "e5m2_dh64" else workloads.E4M3
    dh = 64 if mode == "e5m2_dh64" else 128
    lay = _custom_layer(lens, Hq=8, Hkv=8, dh=dh, fmt=fmt, seed=271)
    if mode == "q_fp8":
        lay.q_scale[:] = np.linspace(0.005, 0.02, lay.q_scale.size).astype(np.float32)
    if mode == "token_head":
        _per_token_magnitudes(lay, 272)
    got, ref, st = _prefill_ex(kvq, lay, nq, seed=273, token_head=mode == "token_head",
                               q_fp8=mode == "q_fp8", window=100 if mode == "window" else None)
    assert st == 0
    _check_prefill(got, ref, lay, nq, f"prefill in tile pairs ({mode})")


@pytest.mark.parametrize("token_head", [False, True])
@pytest.mark.parametrize("gran", [workloads.PER_TENSOR, workloads.PER_HEAD])
def test_prefill_q_fp8(kvq, token_head, gran):
    lay = _custom_layer([300, 70, 129], Hq=32, Hkv=8, dh=128, gran=gran, seed=240)
    lay.q_scale[:] = np.linspace(0.005, 0.02, lay.q_scale.size).astype(np.float32)
    got, ref, st = _prefill_ex(kvq, lay, [64, 70, 1], seed=241, token_head=token_head, q_fp8=True)
    assert st == 0
    _check_prefill(got, ref, lay, [64, 70, 1], f"q fp8 prefill token_head={token_head}")


@pytest.mark.parametrize("window", [1, 100])
def test_prefill_token_head_window_and_bad_block(kvq, window):
    lay = _custom_layer([600, 40], Hq=8, Hkv=2, dh=128, seed=250)
    _per_token_magnitudes(lay, 251)
    got, ref, st = _prefill_ex(kvq, lay, [150, 40], seed=252, token_head=True, window=window)
    assert st == 0
    _check_prefill(got, ref, lay, [150, 40], f"token-head prefill window={window}")
    # an out-of-range block id in the prefix: its 16 tokens are masked out;
    # the reference re-packs the other tokens (the queries keep their order)
    bt = lay.st.block_tables.copy()
    bt[0, 20] = lay.st.num_blocks + 3
    r = np.random.default_rng(253)
    cu = np.array([0, 150, 190], np.int32)
    q = workloads.f32_to_bf16_bits(r.standard_normal((190, 8, 128)).astype(np.float32))
    d = DeviceLayer(lay, token_head=True)
    d.write()
    out = torch.full((190, 8, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    kvq.kvq_prefill_attn(to_dev(q), to_dev(cu), 150, d.kc, d.vc, to_dev(bt), d.sl, d.ksc, d.vsc,
                         kvq.KVQ_SCALE_PER_TOKEN_HEAD, lay.fmt, 0, out, dev_status=d.status)
    assert d.status_word() == kvq.KVQ_DEV_BAD_BLOCK
    K, V, sK, sV = oracle_caches(lay, token_head=True)
    lens = lay.st.seq_lens
    keep = [np.array([t for t in range(lens[0]) if not 320 <= t < 336]), np.arange(lens[1])]
    st2 = workloads._structure(np.array([len(k) for k in keep]), np.random.default_rng(254))
    K2 = oracle.new_cache(st2.num_blocks, 2, 16, 128, lay.fmt)
    V2 = oracle.new_cache(st2.num_blocks, 2, 16, 128, lay.fmt)
    sK2 = np.zeros((st2.num_blocks, 2, 16), np.float32)
    sV2 = np.zeros_like(sK2)
    for b, toks in enumerate(keep):
        for i, t in enumerate(toks):
            bo, oo = int(lay.st.block_tables[b, t // 16]), t % 16
            bn, on = int(st2.block_tables[b, i // 16]), i % 16
            K2[bn, :, on], V2[bn, :, on] = K[bo, :, oo], V[bo, :, oo]
            sK2[bn, :, on], sV2[bn, :, on] = sK[bo, :, oo], sV[bo, :, oo]
    ref = oracle.prefill_attn(q, cu, K2, V2, st2.block_tables, st2.seq_lens, sK2, sV2,
                              oracle.PER_TOKEN_HEAD, lay.fmt)
    check_attention(bf16_out_to_f64(out), ref, "token-head prefill, masked block")


def test_prefill_one_query_matches_decode_token_head_and_q_fp8(kvq):
    """n_b = 1 queries over a per-(token, head) cache with the FP8-domain query:
    the prefill's rows equal the decode's (both against the oracle)."""
    lay = _custom_layer([300, 1, 45, 1000], Hq=32, Hkv=8, dh=128, seed=260)
    lay.q_scale[:] = np.linspace(0.01, 0.03, lay.q_scale.size).astype(np.float32)
    got, ref, st = _prefill_ex(kvq, lay, [1, 1, 1, 1], seed=261, token_head=True, q_fp8=True)
    assert st == 0
    check_attention(got, ref, "prefill n=1, token-head, q fp8")
