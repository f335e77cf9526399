"""Seeded synthetic inputs for the FP8 paged KV-cache path.

This module only draws inputs: lengths, block tables, slot mappings, bf16
Q/K/V values and the calibration-style scales (amax / format maximum) that
stand in for offline calibration.  It holds none of the method's arithmetic
(no FP8 encoding, no attention) and imports neither the oracle nor the CUDA
library, so both sides of a parity test can take their inputs from here.

The five workloads:
  1 tiny: B=2, L=[100, 37], Hq=8, Hkv=2, dh=64, bs=16, one layer, N(0,1),
    scales 1.0, E4M3 per tensor; block table = a random permutation of the
    10 physical blocks.
  2 Llama-3.1-8B-shaped decode layer: B=32, 2048 cached tokens + 1 new token
    each, Hq=32, Hkv=8, dh=128; N(0,1) with 4 seeded outlier channels per KV
    head scaled x10 in K; per-tensor k/v scale amax/448; E4M3.
  3 per-head scales: B=64, L ~ U[512, 8192]; per-KV-head std log-uniform in
    [0.1, 10] for K and V separately; per-head scales amax/448 (E4M3) or
    amax/57344 (E5M2).
  4 long context: B=1, L=32768, 32 layers of independent N(0,1) K/V,
    per-head E4M3 scales.
  5 mixed skip-layer batch: B=128, L = round(LogNormal(ln 2048, 1)) clipped to
    [1, 16384], 32 layers; layers with i % 4 == 3 are sliding-window (4096)
    layers kept in bf16, the rest FP8 E4M3 per head.

Values are drawn in float32 and rounded to bf16 (round to nearest even).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BF16, E4M3, E5M2 = 0, 1, 2
PER_TENSOR, PER_HEAD = 0, 1
FMT_MAX = {E4M3: np.float32(448.0), E5M2: np.float32(57344.0)}
BLOCK_SIZE = 16

# random streams per (config, layer)
_S_STRUCT, _S_Q, _S_K, _S_V, _S_AUX = 0, 1, 2, 3, 4


def rng(config_seed: int, layer: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([config_seed, layer, stream])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 samples to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Structure:
    """Sequence lengths and the paged layout shared by every layer of a workload."""
    seq_lens: np.ndarray      # int32 [B]; includes the token decoded this step
    block_tables: np.ndarray  # int32 [B][max_blocks_per_seq]; unused entries -1
    num_blocks: int
    slot_mapping: np.ndarray  # int64 [N]; token order: seq 0 positions 0.., seq 1 ...
    token_seq: np.ndarray     # int32 [N] sequence of each token
    token_pos: np.ndarray     # int32 [N] position of each token in its sequence


@dataclasses.dataclass
class Layer:
    """One attention layer's inputs."""
    cfg: int
    layer: int
    B: int
    Hq: int
    Hkv: int
    dh: int
    bs: int
    fmt: int
    gran: int
    window: int
    st: Structure
    q: np.ndarray        # bf16 bits [B][Hq][dh]
    k: np.ndarray        # bf16 bits [N][Hkv][dh]  (all tokens of all sequences)
    v: np.ndarray        # bf16 bits [N][Hkv][dh]
    q_scale: np.ndarray  # float32 [1] or [Hq]
    k_scale: np.ndarray  # float32 [1] or [Hkv]
    v_scale: np.ndarray  # float32 [1] or [Hkv]

    @property
    def new_token_mask(self) -> np.ndarray:
        """Tokens decoded this step: the last position of every sequence."""
        return self.st.token_pos == (self.st.seq_lens[self.st.token_seq] - 1)


def _structure(seq_lens: np.ndarray, r: np.random.Generator, bs: int = BLOCK_SIZE,
               extra_blocks: int = 0) -> Structure:
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    nblk = (seq_lens.astype(np.int64) + bs - 1) // bs
    num_blocks = int(nblk.sum()) + extra_blocks
    perm = r.permutation(num_blocks).astype(np.int32)
    max_blocks = int(nblk.max()) if len(nblk) else 1
    bt = np.full((len(seq_lens), max(max_blocks, 1)), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[off:off + n]
        off += int(n)
    N = int(seq_lens.astype(np.int64).sum())
    token_seq = np.repeat(np.arange(len(seq_lens), dtype=np.int32), seq_lens)
    starts = np.concatenate([[0], np.cumsum(seq_lens.astype(np.int64))[:-1]])
    token_pos = (np.arange(N, dtype=np.int64) - np.repeat(starts, seq_lens)).astype(np.int32)
    blk = bt[token_seq, token_pos // bs].astype(np.int64)
    slot = blk * bs + (token_pos % bs)
    return Structure(seq_lens, bt, num_blocks, slot.astype(np.int64), token_seq, token_pos)


def _amax_scale(bits: np.ndarray, fmt: int, axis=None) -> np.ndarray:
    a = np.abs(bf16_bits_to_f32(bits))
    amax = a.max(axis=axis) if axis is not None else np.array([a.max()])
    return (amax.astype(np.float32) / FMT_MAX[fmt]).astype(np.float32).reshape(-1)


def _normal_bits(r: np.random.Generator, shape, std=None) -> np.ndarray:
    x = r.standard_normal(size=shape, dtype=np.float32)
    if std is not None:
        x *= std
    return f32_to_bf16_bits(x)


# --------------------------------------------------------------------------

NUM_LAYERS = {1: 1, 2: 1, 3: 1, 4: 32, 5: 32}
SHAPES = {  # (Hq, Hkv, dh)
    1: (8, 2, 64), 2: (32, 8, 128), 3: (32, 8, 128), 4: (32, 8, 128), 5: (32, 8, 128)}
DESCRIPTION = {
    1: "tiny: B=2 L=[100,37] Hq=8 Hkv=2 dh=64 bs=16 E4M3 per-tensor scale 1.0",
    2: "llama3.1-8b decode layer: B=32 L=2048+1 Hq=32 Hkv=8 dh=128 E4M3 per-tensor amax/448",
    3: "per-head scales: B=64 L~U[512,8192] Hq=32 Hkv=8 dh=128 per-head amax/fmt_max",
    4: "long context: B=1 L=32768 32 layers Hq=32 Hkv=8 dh=128 E4M3 per-head",
    5: "mixed skip layers: B=128 L~LogNormal(ln2048,1) clip[1,16384] 32 layers, "
       "i%4==3 bf16 window 4096, else E4M3 per-head",
}


def structure(cfg: int) -> Structure:
    r = rng(cfg, 0, _S_STRUCT)
    if cfg == 1:
        lens = np.array([100, 37])
    elif cfg == 2:
        lens = np.full(32, 2049)
    elif cfg == 3:
        lens = r.integers(512, 8192, size=64, endpoint=True)
    elif cfg == 4:
        lens = np.array([32768])
    elif cfg == 5:
        x = r.normal(loc=math.log(2048.0), scale=1.0, size=128)
        lens = np.clip(np.rint(np.exp(x)), 1, 16384).astype(np.int64)
    else:
        raise ValueError(cfg)
    return _structure(lens, r)


def layer_format(cfg: int, layer: int, fmt3: int = E4M3):
    """(fmt, granularity, window) of one layer of a workload."""
    if cfg == 1:
        return E4M3, PER_TENSOR, 0
    if cfg == 2:
        return E4M3, PER_TENSOR, 0
    if cfg == 3:
        return fmt3, PER_HEAD, 0
    if cfg == 4:
        return E4M3, PER_HEAD, 0
    if cfg == 5:
        return (BF16, PER_HEAD, 4096) if layer % 4 == 3 else (E4M3, PER_HEAD, 0)
    raise ValueError(cfg)


def make_layer(cfg: int, layer: int = 0, fmt3: int = E4M3, st: Structure | None = None) -> Layer:
    """Inputs of one layer of workload `cfg` (config 3 takes E4M3 or E5M2 via fmt3)."""
    Hq, Hkv, dh = SHAPES[cfg]
    st = st if st is not None else structure(cfg)
    B = len(st.seq_lens)
    N = len(st.slot_mapping)
    fmt, gran, window = layer_format(cfg, layer, fmt3)
    q = _normal_bits(rng(cfg, layer, _S_Q), (B, Hq, dh))
    if cfg == 2:
        ra = rng(cfg, layer, _S_AUX)
        kf = rng(cfg, layer, _S_K).standard_normal(size=(N, Hkv, dh), dtype=np.float32)
        for h in range(Hkv):
            ch = ra.choice(dh, size=4, replace=False)
            kf[:, h, ch] *= np.float32(10.0)
        k = f32_to_bf16_bits(kf)
        del kf
        v = _normal_bits(rng(cfg, layer, _S_V), (N, Hkv, dh))
    elif cfg == 3:
        ra = rng(cfg, layer, _S_AUX)
        sk = np.exp(ra.uniform(math.log(0.1), math.log(10.0), size=Hkv)).astype(np.float32)
        sv = np.exp(ra.uniform(math.log(0.1), math.log(10.0), size=Hkv)).astype(np.float32)
        k = _normal_bits(rng(cfg, layer, _S_K), (N, Hkv, dh), std=sk[None, :, None])
        v = _normal_bits(rng(cfg, layer, _S_V), (N, Hkv, dh), std=sv[None, :, None])
    else:
        k = _normal_bits(rng(cfg, layer, _S_K), (N, Hkv, dh))
        v = _normal_bits(rng(cfg, layer, _S_V), (N, Hkv, dh))

    if fmt == BF16:
        one = np.ones(1, np.float32)
        qs, ks, vs = one, one, one
        if gran == PER_HEAD:
            qs, ks, vs = np.ones(Hq, np.float32), np.ones(Hkv, np.float32), np.ones(Hkv, np.float32)
    elif cfg == 1:
        qs = ks = vs = np.ones(1, np.float32)
    elif gran == PER_TENSOR:
        qs, ks, vs = _amax_scale(q, fmt), _amax_scale(k, fmt), _amax_scale(v, fmt)
    else:
        qs = _amax_scale(q, fmt, axis=(0, 2))
        ks = _amax_scale(k, fmt, axis=(0, 2))
        vs = _amax_scale(v, fmt, axis=(0, 2))
    return Layer(cfg, layer, B, Hq, Hkv, dh, BLOCK_SIZE, fmt, gran, window, st, q, k, v,
                 qs, ks, vs)


def sample_pairs(B: int, Hq: int, n: int, seed: int) -> np.ndarray:
    """A seeded sample of (sequence, query head) pairs for full-size spot checks."""
    r = rng(seed, 999, _S_AUX)
    idx = r.choice(B * Hq, size=min(n, B * Hq), replace=False)
    return np.stack([idx // Hq, idx % Hq], axis=1).astype(np.int32)
