"""CPU oracle for the FP8 paged KV-cache path (test infrastructure).

This package is TEST INFRASTRUCTURE.  Only the test suite, the smoke check
in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import
it.  The product library never loads it, and it never loads the product: the
two share no code.  The arithmetic lives in ``kvq_oracle.c`` (plain C,
float64 attention, bit-level FP8 codec); this module compiles it with gcc and
wraps it with ctypes over numpy arrays.

Sources (page titles and sections):
  * "10.4 KV Cache quantization: INT8, KIVI 2-bit, FP8 KV", sections 10.4.1
    (KV size formula), 10.4.2 (write / read / attention over the dequantized
    cache), 10.4.3 (per-token scales and their metadata bytes), 10.4.5 (FP8
    path: cast_fp8(K/sK) then cast_float(K_fp8) * sK).
  * "vLLM FP8 quantized KV cache guide": scale shapes [1] (per tensor) and
    [num_kv_heads] (per attention head), ``fp8`` as an alias of ``fp8_e4m3``,
    uint8 storage with FP8 bit semantics; scale calibration, way two (scales
    from statistics of the K/V activations; here their absolute maximum).

Every function here is pinned by tests in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

BF16, E4M3, E5M2 = 0, 1, 2
PER_TENSOR, PER_HEAD, PER_TOKEN_HEAD = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkvq_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable C11, no CPU-specific flags)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            L.kvqo_encode.argtypes = [i32, ctypes.c_float]
            L.kvqo_encode.restype = ctypes.c_uint8
            L.kvqo_decode.argtypes = [i32, ctypes.c_uint8]
            L.kvqo_decode.restype = ctypes.c_double
            L.kvqo_f32_to_bf16.argtypes = [ctypes.c_float]
            L.kvqo_f32_to_bf16.restype = ctypes.c_uint16
            L.kvqo_encode_f32_array.argtypes = [i32, vp, vp, i64]
            L.kvqo_decode_array.argtypes = [i32, vp, vp, i64]
            L.kvqo_quantize_bf16_array.argtypes = [i32, vp, ctypes.c_float, vp, i64]
            L.kvqo_write.argtypes = [vp, vp, i64, vp, i64, i32, i32, vp, vp, i64, i32, vp, vp,
                                     i32, i32, i32]
            L.kvqo_write.restype = i64
            L.kvqo_write_token_head.argtypes = [vp, vp, i64, vp, i64, i32, i32, vp, vp, i64,
                                                i32, vp, vp, i32, i32]
            L.kvqo_write_token_head.restype = i64
            L.kvqo_decode_attn.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i64, i32,
                                           vp, vp, i32, i32, vp, i32, i32, vp, i64, vp, i32]
            L.kvqo_decode_attn.restype = i64
            L.kvqo_prefill_attn.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i64,
                                            i32, vp, vp, i32, i32, vp, i32, i32, vp, i64, vp, i32]
            L.kvqo_prefill_attn.restype = i64
            L.kvqo_dequant.argtypes = [vp, vp, i64, i32, i32, i32, vp, i32, i32]
            L.kvqo_max_threads.restype = i32
            _lib = L
    return _lib


# --------------------------------------------------------------------------
# Codec
# --------------------------------------------------------------------------

def encode(fmt: int, x) -> np.ndarray:
    """FP8 codes (uint8) of binary32 values: RNE, satfinite, signed zero kept."""
    x = np.asarray(x, dtype=np.float32)
    shape = x.shape
    x = np.ascontiguousarray(x).reshape(-1)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().kvqo_encode_f32_array(fmt, _p(x), _p(out), x.size)
    return out.reshape(shape)


def decode(fmt: int, codes) -> np.ndarray:
    """Exact float64 values of FP8 codes (NaN codes give NaN, E5M2 inf gives inf)."""
    c = np.asarray(codes, dtype=np.uint8)
    shape = c.shape
    c = np.ascontiguousarray(c).reshape(-1)
    out = np.empty(c.shape, dtype=np.float64)
    lib().kvqo_decode_array(fmt, _p(c), _p(out), c.size)
    return out.reshape(shape)


def quantize_bf16(fmt: int, x_bf16_bits, scale: float) -> np.ndarray:
    """cast_fp8(x / s): binary32 quotient of a bf16 input, then FP8 RNE-satfinite."""
    x = np.asarray(x_bf16_bits, dtype=np.uint16)
    shape = x.shape
    x = np.ascontiguousarray(x).reshape(-1)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().kvqo_quantize_bf16_array(fmt, _p(x), ctypes.c_float(scale), _p(out), x.size)
    return out.reshape(shape)


def f32_to_bf16(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib().kvqo_f32_to_bf16(float(v)) for v in x], dtype=np.uint16)


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# KV size formula (section 10.4.1)
# --------------------------------------------------------------------------

def kv_bytes(layers: int, batch: int, kv_heads: int, seq: int, head_dim: int,
             bytes_per_element: float, scale_bytes_per_row: float = 0) -> float:
    """M_KV = 2 * L * B * Hkv * S * dh * bytes (2 = K and V; Hkv, not Hq),
    plus, with per-(token, head) scales (section 10.4.3), the scale bytes of
    each K row and each V row."""
    return 2 * layers * batch * kv_heads * seq * (head_dim * bytes_per_element + scale_bytes_per_row)


# --------------------------------------------------------------------------
# Write / decode / dequant
# --------------------------------------------------------------------------

def _cache_dtype(fmt):
    return np.uint16 if fmt == BF16 else np.uint8


def new_cache(num_blocks, num_kv_heads, block_size, head_dim, fmt, fill=0):
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    return np.full(shape, fill, dtype=_cache_dtype(fmt))


def new_scale_cache(num_blocks, num_kv_heads, block_size, fill=0.0):
    """Per-(token, KV head) scales beside the pages: float32 [blocks][Hkv][bs]."""
    return np.full((num_blocks, num_kv_heads, block_size), fill, dtype=np.float32)


def write(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, granularity, fmt,
          token_stride=None, nthreads=0) -> int:
    """Quantize-and-scatter (in place on k_cache / v_cache). Returns bad-slot count.

    With ``granularity == PER_TOKEN_HEAD`` k_scale / v_scale are the scale
    caches (float32 [blocks][Hkv][bs], from ``new_scale_cache``): every
    written row's scale amax / fmt_max (1 if 0) is stored there, in place."""
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    n, hkv, dh = k.shape
    stride = hkv * dh if token_stride is None else token_stride
    slot = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    if granularity == PER_TOKEN_HEAD:
        nb, hkv2, bs, dh2 = k_cache.shape
        assert fmt in (E4M3, E5M2) and hkv2 == hkv and dh2 == dh
        for a in (k_scale, v_scale):
            assert a.dtype == np.float32 and a.shape == (nb, hkv, bs) and a.flags.c_contiguous
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
        return int(lib().kvqo_write_token_head(_p(k), _p(v), stride, _p(slot), n, hkv, dh,
                                               _p(k_cache), _p(v_cache), nb, bs, _p(k_scale),
                                               _p(v_scale), fmt, nthreads))
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    nb, hkv2, bs, dh2 = k_cache.shape
    assert hkv2 == hkv and dh2 == dh and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    assert k_cache.dtype == _cache_dtype(fmt) and v_cache.dtype == _cache_dtype(fmt)
    return int(lib().kvqo_write(_p(k), _p(v), stride, _p(slot), n, hkv, dh, _p(k_cache),
                                _p(v_cache), nb, bs, _p(ks), _p(vs), granularity, fmt, nthreads))


def decode_attn(q, k_cache, v_cache, block_tables, seq_lens, k_scale, v_scale, granularity,
                fmt, window=0, pairs=None, nthreads=0, q_scale=None) -> np.ndarray:
    """Float64 decode attention over the dequantized paged cache.

    q: bf16 bits [B][Hq][dh]. Returns float64 [B][Hq][dh], or [len(pairs)][dh]
    when ``pairs`` (int array [n][2] of (b, h)) is given.  With ``q_scale``
    ([1] or [Hq] fp32) the query is first quantized to the cache's FP8 format
    and restored, dec(enc(fp32(q) / sQ)) * sQ (the FP8-domain mode).
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    B, hq, dh = q.shape
    nb, hkv, bs, dh2 = k_cache.shape
    assert dh2 == dh
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    ks = np.ascontiguousarray(k_scale if k_scale is not None else [1.0], dtype=np.float32)
    vs = np.ascontiguousarray(v_scale if v_scale is not None else [1.0], dtype=np.float32)
    if pairs is None:
        out = np.empty((B, hq, dh), dtype=np.float64)
        pr, npairs = None, 0
    else:
        pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        npairs = pr.shape[0]
        out = np.empty((npairs, dh), dtype=np.float64)
    qs = None if q_scale is None else np.ascontiguousarray(q_scale, dtype=np.float32).reshape(-1)
    if qs is not None and qs.size not in (1, hq):
        raise ValueError("q_scale must have 1 or num_q_heads entries")
    bad = lib().kvqo_decode_attn(_p(q), _p(np.ascontiguousarray(k_cache)),
                                 _p(np.ascontiguousarray(v_cache)), _p(bt), bt.shape[1], _p(sl),
                                 B, hq, hkv, dh, nb, bs, _p(ks), _p(vs), granularity, fmt,
                                 _p(qs), 0 if qs is None else int(qs.size == hq and hq > 1),
                                 window, _p(pr), npairs, _p(out), nthreads)
    if bad:
        raise ValueError(f"oracle decode: {bad} (sequence, head) pairs had out-of-range inputs")
    return out


def prefill_attn(q, cu_q, k_cache, v_cache, block_tables, seq_lens, k_scale, v_scale,
                 granularity, fmt, window=0, pairs=None, nthreads=0, q_scale=None) -> np.ndarray:
    """Float64 prefill / prefix-hit attention over the dequantized paged cache.

    q: bf16 bits [total_q][Hq][dh]; cu_q int [B+1] query row offsets.  The
    n_b = cu_q[b+1] - cu_q[b] queries of sequence b are its last n_b tokens
    (positions L_b - n_b .. L_b - 1, L_b = seq_lens[b]); each attends causally
    to the cached tokens up to its own position.  Returns float64
    [total_q][Hq][dh], or [len(pairs)][dh] for pairs of (query row, head)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    total_q, hq, dh = q.shape
    cu = np.ascontiguousarray(cu_q, dtype=np.int32)
    B = cu.size - 1
    assert cu[0] == 0 and cu[-1] == total_q
    nb, hkv, bs, dh2 = k_cache.shape
    assert dh2 == dh
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    ks = np.ascontiguousarray(k_scale if k_scale is not None else [1.0], dtype=np.float32)
    vs = np.ascontiguousarray(v_scale if v_scale is not None else [1.0], dtype=np.float32)
    if pairs is None:
        out = np.empty((total_q, hq, dh), dtype=np.float64)
        pr, npairs = None, 0
    else:
        pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        npairs = pr.shape[0]
        out = np.empty((npairs, dh), dtype=np.float64)
    qs = None if q_scale is None else np.ascontiguousarray(q_scale, dtype=np.float32).reshape(-1)
    if qs is not None and qs.size not in (1, hq):
        raise ValueError("q_scale must have 1 or num_q_heads entries")
    bad = lib().kvqo_prefill_attn(_p(q), _p(cu), _p(np.ascontiguousarray(k_cache)),
                                  _p(np.ascontiguousarray(v_cache)), _p(bt), bt.shape[1], _p(sl),
                                  B, hq, hkv, dh, nb, bs, _p(ks), _p(vs), granularity, fmt,
                                  _p(qs), 0 if qs is None else int(qs.size == hq and hq > 1),
                                  window, _p(pr), npairs, _p(out), nthreads)
    if bad:
        raise ValueError(f"oracle prefill: {bad} (row, head) pairs had out-of-range inputs")
    return out


def dequant(cache_codes, scale, granularity, fmt) -> np.ndarray:
    """Unfused-path dequant: bf16(fp32(cast_float(code) * s)) per element."""
    c = np.ascontiguousarray(cache_codes, dtype=np.uint8)
    nb, hkv, bs, dh = c.shape
    s = np.ascontiguousarray(scale, dtype=np.float32)
    out = np.empty(c.shape, dtype=np.uint16)
    lib().kvqo_dequant(_p(c), _p(out), nb, hkv, bs, dh, _p(s), granularity, fmt)
    return out


# --------------------------------------------------------------------------
# Scale calibration ("vLLM FP8 quantized KV cache guide", scale calibration,
# way two; scale = amax / format max)
# --------------------------------------------------------------------------

FMT_MAX = {E4M3: 448.0, E5M2: 57344.0}


def calibrate(x_bf16_bits, granularity, fmt) -> np.ndarray:
    """Scales of one tensor x, bf16 bits [N][Hkv][dh]: amax = the largest
    |x| over its finite values, of each KV head (per head) or of all of them
    (per tensor); s = float32(amax) / float32(fmt_max), one binary32 division
    rounded to nearest even; s = 1 where that is 0."""
    b = np.asarray(x_bf16_bits, dtype=np.uint16)
    hkv = b.shape[1]
    a = np.abs((b.astype(np.uint32) << 16).view(np.float32))
    a = np.where(np.isfinite(a), a, np.float32(0))
    if granularity == PER_HEAD:
        amax = a.transpose(1, 0, 2).reshape(hkv, -1).max(axis=1) if b.shape[0] else np.zeros(hkv, np.float32)
    else:
        amax = np.array([a.max() if a.size else 0.0], np.float32)
    s = (amax.astype(np.float32) / np.float32(FMT_MAX[fmt])).astype(np.float32)
    return np.where(s > 0, s, np.float32(1)).astype(np.float32)


def max_threads() -> int:
    return int(lib().kvqo_max_threads())
