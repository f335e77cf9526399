"""Python binding of libkvq (FP8 paged KV cache for GB300).

Argument marshalling only: every step of the path runs in the CUDA kernels of
``_build/libkvq.so``, reached through the C ABI declared in
``include/kvq.h``.  The functions carry the C names.  Tensors are torch CUDA
tensors (torch provides device memory and streams); pointers, sizes and the
current stream are passed to the library, a negative status raises
``KvqError``.  There is no fallback: importing this package without the
built library raises ImportError.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkvq.so")

KVQ_FMT_BF16, KVQ_FMT_E4M3, KVQ_FMT_E5M2 = 0, 1, 2
KVQ_SCALE_PER_TENSOR, KVQ_SCALE_PER_HEAD, KVQ_SCALE_PER_TOKEN_HEAD = 0, 1, 2
KVQ_OK, KVQ_ERR_NULL, KVQ_ERR_SHAPE, KVQ_ERR_ALIGN = 0, -1, -2, -3
KVQ_ERR_UNSUPPORTED, KVQ_ERR_WORKSPACE, KVQ_ERR_CUDA, KVQ_ERR_ARG = -4, -5, -6, -7
KVQ_DEV_BAD_SLOT, KVQ_DEV_BAD_BLOCK, KVQ_DEV_BAD_SEQLEN, KVQ_DEV_WAIT_TIMEOUT = 1, 2, 4, 8
KVQ_DEV_INTERNAL = 16
KVQ_DEV_BAD_QLEN = 32
KVQ_Q_FP8 = 1
KVQ_CACHE_READY = 2
KVQ_STATIC_SCRATCH_BYTES = 16 << 20
BLOCK_SIZE = 16

# exported symbol -> (restype, argtypes)
_vp, _i32, _i64, _u32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint, ctypes.c_size_t
SIGNATURES = {
    "kvq_write": (_i32, [_vp, _vp, _i64, _vp, _i64, _i32, _i32, _vp, _vp, _i64, _i32, _vp, _i32,
                         _vp, _i32, _i32, _i32, _vp, _vp]),
    "kvq_write_token_head": (_i32, [_vp, _vp, _i64, _vp, _i64, _i32, _i32, _vp, _vp, _i64, _i32,
                                    _vp, _vp, _i32, _vp, _vp]),
    "kvq_decode_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "kvq_decode_attn": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i64, _i32,
                               _vp, _i32, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _u32, _vp, _sz,
                               _vp, _vp, _vp]),
    "kvq_decode_attn_static": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i64,
                                      _i32, _vp, _i32, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                      _u32, _vp, _vp, _vp]),
    "kvq_decode_static_reset": (_i32, [_vp]),
    "kvq_prefill_attn": (_i32, [_vp, _vp, _i64, _i32, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32,
                                _i32, _i64, _i32, _vp, _i32, _vp, _i32, _vp, _i32, _i32, _i32,
                                _i32, _u32, _vp, _vp, _vp]),
    "kvq_dequant_cache": (_i32, [_vp, _vp, _i64, _i32, _i32, _i32, _vp, _i32, _i32, _i32, _vp]),
    "kvq_calibrate_scales": (_i32, [_vp, _vp, _i64, _i64, _i32, _i32, _i32, _i32, _vp, _vp, _vp,
                                    _vp]),
    "kvq_parse_dtype": (_i32, [ctypes.c_char_p]),
    "kvq_layer_fmt": (_i32, [_i32, _i32, _i32, ctypes.POINTER(ctypes.c_char_p), _i32]),
    "kvq_status_string": (ctypes.c_char_p, [_i32]),
    "kvq_version": (_i32, []),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libkvq is not built ({LIB_PATH} missing); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def lib():
    return _lib


class KvqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kvq_status_string(status)} ({status})")


def _check(status: int, where: str) -> None:
    if status != KVQ_OK:
        raise KvqError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _len(t):
    return 0 if t is None else int(t.numel())


def _need(t, where, name, size=None, dtype=None, contiguous=True, min_numel=None):
    """The C ABI sees only a pointer: check what it cannot, before the call
    (element type, dense layout, length), so that a wrong tensor raises here
    instead of being read out of bounds on the device."""
    if t is None:
        return
    if dtype is not None and t.dtype != dtype:
        raise KvqError(KVQ_ERR_ARG, f"{where}: {name} must be {dtype}, got {t.dtype}")
    if size is not None and t.element_size() != size:
        raise KvqError(KVQ_ERR_ARG, f"{where}: {name} must have {size}-byte elements, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise KvqError(KVQ_ERR_SHAPE, f"{where}: {name} must be contiguous")
    if min_numel is not None and t.numel() < min_numel:
        raise KvqError(KVQ_ERR_SHAPE, f"{where}: {name} holds {t.numel()} elements, needs {min_numel}")


def _cache_size(fmt):
    """Element size of a cache in format fmt (None for an unknown format,
    which the library itself rejects)."""
    return {KVQ_FMT_BF16: 2, KVQ_FMT_E4M3: 1, KVQ_FMT_E5M2: 1}.get(fmt)


def _need_all(where, *specs):
    """_need on every (tensor, name, ...) spec, then every tensor in CUDA memory."""
    for spec in specs:
        _need(spec[0], where, *spec[1:])
    for spec in specs:
        if spec[0] is not None and not spec[0].is_cuda:
            raise KvqError(KVQ_ERR_ARG, f"{where}: {spec[1]} must be a CUDA tensor")


# --------------------------------------------------------------------------
# compute entry points (torch CUDA tensors)
# --------------------------------------------------------------------------

def _check_write_args(where, k, v, slot_mapping, k_cache, v_cache, fmt, dev_status, *more):
    import torch
    n = k.shape[0]
    _need_all(where, (k, "k", 2, None, False), (v, "v", 2, None, False),
              (slot_mapping, "slot_mapping", None, torch.int64, True, n),
              (k_cache, "k_cache", _cache_size(fmt)), (v_cache, "v_cache", _cache_size(fmt)),
              (dev_status, "dev_status", 4, None, True, 1), *more)


def kvq_write(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, scale_granularity, fmt,
              dev_status=None, stream=None, token_stride=None) -> None:
    """Quantize-and-scatter: k, v bf16 [N][Hkv][dh] (token stride may exceed Hkv*dh);
    caches [num_blocks][Hkv][16][dh] uint8 (FP8) or bf16."""
    n, hkv, dh = k.shape
    stride = k.stride(0) if token_stride is None else token_stride
    if v.stride(0) != stride or k.stride(1) != dh or k.stride(2) != 1 or v.stride(1) != dh:
        raise KvqError(KVQ_ERR_SHAPE, "kvq_write")
    nb, hkv2, bs, dh2 = k_cache.shape
    if (hkv2, dh2) != (hkv, dh) or v_cache.shape != k_cache.shape or tuple(v.shape) != (n, hkv, dh):
        raise KvqError(KVQ_ERR_SHAPE, "kvq_write")
    _check_write_args("kvq_write", k, v, slot_mapping, k_cache, v_cache, fmt, dev_status,
                      (k_scale, "k_scale", 4), (v_scale, "v_scale", 4))
    st = _lib.kvq_write(_ptr(k), _ptr(v), stride, _ptr(slot_mapping), n, hkv, dh, _ptr(k_cache),
                        _ptr(v_cache), nb, bs, _ptr(k_scale), _len(k_scale), _ptr(v_scale),
                        _len(v_scale), scale_granularity, fmt, _ptr(dev_status), _stream(stream))
    _check(st, "kvq_write")


def kvq_write_token_head(k, v, slot_mapping, k_cache, v_cache, k_scale_cache, v_scale_cache,
                         fmt, dev_status=None, stream=None, token_stride=None) -> None:
    """Quantize-and-scatter with per-(token, KV head) scales: every written
    row's scale amax / fmt_max goes to the scale caches fp32
    [num_blocks][Hkv][16] (see ``new_scale_cache``)."""
    n, hkv, dh = k.shape
    stride = k.stride(0) if token_stride is None else token_stride
    if v.stride(0) != stride or k.stride(1) != dh or k.stride(2) != 1 or v.stride(1) != dh:
        raise KvqError(KVQ_ERR_SHAPE, "kvq_write_token_head")
    nb, hkv2, bs, dh2 = k_cache.shape
    if (hkv2, dh2) != (hkv, dh) or v_cache.shape != k_cache.shape or tuple(v.shape) != (n, hkv, dh):
        raise KvqError(KVQ_ERR_SHAPE, "kvq_write_token_head")
    for sc in (k_scale_cache, v_scale_cache):
        if tuple(sc.shape) != (nb, hkv, bs) or not sc.is_contiguous():
            raise KvqError(KVQ_ERR_SHAPE, "kvq_write_token_head")
    _check_write_args("kvq_write_token_head", k, v, slot_mapping, k_cache, v_cache, fmt,
                      dev_status, (k_scale_cache, "k_scale_cache", 4),
                      (v_scale_cache, "v_scale_cache", 4))
    st = _lib.kvq_write_token_head(_ptr(k), _ptr(v), stride, _ptr(slot_mapping), n, hkv, dh,
                                   _ptr(k_cache), _ptr(v_cache), nb, bs, _ptr(k_scale_cache),
                                   _ptr(v_scale_cache), fmt, _ptr(dev_status), _stream(stream))
    _check(st, "kvq_write_token_head")


def kvq_calibrate_scales(k, v, k_scale, v_scale, scale_granularity, fmt, dev_status=None,
                         stream=None, token_stride=None) -> None:
    """Scales from the data: k, v bf16 [N][Hkv][dh] -> k_scale, v_scale fp32
    ([1] or [Hkv]) = amax / fmt_max."""
    n, hkv, dh = k.shape
    stride = k.stride(0) if token_stride is None else token_stride
    if v.stride(0) != stride or k.stride(1) != dh or k.stride(2) != 1 or v.stride(1) != dh or \
            tuple(v.shape) != (n, hkv, dh):
        raise KvqError(KVQ_ERR_SHAPE, "kvq_calibrate_scales")
    want = hkv if scale_granularity == KVQ_SCALE_PER_HEAD else 1
    if k_scale.numel() != want or v_scale.numel() != want:
        raise KvqError(KVQ_ERR_SHAPE, "kvq_calibrate_scales")
    _need_all("kvq_calibrate_scales", (k, "k", 2, None, False), (v, "v", 2, None, False),
              (k_scale, "k_scale", 4), (v_scale, "v_scale", 4),
              (dev_status, "dev_status", 4, None, True, 1))
    st = _lib.kvq_calibrate_scales(_ptr(k), _ptr(v), stride, n, hkv, dh, scale_granularity, fmt,
                                   _ptr(k_scale), _ptr(v_scale), _ptr(dev_status), _stream(stream))
    _check(st, "kvq_calibrate_scales")


def kvq_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, num_sms=0) -> int:
    return int(_lib.kvq_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                              num_sms))


def _check_attn_args(where, q, k_cache, v_cache, block_tables, seq_lens, B, scales, fmt, out,
                     dev_status, *more):
    import torch
    _need_all(where, (q, "q", 2), (out, "out", 2),
              (k_cache, "k_cache", _cache_size(fmt)), (v_cache, "v_cache", _cache_size(fmt)),
              (block_tables, "block_tables", None, torch.int32),
              (seq_lens, "seq_lens", None, torch.int32, True, B),
              (dev_status, "dev_status", 4, None, True, 1),
              *[(sc, name, 4) for sc, name in zip(scales, ("q_scale", "k_scale", "v_scale"))],
              *more)


def kvq_decode_attn(q, k_cache, v_cache, block_tables, seq_lens, q_scale, k_scale, v_scale,
                    scale_granularity, fmt, sliding_window, workspace, out, dev_status=None,
                    stream=None, flags=0) -> None:
    """Decode attention: q bf16 [B][Hq][dh] -> out bf16 [B][Hq][dh]."""
    B, hq, dh = q.shape
    nb, hkv, bs, dh2 = k_cache.shape
    if dh2 != dh or tuple(out.shape) != (B, hq, dh) or block_tables.shape[0] != B:
        raise KvqError(KVQ_ERR_SHAPE, "kvq_decode_attn")
    _check_attn_args("kvq_decode_attn", q, k_cache, v_cache, block_tables, seq_lens, B,
                     (q_scale, k_scale, v_scale), fmt, out, dev_status, (workspace, "workspace"))
    st = _lib.kvq_decode_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                              block_tables.shape[1], _ptr(seq_lens), B, hq, hkv, dh, nb, bs,
                              _ptr(q_scale), _len(q_scale), _ptr(k_scale), _len(k_scale),
                              _ptr(v_scale), _len(v_scale), scale_granularity, fmt,
                              sliding_window, flags, _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _ptr(out),
                              _ptr(dev_status), _stream(stream))
    _check(st, "kvq_decode_attn")


def kvq_decode_attn_static(q, k_cache, v_cache, block_tables, seq_lens, q_scale, k_scale,
                           v_scale, scale_granularity, fmt, sliding_window, out, dev_status=None,
                           stream=None, flags=0) -> None:
    """kvq_decode_attn with the library's own static scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    B, hq, dh = q.shape
    nb, hkv, bs, dh2 = k_cache.shape
    if dh2 != dh or tuple(out.shape) != (B, hq, dh) or block_tables.shape[0] != B:
        raise KvqError(KVQ_ERR_SHAPE, "kvq_decode_attn_static")
    _check_attn_args("kvq_decode_attn_static", q, k_cache, v_cache, block_tables, seq_lens, B,
                     (q_scale, k_scale, v_scale), fmt, out, dev_status)
    st = _lib.kvq_decode_attn_static(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                     block_tables.shape[1], _ptr(seq_lens), B, hq, hkv, dh, nb,
                                     bs, _ptr(q_scale), _len(q_scale), _ptr(k_scale),
                                     _len(k_scale), _ptr(v_scale), _len(v_scale),
                                     scale_granularity, fmt, sliding_window, flags, _ptr(out),
                                     _ptr(dev_status), _stream(stream))
    _check(st, "kvq_decode_attn_static")


def kvq_decode_static_reset(stream=None) -> None:
    """Clear the static scratch array's counters on the current device (after
    a kvq_decode_attn_static call reported KVQ_DEV_WAIT_TIMEOUT)."""
    _check(_lib.kvq_decode_static_reset(_stream(stream)), "kvq_decode_static_reset")


def kvq_prefill_attn(q, cu_q_lens, max_q_len, k_cache, v_cache, block_tables, seq_lens,
                     k_scale, v_scale, scale_granularity, fmt, sliding_window, out,
                     dev_status=None, stream=None, q_scale=None, flags=0) -> None:
    """Prefill / prefix-hit attention: q bf16 [total_q][Hq][dh], cu_q_lens int32
    [B+1] (device), max_q_len a host bound of the per-sequence query counts;
    the queries are each sequence's last tokens, attending causally.  With
    KVQ_SCALE_PER_TOKEN_HEAD, k_scale / v_scale are the scale caches of
    kvq_write_token_head; flags=KVQ_Q_FP8 takes q_scale ([1] or [Hq])."""
    total_q, hq, dh = q.shape
    nb, hkv, bs, dh2 = k_cache.shape
    B = seq_lens.shape[0]
    if dh2 != dh or tuple(out.shape) != (total_q, hq, dh) or cu_q_lens.shape[0] != B + 1 or \
            block_tables.shape[0] != B:
        raise KvqError(KVQ_ERR_SHAPE, "kvq_prefill_attn")
    import torch
    _check_attn_args("kvq_prefill_attn", q, k_cache, v_cache, block_tables, seq_lens, B,
                     (q_scale, k_scale, v_scale), fmt, out, dev_status,
                     (cu_q_lens, "cu_q_lens", None, torch.int32))
    st = _lib.kvq_prefill_attn(_ptr(q), _ptr(cu_q_lens), total_q, int(max_q_len), _ptr(k_cache),
                               _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                               _ptr(seq_lens), B, hq, hkv, dh, nb, bs, _ptr(q_scale),
                               _len(q_scale), _ptr(k_scale), _len(k_scale), _ptr(v_scale),
                               _len(v_scale), scale_granularity, fmt, sliding_window, flags,
                               _ptr(out), _ptr(dev_status), _stream(stream))
    _check(st, "kvq_prefill_attn")


def kvq_dequant_cache(src, dst_bf16, scale, scale_granularity, fmt, stream=None) -> None:
    nb, hkv, bs, dh = src.shape
    if tuple(dst_bf16.shape) != tuple(src.shape):
        raise KvqError(KVQ_ERR_SHAPE, "kvq_dequant_cache")
    _need_all("kvq_dequant_cache", (src, "src", _cache_size(fmt)), (dst_bf16, "dst_bf16", 2),
              (scale, "scale", 4))
    st = _lib.kvq_dequant_cache(_ptr(src), _ptr(dst_bf16), nb, hkv, bs, dh, _ptr(scale),
                                _len(scale), scale_granularity, fmt, _stream(stream))
    _check(st, "kvq_dequant_cache")


# --------------------------------------------------------------------------
# host helpers
# --------------------------------------------------------------------------

def kvq_parse_dtype(s: str) -> int:
    return int(_lib.kvq_parse_dtype(None if s is None else s.encode()))


def kvq_layer_fmt(fmt: int, layer_idx: int, is_sliding: bool, skip) -> int:
    arr = (ctypes.c_char_p * max(len(skip), 1))(*[x.encode() for x in skip])
    return int(_lib.kvq_layer_fmt(fmt, layer_idx, 1 if is_sliding else 0, arr, len(skip)))


def kvq_status_string(status: int) -> str:
    return _lib.kvq_status_string(status).decode()


def kvq_version() -> int:
    return int(_lib.kvq_version())


# --------------------------------------------------------------------------
# allocation helpers (torch memory; no compute)
# --------------------------------------------------------------------------

def new_cache(num_blocks, num_kv_heads, head_dim, fmt, device="cuda"):
    import torch
    dt = torch.bfloat16 if fmt == KVQ_FMT_BF16 else torch.uint8
    return torch.empty((num_blocks, num_kv_heads, BLOCK_SIZE, head_dim), dtype=dt, device=device)


def new_scale_cache(num_blocks, num_kv_heads, device="cuda"):
    """Per-(token, KV head) scales beside the pages: fp32 [num_blocks][Hkv][16]."""
    import torch
    return torch.empty((num_blocks, num_kv_heads, BLOCK_SIZE), dtype=torch.float32, device=device)


KVQ_WS_COUNTER_BYTES = 65536 * 4  # leading workspace bytes that must start at zero


def new_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, device="cuda"):
    """A decode workspace, zero-filled (its counters must start at zero)."""
    import torch
    n = kvq_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim)
    if n == 0:
        raise KvqError(KVQ_ERR_ARG, "kvq_decode_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)
