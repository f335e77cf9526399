"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every entry point include/kvq.h declares, the host helpers follow the
kv_cache_dtype and skip-layer rules of the "vLLM FP8 quantized KV cache
guide", and argument validation returns its status before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import fp8_quantized_paged_gb300 as m
    return m


def header_functions():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    return set(re.findall(r"KVQ_API\s+[\w\s\*]+?\b(kvq_\w+)\s*\(", text))


def test_exports_every_declared_symbol(kvq):
    declared = header_functions()
    assert declared == {"kvq_write", "kvq_decode_workspace_size", "kvq_decode_attn",
                        "kvq_decode_attn_static", "kvq_dequant_cache", "kvq_parse_dtype",
                        "kvq_layer_fmt", "kvq_status_string", "kvq_version", "kvq_calibrate_scales",
                        "kvq_write_token_head", "kvq_prefill_attn", "kvq_decode_static_reset"}
    raw = ctypes.CDLL(kvq.LIB_PATH)
    for name in declared:
        assert getattr(raw, name) is not None
    assert set(kvq.SIGNATURES) == declared


def test_parse_dtype(kvq):
    assert kvq.kvq_parse_dtype("fp8") == kvq.KVQ_FMT_E4M3
    assert kvq.kvq_parse_dtype("fp8_e4m3") == kvq.KVQ_FMT_E4M3
    assert kvq.kvq_parse_dtype("fp8_e5m2") == kvq.KVQ_FMT_E5M2
    for s in ("auto", "bfloat16", "bf16"):
        assert kvq.kvq_parse_dtype(s) == kvq.KVQ_FMT_BF16
    for s in ("fp8_inc", "nvfp4", "int8", "", "FP8"):
        assert kvq.kvq_parse_dtype(s) == kvq.KVQ_ERR_UNSUPPORTED
    assert kvq.kvq_parse_dtype(None) == kvq.KVQ_ERR_NULL


def test_skip_layer_rule(kvq):
    E4 = kvq.KVQ_FMT_E4M3
    # attention-type token: every sliding-window layer, and only those
    for layer in range(8):
        sliding = layer % 4 == 3
        want = kvq.KVQ_FMT_BF16 if sliding else E4
        assert kvq.kvq_layer_fmt(E4, layer, sliding, ["sliding_window"]) == want
    # layer-index tokens
    for layer in range(30):
        want = kvq.KVQ_FMT_BF16 if layer in (0, 1, 23) else E4
        assert kvq.kvq_layer_fmt(E4, layer, False, ["0", "1", "23"]) == want
    # both kinds at once; index match without the sliding flag
    assert kvq.kvq_layer_fmt(E4, 3, True, ["5", "sliding_window"]) == kvq.KVQ_FMT_BF16
    assert kvq.kvq_layer_fmt(E4, 5, False, ["5", "sliding_window"]) == kvq.KVQ_FMT_BF16
    assert kvq.kvq_layer_fmt(E4, 6, False, ["5", "sliding_window"]) == E4
    assert kvq.kvq_layer_fmt(kvq.KVQ_FMT_E5M2, 2, True, []) == kvq.KVQ_FMT_E5M2
    assert kvq.kvq_layer_fmt(E4, 12, False, ["1"]) == E4  # "12" is not "1"
    assert kvq.kvq_layer_fmt(7, 0, False, []) == kvq.KVQ_ERR_ARG
    assert kvq.kvq_layer_fmt(E4, -1, False, []) == kvq.KVQ_ERR_ARG


def test_status_strings(kvq):
    for st in range(-7, 1):
        assert kvq.kvq_status_string(st)
    assert kvq.kvq_status_string(-99) == "unknown status"
    assert kvq.kvq_version() >= 100


def test_workspace_size(kvq):
    f = kvq.kvq_decode_workspace_size
    assert f(32, 32, 8, 128, 152) > 0
    assert f(64, 32, 8, 128, 152) > f(32, 32, 8, 128, 152)
    assert f(32, 32, 8, 128, 152) > f(32, 32, 8, 64, 152)
    assert f(0, 32, 8, 128, 152) == 0
    assert f(4, 30, 8, 128, 152) == 0   # Hq % Hkv != 0
    assert f(4, 32, 8, 96, 152) == 0    # head_dim


# ---- argument validation (fake device pointers; every case returns before CUDA)

A = 0x10000  # a 16-byte aligned fake address, never dereferenced


def _write(kvq, **kw):
    args = dict(k=A, v=A, token_stride=1024, slots=A, n=4, hkv=8, dh=128, kc=A, vc=A, nb=10,
                bs=16, ks=A, ksl=1, vs=A, vsl=1, gran=0, fmt=1, status=None)
    args.update(kw)
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return kvq.lib().kvq_write(p(args["k"]), p(args["v"]), args["token_stride"], p(args["slots"]),
                               args["n"], args["hkv"], args["dh"], p(args["kc"]), p(args["vc"]),
                               args["nb"], args["bs"], p(args["ks"]), args["ksl"], p(args["vs"]),
                               args["vsl"], args["gran"], args["fmt"], p(args["status"]), None)


def test_write_validation(kvq):
    assert _write(kvq, kc=None) == kvq.KVQ_ERR_NULL
    assert _write(kvq, k=None) == kvq.KVQ_ERR_NULL
    assert _write(kvq, ks=None) == kvq.KVQ_ERR_NULL
    assert _write(kvq, fmt=3) == kvq.KVQ_ERR_ARG
    assert _write(kvq, gran=2) == kvq.KVQ_ERR_ARG
    assert _write(kvq, n=-1) == kvq.KVQ_ERR_ARG
    assert _write(kvq, dh=96) == kvq.KVQ_ERR_UNSUPPORTED
    assert _write(kvq, bs=32) == kvq.KVQ_ERR_UNSUPPORTED
    assert _write(kvq, token_stride=512) == kvq.KVQ_ERR_SHAPE
    assert _write(kvq, token_stride=1028) == kvq.KVQ_ERR_ALIGN
    assert _write(kvq, k=A + 2) == kvq.KVQ_ERR_ALIGN
    assert _write(kvq, kc=A + 8) == kvq.KVQ_ERR_ALIGN
    # scale shapes: [1] per tensor, [Hkv] per head
    assert _write(kvq, ksl=8) == kvq.KVQ_ERR_SHAPE
    assert _write(kvq, gran=1) == kvq.KVQ_ERR_SHAPE
    assert _write(kvq, gran=1, ksl=8, vsl=32) == kvq.KVQ_ERR_SHAPE
    # bf16 layers ignore scales; zero tokens is a no-op
    assert _write(kvq, n=0) == kvq.KVQ_OK
    assert _write(kvq, n=0, fmt=0, ks=None, vs=None, ksl=0, vsl=0) == kvq.KVQ_OK


def _write_th(kvq, **kw):
    args = dict(k=A, v=A, token_stride=1024, slots=A, n=4, hkv=8, dh=128, kc=A, vc=A, nb=10,
                bs=16, ksc=A, vsc=A, fmt=1, status=None)
    args.update(kw)
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return kvq.lib().kvq_write_token_head(
        p(args["k"]), p(args["v"]), args["token_stride"], p(args["slots"]), args["n"],
        args["hkv"], args["dh"], p(args["kc"]), p(args["vc"]), args["nb"], args["bs"],
        p(args["ksc"]), p(args["vsc"]), args["fmt"], p(args["status"]), None)


def test_write_token_head_validation(kvq):
    assert _write_th(kvq, ksc=None) == kvq.KVQ_ERR_NULL
    assert _write_th(kvq, vsc=None) == kvq.KVQ_ERR_NULL
    assert _write_th(kvq, fmt=0) == kvq.KVQ_ERR_UNSUPPORTED  # bf16 has no scales
    assert _write_th(kvq, fmt=5) == kvq.KVQ_ERR_ARG
    assert _write_th(kvq, ksc=A + 4) == kvq.KVQ_ERR_ALIGN
    assert _write_th(kvq, kc=None) == kvq.KVQ_ERR_NULL
    assert _write_th(kvq, n=-1) == kvq.KVQ_ERR_ARG
    assert _write_th(kvq, dh=96) == kvq.KVQ_ERR_UNSUPPORTED
    assert _write_th(kvq, token_stride=512) == kvq.KVQ_ERR_SHAPE
    assert _write_th(kvq, k=A + 2) == kvq.KVQ_ERR_ALIGN
    assert _write_th(kvq, n=0) == kvq.KVQ_OK


def _prefill(kvq, **kw):
    args = dict(q=A, cu=A, nq=64, maxq=32, kc=A, vc=A, bt=A, maxb=4, sl=A, B=2, hq=32, hkv=8,
                dh=128, nb=8, bs=16, qs=None, qsl=0, ks=A, ksl=1, vs=A, vsl=1, gran=0, fmt=1,
                win=0, flags=0, out=A)
    args.update(kw)
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return kvq.lib().kvq_prefill_attn(
        p(args["q"]), p(args["cu"]), args["nq"], args["maxq"], p(args["kc"]), p(args["vc"]),
        p(args["bt"]), args["maxb"], p(args["sl"]), args["B"], args["hq"], args["hkv"], args["dh"],
        args["nb"], args["bs"], p(args["qs"]), args["qsl"], p(args["ks"]), args["ksl"],
        p(args["vs"]), args["vsl"], args["gran"], args["fmt"], args["win"], args["flags"],
        p(args["out"]), None, None)


def test_prefill_validation(kvq):
    assert _prefill(kvq, q=None) == kvq.KVQ_ERR_NULL
    assert _prefill(kvq, cu=None) == kvq.KVQ_ERR_NULL
    assert _prefill(kvq, fmt=3) == kvq.KVQ_ERR_ARG
    assert _prefill(kvq, gran=2) == kvq.KVQ_ERR_SHAPE  # per-token scales want the scale caches
    assert _prefill(kvq, gran=2, ksl=8 * 8 * 16, vsl=8 * 8 * 16, nq=0) == kvq.KVQ_OK
    assert _prefill(kvq, gran=2, ksl=8 * 8 * 16, vsl=8 * 8 * 16, ks=A + 4) == kvq.KVQ_ERR_ALIGN
    assert _prefill(kvq, gran=2, fmt=0) == kvq.KVQ_ERR_ARG  # bf16 cache: no scales
    assert _prefill(kvq, gran=3) == kvq.KVQ_ERR_ARG
    assert _prefill(kvq, flags=2) == kvq.KVQ_ERR_ARG        # KVQ_CACHE_READY: decode only
    assert _prefill(kvq, flags=1) == kvq.KVQ_ERR_NULL       # KVQ_Q_FP8 wants q_scale
    assert _prefill(kvq, flags=1, qs=A, qsl=5) == kvq.KVQ_ERR_SHAPE
    assert _prefill(kvq, flags=1, qs=A, qsl=32, nq=0) == kvq.KVQ_OK
    assert _prefill(kvq, flags=1, qs=A, qsl=1, fmt=0) == kvq.KVQ_ERR_ARG
    assert _prefill(kvq, B=0) == kvq.KVQ_ERR_ARG
    assert _prefill(kvq, nq=-1) == kvq.KVQ_ERR_ARG
    assert _prefill(kvq, win=-2) == kvq.KVQ_ERR_ARG
    assert _prefill(kvq, dh=96) == kvq.KVQ_ERR_UNSUPPORTED
    assert _prefill(kvq, bs=32) == kvq.KVQ_ERR_UNSUPPORTED
    assert _prefill(kvq, hq=30) == kvq.KVQ_ERR_SHAPE
    assert _prefill(kvq, hq=48) == kvq.KVQ_ERR_UNSUPPORTED  # group of 6
    assert _prefill(kvq, hq=128) == kvq.KVQ_ERR_UNSUPPORTED  # group of 16
    assert _prefill(kvq, out=A + 4) == kvq.KVQ_ERR_ALIGN
    assert _prefill(kvq, cu=A + 2) == kvq.KVQ_ERR_ALIGN
    assert _prefill(kvq, ks=None) == kvq.KVQ_ERR_NULL
    assert _prefill(kvq, gran=1) == kvq.KVQ_ERR_SHAPE
    assert _prefill(kvq, nq=0) == kvq.KVQ_OK
    assert _prefill(kvq, maxq=0) == kvq.KVQ_OK
    assert _prefill(kvq, fmt=0, ks=None, vs=None, nq=0) == kvq.KVQ_OK


def _decode(kvq, **kw):
    args = dict(q=A, kc=A, vc=A, bt=A, maxb=4, sl=A, B=2, hq=32, hkv=8, dh=128, nb=8, bs=16,
                qs=None, qsl=0, ks=A, ksl=1, vs=A, vsl=1, gran=0, fmt=1, win=0, flags=0, ws=A,
                wsb=1 << 30, out=A)
    args.update(kw)
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return kvq.lib().kvq_decode_attn(
        p(args["q"]), p(args["kc"]), p(args["vc"]), p(args["bt"]), args["maxb"], p(args["sl"]),
        args["B"], args["hq"], args["hkv"], args["dh"], args["nb"], args["bs"], p(args["qs"]),
        args["qsl"], p(args["ks"]), args["ksl"], p(args["vs"]), args["vsl"], args["gran"],
        args["fmt"], args["win"], args["flags"], p(args["ws"]), args["wsb"], p(args["out"]), None,
        None)


def test_decode_validation(kvq):
    assert _decode(kvq, q=None) == kvq.KVQ_ERR_NULL
    assert _decode(kvq, ws=None) == kvq.KVQ_ERR_NULL
    assert _decode(kvq, fmt=-1) == kvq.KVQ_ERR_ARG
    assert _decode(kvq, B=0) == kvq.KVQ_ERR_ARG
    assert _decode(kvq, win=-1) == kvq.KVQ_ERR_ARG
    assert _decode(kvq, flags=kvq.KVQ_Q_FP8) == kvq.KVQ_ERR_NULL  # the mode needs q_scale
    assert _decode(kvq, flags=kvq.KVQ_Q_FP8, fmt=0, qs=A, qsl=1) == kvq.KVQ_ERR_UNSUPPORTED
    assert _decode(kvq, flags=kvq.KVQ_Q_FP8, qs=A, qsl=32) == kvq.KVQ_ERR_SHAPE
    assert _decode(kvq, flags=4) == kvq.KVQ_ERR_ARG
    assert _decode(kvq, dh=80) == kvq.KVQ_ERR_UNSUPPORTED
    assert _decode(kvq, bs=8) == kvq.KVQ_ERR_UNSUPPORTED
    assert _decode(kvq, hq=30) == kvq.KVQ_ERR_SHAPE
    assert _decode(kvq, hq=128) == kvq.KVQ_ERR_UNSUPPORTED  # group of 16 > 8
    assert _decode(kvq, B=5000) == kvq.KVQ_ERR_UNSUPPORTED
    assert _decode(kvq, out=A + 4) == kvq.KVQ_ERR_ALIGN
    assert _decode(kvq, ws=A + 16) == kvq.KVQ_ERR_ALIGN
    assert _decode(kvq, ks=None) == kvq.KVQ_ERR_NULL
    assert _decode(kvq, gran=1) == kvq.KVQ_ERR_SHAPE            # k/v scale must be [Hkv]
    assert _decode(kvq, gran=1, ksl=8, vsl=8, qs=A, qsl=8) == kvq.KVQ_ERR_SHAPE  # q scale [Hq]
    assert _decode(kvq, qs=A, qsl=32) == kvq.KVQ_ERR_SHAPE      # per tensor q scale is [1]
    # per-(token, head) scales: the scale caches [num_blocks][Hkv][16]
    th = dict(gran=2, ksl=8 * 8 * 16, vsl=8 * 8 * 16)
    assert _decode(kvq, gran=3) == kvq.KVQ_ERR_ARG
    assert _decode(kvq, gran=2) == kvq.KVQ_ERR_SHAPE
    assert _decode(kvq, **dict(th, vsl=8)) == kvq.KVQ_ERR_SHAPE
    assert _decode(kvq, **dict(th, ks=A + 4)) == kvq.KVQ_ERR_ALIGN
    assert _decode(kvq, **dict(th, qs=A, qsl=8)) == kvq.KVQ_ERR_SHAPE  # q scale: [1] or [Hq]


def test_python_constants_mirror_the_header():
    """Every #define of include/kvq.h that the binding also names has the
    same value there."""
    import fp8_quantized_paged_gb300 as kvq
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    found = 0
    for name, expr in re.findall(r"#define\s+(KVQ_\w+)\s+(.+?)\s*(?:/\*.*)?$", text, re.M):
        if not hasattr(kvq, name):
            continue
        val = eval(re.sub(r"(\d+)u\b", r"\1", expr.replace("(size_t)", "")))
        assert getattr(kvq, name) == val, name
        found += 1
    for name, val in re.findall(r"\b(KVQ_\w+)\s*=\s*(-?\d+)", text):  # enumerators
        if hasattr(kvq, name):
            assert getattr(kvq, name) == int(val), name
            found += 1
    assert found >= 15
