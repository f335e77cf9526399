"""Bounded device waits that run out.

Every mbarrier wait of the kernels polls a bounded number of times; when the
bound is reached the kernel raises KVQ_DEV_WAIT_TIMEOUT in dev_status, its
roles stop at the same barriers, wait (bounded) for their copies in flight and
return, so the CUDA context stays usable.  These tests build a copy of the
library with the test hooks compiled in and the bound cut to 2^16 polls, make
CTA 0's producer withhold the copy of one page (a full barrier that nothing
completes), and check that the status reports the timeout, that the call
returns promptly, and that after the workspace counters are cleared -- for
the static-scratch entry, after kvq_decode_static_reset -- the next call is
correct.  No GPU fault is involved: the hook only skips issuing a copy.
"""
import ctypes
import os
import time

import numpy as np
import pytest
import torch

from kvq_testlib import DeviceLayer, bf16_out_to_f64, check_attention, oracle_caches, oracle_decode
from test_gpu_parity import _custom_layer

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WITHHELD = 3  # stream position of CTA 0's page whose copy is withheld


@pytest.fixture(scope="module")
def kvq():
    import fp8_quantized_paged_gb300 as m
    return m


@pytest.fixture(scope="module")
def tlib(kvq):
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_kvq_build", os.path.join(ROOT, "fp8_quantized_paged_gb300", "build.py"))
    bmod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bmod)
    lib = ctypes.CDLL(bmod.build_test_lib())
    for name, (res, args) in kvq.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    lib.kvq_test_withhold_page.restype = None
    lib.kvq_test_withhold_page.argtypes = [ctypes.c_int]
    yield lib
    lib.kvq_test_withhold_page(-1)


def _layer():
    # four sequences of 4096 tokens over 8 KV heads: CTA 0's range holds pages
    return _custom_layer([4096] * 4, Hq=32, Hkv=8, dh=128, seed=500)


def _args(d, static):
    lay = d.lay
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    head = [p(d.q), p(d.kc), p(d.vc), p(d.bt), d.bt.shape[1], p(d.sl), lay.B, lay.Hq, lay.Hkv,
            lay.dh, d.kc.shape[0], 16, None, 0, p(d.ks), d.ks.numel(), p(d.vs), d.vs.numel(),
            lay.gran, lay.fmt, lay.window, 0]
    tail = [p(d.out), p(d.status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)]
    if static:
        return head + tail
    return head + [p(d.ws), d.ws.numel() * d.ws.element_size()] + tail


def _call(lib, d, static):
    fn = lib.kvq_decode_attn_static if static else lib.kvq_decode_attn
    d.status.zero_()
    t0 = time.time()
    assert fn(*_args(d, static)) == 0
    torch.cuda.synchronize()
    return time.time() - t0


@pytest.mark.parametrize("static", [False, True])
def test_withheld_page_times_out_then_recovers(kvq, tlib, static):
    lay = _layer()
    d = DeviceLayer(lay)
    d.write()
    K, V = oracle_caches(lay)
    ref = oracle_decode(lay, K, V)

    tlib.kvq_test_withhold_page(WITHHELD)
    secs = _call(tlib, d, static)
    st = int(d.status.item())
    assert st & kvq.KVQ_DEV_WAIT_TIMEOUT, f"status {st}"
    assert secs < 30.0  # bounded: the waits gave up

    # the context is usable, and once the counters are cleared the next call is right
    tlib.kvq_test_withhold_page(-1)
    if static:
        assert tlib.kvq_decode_static_reset(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    else:
        d.ws[: kvq.KVQ_WS_COUNTER_BYTES].zero_()
    _call(tlib, d, static)
    assert int(d.status.item()) == 0
    check_attention(bf16_out_to_f64(d.out), ref, "after the timeout")
    # and again, without clearing: a completed call leaves the counters zero
    d.out.zero_()
    _call(tlib, d, static)
    assert int(d.status.item()) == 0
    check_attention(bf16_out_to_f64(d.out), ref, "the call after")


def test_product_library_has_no_test_hook(kvq):
    raw = ctypes.CDLL(kvq.LIB_PATH)
    with pytest.raises(AttributeError):
        getattr(raw, "kvq_test_withhold_page")
