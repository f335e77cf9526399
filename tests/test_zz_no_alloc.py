"""kvq_decode_attn_static: decode attention for callers that cannot allocate
device memory (a plugin given only input and output pointers, or a serving
loop whose memory plan is fixed and may not call cudaMalloc on the decode
path).  Its scratch is an array inside the library, so its output must match
kvq_decode_attn with a caller workspace, call after call.

This file is collected last on purpose: it must pass alone in a fresh
process and after every other test."""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from kvq_testlib import DeviceLayer, bf16_out_to_f64, check_attention

pytestmark = pytest.mark.gpu


def _call_static(kvq, d, out):
    lay = d.lay
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return kvq.lib().kvq_decode_attn_static(
        p(d.q), p(d.kc), p(d.vc), p(d.bt), d.bt.shape[1], p(d.sl), lay.B, lay.Hq, lay.Hkv, lay.dh,
        d.kc.shape[0], 16, p(d.qs), d.qs.numel(), p(d.ks), d.ks.numel(), p(d.vs), d.vs.numel(),
        lay.gran, lay.fmt, lay.window, 0, p(out), p(d.status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("cfg,layer", [(2, 0), (5, 3)], ids=["llama8b_fp8", "mixed_bf16_window"])
def test_static_scratch_matches_workspace_entry_point(cfg, layer):
    import fp8_quantized_paged_gb300 as kvq
    lay = workloads.make_layer(cfg, layer)
    d = DeviceLayer(lay)
    d.write()
    ref = bf16_out_to_f64(d.decode())
    assert d.status_word() == 0
    for _ in range(2):  # two calls in a row share the same scratch array
        out = torch.full((lay.B, lay.Hq, lay.dh), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        assert _call_static(kvq, d, out) == kvq.KVQ_OK
        assert d.status_word() == 0
        got = bf16_out_to_f64(out)
        check_attention(got, ref, "static scratch vs caller workspace")
        np.testing.assert_array_equal(got, ref)  # same kernels, same inputs


def test_static_scratch_rejects_sizes_beyond_its_array():
    import fp8_quantized_paged_gb300 as kvq
    need = kvq.kvq_decode_workspace_size(4096, 64, 8, 128)
    assert need > kvq.KVQ_STATIC_SCRATCH_BYTES
    A = ctypes.c_void_p(0x10000)  # never dereferenced: the call returns first
    st = kvq.lib().kvq_decode_attn_static(A, A, A, A, 4, A, 4096, 64, 8, 128, 8, 16, None, 0, A,
                                          1, A, 1, 0, 1, 0, 0, A, None, None)
    assert st == kvq.KVQ_ERR_WORKSPACE
