"""The Python binding checks what the C ABI cannot see behind a pointer
(element type, dense layout, length, CUDA memory) and raises before any
library call.  Every case here fails one check, so nothing reaches the device
(no GPU needed)."""
import pytest
import torch

B, HQ, HKV, DH, NB = 2, 8, 2, 64, 6
# status codes and enums of include/kvq.h (the package is imported by the
# fixture, after the library is built)
ERR_SHAPE, ERR_ARG = -2, -7
FMT_BF16, FMT_E4M3 = 0, 1
PER_HEAD = 1


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import fp8_quantized_paged_gb300 as m
    return m


def _args(**over):
    """Host tensors shaped like a valid decode call (the device check, which
    comes last, is the only one they fail)."""
    a = dict(q=torch.zeros((B, HQ, DH), dtype=torch.bfloat16),
             kc=torch.zeros((NB, HKV, 16, DH), dtype=torch.uint8),
             vc=torch.zeros((NB, HKV, 16, DH), dtype=torch.uint8),
             bt=torch.zeros((B, 3), dtype=torch.int32),
             sl=torch.ones(B, dtype=torch.int32),
             ks=torch.ones(HKV, dtype=torch.float32),
             vs=torch.ones(HKV, dtype=torch.float32),
             ws=torch.zeros(1 << 20, dtype=torch.uint8),
             out=torch.zeros((B, HQ, DH), dtype=torch.bfloat16))
    a.update(over)
    return a


def _decode(kvq, a, fmt=FMT_E4M3):
    kvq.kvq_decode_attn(a["q"], a["kc"], a["vc"], a["bt"], a["sl"], None, a["ks"], a["vs"],
                        PER_HEAD, fmt, 0, a["ws"], a["out"])


def _status(kvq, fn):
    with pytest.raises(kvq.KvqError) as e:
        fn()
    return e.value.status, str(e.value)


def test_host_tensors_rejected(kvq):
    st, msg = _status(kvq, lambda: _decode(kvq, _args()))
    assert st == ERR_ARG and "CUDA" in msg


@pytest.mark.parametrize("over,status,word", [
    (dict(kc=torch.zeros((NB, HKV, 16, DH), dtype=torch.bfloat16)), ERR_ARG, "k_cache"),
    (dict(bt=torch.zeros((B, 3), dtype=torch.int64)), ERR_ARG, "block_tables"),
    (dict(sl=torch.ones(B, dtype=torch.int64)), ERR_ARG, "seq_lens"),
    (dict(sl=torch.ones(B - 1, dtype=torch.int32)), ERR_SHAPE, "seq_lens"),
    (dict(ks=torch.ones(HKV, dtype=torch.float64)), ERR_ARG, "k_scale"),
    (dict(q=torch.zeros((HQ, B, DH), dtype=torch.bfloat16).transpose(0, 1)), ERR_SHAPE, "q"),
    (dict(q=torch.zeros((B, HQ, DH), dtype=torch.float32)), ERR_ARG, "q"),
    (dict(out=torch.zeros((B, HQ, DH), dtype=torch.float32)), ERR_ARG, "out"),
])
def test_decode_argument_checks(kvq, over, status, word):
    st, msg = _status(kvq, lambda: _decode(kvq, _args(**over)))
    assert st == status and word in msg


def test_bf16_format_needs_bf16_caches(kvq):
    # one-byte caches read as bf16 would run past the allocation
    st, msg = _status(kvq, lambda: _decode(kvq, _args(), fmt=FMT_BF16))
    assert st == ERR_ARG and "k_cache" in msg


def test_write_argument_checks(kvq):
    n = 5
    k = torch.zeros((n, HKV, DH), dtype=torch.bfloat16)
    kc = torch.zeros((NB, HKV, 16, DH), dtype=torch.uint8)
    s = torch.ones(HKV, dtype=torch.float32)
    slots32 = torch.zeros(n, dtype=torch.int32)
    st, msg = _status(kvq, lambda: kvq.kvq_write(k, k, slots32, kc, kc, s, s, PER_HEAD,
                                                 FMT_E4M3))
    assert st == ERR_ARG and "slot_mapping" in msg
    short = torch.zeros(n - 1, dtype=torch.int64)
    st, msg = _status(kvq, lambda: kvq.kvq_write(k, k, short, kc, kc, s, s, PER_HEAD,
                                                 FMT_E4M3))
    assert st == ERR_SHAPE and "slot_mapping" in msg
    slots = torch.zeros(n, dtype=torch.int64)
    st, msg = _status(kvq, lambda: kvq.kvq_write(k, k, slots, kc, kc, s, s, PER_HEAD,
                                                 FMT_E4M3))
    assert st == ERR_ARG and "CUDA" in msg


def test_dequant_and_calibration_checks(kvq):
    kc = torch.zeros((NB, HKV, 16, DH), dtype=torch.uint8)
    s = torch.ones(HKV, dtype=torch.float32)
    f32 = torch.zeros(kc.shape, dtype=torch.float32)
    st, msg = _status(kvq, lambda: kvq.kvq_dequant_cache(kc, f32, s, PER_HEAD, FMT_E4M3))
    assert st == ERR_ARG and "dst_bf16" in msg
    k = torch.zeros((4, HKV, DH), dtype=torch.bfloat16)
    st, msg = _status(kvq, lambda: kvq.kvq_calibrate_scales(k, k, s.double(), s, PER_HEAD,
                                                            FMT_E4M3))
    assert st == ERR_ARG and "k_scale" in msg
