"""Helpers shared by the GPU parity tests: move the seeded workload inputs to
the device, run the library through its binding, and compare with the CPU
oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

# Attention tolerance, elementwise: |gpu - ref| <= ABS + REL * |ref|, with ref
# the float64 oracle over the same dequantized cache and gpu the bf16 output.
ABS_TOL, REL_TOL = 2e-3, 1e-2


def to_dev(a, dev="cuda"):
    """numpy -> device tensor; uint16 arrays hold bf16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def to_np(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_out_to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_attention(got, ref, what="", extra=0.0):
    """extra: a further absolute term of the bound, per element (broadcast)."""
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    bound = ABS_TOL + REL_TOL * np.abs(ref) + extra
    bad = ~(err <= bound)
    assert not bad.any(), (
        f"{what}: {int(bad.sum())} of {err.size} elements out of tolerance; "
        f"max abs err {np.nanmax(err):.3e}, worst ratio {np.nanmax(err / bound):.2f}")
    return float(err.max()) if err.size else 0.0


class DeviceLayer:
    """One workload layer resident on the GPU, with its paged caches."""

    def __init__(self, lay: workloads.Layer, dev="cuda", fill=0, token_head=False):
        import fp8_quantized_paged_gb300 as kvq
        self.kvq = kvq
        self.lay = lay
        st = lay.st
        self.dev = dev
        self.q = to_dev(lay.q, dev)
        self.k = to_dev(lay.k, dev)
        self.v = to_dev(lay.v, dev)
        self.slots = to_dev(st.slot_mapping, dev)
        self.bt = to_dev(st.block_tables, dev)
        self.sl = to_dev(st.seq_lens, dev)
        self.qs = to_dev(lay.q_scale, dev)
        self.ks = to_dev(lay.k_scale, dev)
        self.vs = to_dev(lay.v_scale, dev)
        self.kc = kvq.new_cache(st.num_blocks, lay.Hkv, lay.dh, lay.fmt, dev)
        self.vc = kvq.new_cache(st.num_blocks, lay.Hkv, lay.dh, lay.fmt, dev)
        self.kc.view(torch.uint8).fill_(fill)
        self.vc.view(torch.uint8).fill_(fill)
        # per-(token, head) scales: caches beside the pages, NaN bytes until written
        self.token_head = token_head
        self.ksc = self.vsc = None
        if token_head:
            self.ksc = kvq.new_scale_cache(st.num_blocks, lay.Hkv, dev)
            self.vsc = kvq.new_scale_cache(st.num_blocks, lay.Hkv, dev)
            self.ksc.view(torch.int32).fill_(-1)
            self.vsc.view(torch.int32).fill_(-1)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = kvq.new_workspace(lay.B, lay.Hq, lay.Hkv, lay.dh, dev)
        self.poison_workspace()
        self.out = torch.empty((lay.B, lay.Hq, lay.dh), dtype=torch.bfloat16, device=dev)

    def poison_workspace(self):
        """NaN bytes everywhere but the counters (which must stay zero), so a
        read of a partial slot nobody wrote shows up."""
        self.ws.fill_(0xFF)
        self.ws[: self.kvq.KVQ_WS_COUNTER_BYTES].zero_()

    def write(self, token_idx=None):
        lay = self.lay
        if token_idx is None:
            k, v, s = self.k, self.v, self.slots
        else:
            idx = torch.as_tensor(np.asarray(token_idx, np.int64), device=self.dev)
            k, v, s = self.k[idx], self.v[idx], self.slots[idx]
        if self.token_head:
            self.kvq.kvq_write_token_head(k, v, s, self.kc, self.vc, self.ksc, self.vsc, lay.fmt,
                                          dev_status=self.status)
            return
        self.kvq.kvq_write(k, v, s, self.kc, self.vc, self.ks, self.vs, lay.gran, lay.fmt,
                           dev_status=self.status)

    def decode(self, window=None, seq_lens=None, block_tables=None, flags=0):
        lay = self.lay
        th = self.token_head
        self.kvq.kvq_decode_attn(self.q, self.kc, self.vc,
                                 self.bt if block_tables is None else block_tables,
                                 self.sl if seq_lens is None else seq_lens, self.qs,
                                 self.ksc if th else self.ks, self.vsc if th else self.vs,
                                 self.kvq.KVQ_SCALE_PER_TOKEN_HEAD if th else lay.gran, lay.fmt,
                                 lay.window if window is None else window, self.ws, self.out,
                                 dev_status=self.status, flags=flags)
        return self.out

    def status_word(self):
        torch.cuda.synchronize()
        return int(self.status.item())


def oracle_caches(lay: workloads.Layer, token_idx=None, fill=0, token_head=False):
    """The oracle's caches; with token_head also its scale caches (NaN where
    unwritten, like the device ones): returns K, V or K, V, sK, sV."""
    st = lay.st
    K = oracle.new_cache(st.num_blocks, lay.Hkv, lay.bs, lay.dh, lay.fmt, fill)
    V = oracle.new_cache(st.num_blocks, lay.Hkv, lay.bs, lay.dh, lay.fmt, fill)
    if token_idx is None:
        k, v, s = lay.k, lay.v, st.slot_mapping
    else:
        k, v, s = lay.k[token_idx], lay.v[token_idx], st.slot_mapping[token_idx]
    if token_head:
        nan = np.frombuffer(np.uint32(0xFFFFFFFF).tobytes(), np.float32)[0]
        sK = oracle.new_scale_cache(st.num_blocks, lay.Hkv, lay.bs, nan)
        sV = oracle.new_scale_cache(st.num_blocks, lay.Hkv, lay.bs, nan)
        assert oracle.write(k, v, s, K, V, sK, sV, oracle.PER_TOKEN_HEAD, lay.fmt) == 0
        return K, V, sK, sV
    bad = oracle.write(k, v, s, K, V, lay.k_scale, lay.v_scale, lay.gran, lay.fmt)
    assert bad == 0
    return K, V


def oracle_decode(lay, K, V, pairs=None, window=None, seq_lens=None, block_tables=None,
                  q_fp8=False, scale_caches=None):
    """Oracle attention; scale_caches = (sK, sV) selects per-(token, head) scales."""
    st = lay.st
    ks, vs, gran = lay.k_scale, lay.v_scale, lay.gran
    if scale_caches is not None:
        ks, vs, gran = scale_caches[0], scale_caches[1], oracle.PER_TOKEN_HEAD
    return oracle.decode_attn(lay.q, K, V, st.block_tables if block_tables is None else block_tables,
                              st.seq_lens if seq_lens is None else seq_lens, ks, vs, gran,
                              lay.fmt,
                              lay.window if window is None else window, pairs=pairs,
                              q_scale=lay.q_scale if q_fp8 else None)


def prefill_p_bound(lay: workloads.Layer, cu_q) -> np.ndarray:
    """The FP8 prefill's extra error term, per (query token, query head, dim).

    Its probabilities reach the PV MMA as f16, each within 2^-12 (half an
    f16 ulp) of its value, so an output element sum_t p_t V_t[d] / l can
    be off by up to 2^-12 max_t |V_t[d]| beyond the accumulation's rounding.
    max_t runs over the sequence's tokens of the query head's KV head, from
    the bf16 inputs, times 1.125 for the FP8 rounding of V (half an E5M2
    ulp, relative)."""
    st = lay.st
    B = len(st.seq_lens)
    v = np.abs(workloads.bf16_bits_to_f32(lay.v)).astype(np.float64)  # [N, Hkv, dh]
    vmax = np.zeros((B, lay.Hkv, lay.dh))
    np.maximum.at(vmax, st.token_seq, v)
    G = lay.Hq // lay.Hkv
    cu_q = np.asarray(cu_q)
    seq_of_q = np.repeat(np.arange(B), np.diff(cu_q))
    per_q = np.repeat(vmax[seq_of_q], G, axis=1)  # [total_q, Hq, dh]
    return 1.125 * 2.0 ** -12 * per_q
