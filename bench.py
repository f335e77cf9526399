"""Benchmark of the FP8 paged KV-cache hot path on GB300.

Workload (the long-context case): one sequence of 32768 tokens, Hq=32,
Hkv=8, dh=128, block_size=16, 32 layers of independent seeded bf16 N(0,1)
K/V with per-head E4M3 scales (amax/448).  One step = the whole hot path over
all 32 layers: quantize-and-scatter all 32768 tokens of every layer into its
FP8 paged cache (2 GiB of cache in total), then one decode-attention step per
layer over that cache.  Every layer's cache is written before the first
decode, so a layer's pages are evicted from L2 by the other layers' traffic
(about 6 GiB per step, inputs far larger than the 129 MB L2).

Prints one JSON line.  ``value`` is the step's algorithmic HBM bytes (write
+ decode) over the device-timed step; the decode-attention and KV-write
figures of the metric are reported beside it, each from CUDA events around
its own calls.  ``--impl reference`` times the CPU oracle on the host cores
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = ("FP8 paged decode-attn HBM GB/s (% of GB300 peak); KV-write GB/s; KV tok/s")
CFG = 4
LAYERS = workloads.NUM_LAYERS[CFG]
HQ, HKV, DH = workloads.SHAPES[CFG]
SEQ = 32768
BS = 16
E = 1  # FP8 element bytes

# ---------------------------------------------------------------- algorithmic bytes


def write_bytes(n_tokens: int) -> int:
    """Per token: read bf16 K and V, write FP8 K and V, read its int64 slot."""
    return n_tokens * (2 * HKV * DH * 2 + 2 * HKV * DH * E + 8)


def decode_bytes(n_tokens: int, n_heads: int = HQ) -> int:
    """KV read of the attended tokens (all KV heads), Q read and O write (bf16),
    block-table entries, seq_len, scales."""
    kv_heads = max(1, n_heads * HKV // HQ)
    return (n_tokens * 2 * kv_heads * DH * E + n_heads * DH * 2 * 2
            + ((n_tokens + BS - 1) // BS) * 4 + 4 + 2 * HKV * 4)


def write_bytes_token_head(n_tokens: int) -> int:
    """The write with per-(token, head) scales: the same, plus the fp32 scale
    of every K and V row."""
    return write_bytes(n_tokens) + n_tokens * 2 * HKV * 4


def decode_bytes_token_head(n_tokens: int) -> int:
    """The decode with per-(token, head) scales: the 16 K and 16 V fp32 scales
    of every page read beside it instead of the per-head scales."""
    pages = (n_tokens + BS - 1) // BS
    return decode_bytes(n_tokens) - 2 * HKV * 4 + pages * HKV * 2 * BS * 4


def unfused_bytes(n_tokens: int) -> int:
    """The unfused path over a cache of n_tokens: the dequant reads the FP8 K
    and V and writes them as bf16, the bf16 decode reads them again (plus the
    decode's Q, O, tables and lengths)."""
    kv = n_tokens * 2 * HKV * DH
    return kv * (1 + 2) + decode_bytes(n_tokens) - n_tokens * 2 * HKV * DH * E + kv * 2 - 2 * HKV * 4


PREFILL_Q = 2048  # prefix-hit prefill: the last 2048 tokens of the 32768 are queries


def prefill_flops(n_q: int, seq: int) -> int:
    """QK^T and PV multiply-adds of the causal prefill of the last n_q of seq
    tokens: query j attends to seq - n_q + j + 1 tokens, 4 dh flops each per
    query head."""
    keys = n_q * (seq - n_q) + n_q * (n_q + 1) // 2
    return keys * HQ * DH * 4


STEP_WRITE_BYTES = LAYERS * write_bytes(SEQ)
STEP_DECODE_BYTES = LAYERS * decode_bytes(SEQ)
STEP_BYTES = STEP_WRITE_BYTES + STEP_DECODE_BYTES

WORKLOAD = {
    "workload": "long context: 1 seq x 32768 tokens, 32 layers, Hq=32 Hkv=8 dh=128 bs=16, "
                "FP8 E4M3 per-head scales; step = write all 32768 tokens of every layer, then "
                "one decode step per layer",
    "layers": LAYERS, "seqs": 1, "seq_len": SEQ, "num_q_heads": HQ, "num_kv_heads": HKV,
    "head_dim": DH, "block_size": BS, "kv_cache_dtype": "fp8_e4m3", "scales": "per-head amax/448",
    "l2": f"inputs larger than L2 (about {STEP_BYTES / 1e9:.1f} GB moved per step)",
}


def measured_tflops() -> float:
    """Dense bf16 tensor peak measured on this GPU model (burst), TFLOP/s."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return 1900.0


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# The source files each recorded kernel is built from (its translation units
# and the headers they include).
KERNEL_SOURCES = {
    "kvq_decode_attn": ["kvq_common.cuh", "kvq_host.h", "kvq_host.cu", "kvq_decode.cuh",
                        "kvq_decode.cu", "kvq_decode_variant.cu"],
    "kvq_write": ["kvq_common.cuh", "kvq_host.h", "kvq_host.cu", "kvq_write.cu"],
}


def _header_code(path: str) -> bytes:
    """The C header without its comments and blank lines: its documentation
    does not change the kernels."""
    with open(path) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    lines = (re.sub(r"//.*", "", ln).strip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln).encode()


def kernel_source_hash(kernel: str) -> str:
    """Hash of one kernel's sources (and the C header's code), so that a
    recorded capture goes stale only when that kernel's code changes."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_quantized_paged_gb300", "csrc")
    for n in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode() + f.read())
    h.update(b"kvq.h" + _header_code(os.path.join(ROOT, "include", "kvq.h")))
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        k = d["kernels"][kernel]
        if k.get("source_hash") != kernel_source_hash(kernel):
            return None
        return k["bytes_per_launch"]
    except Exception:
        return None


# ---------------------------------------------------------------- ranks


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Slowest rank's value (the job's time) via an all-reduce MAX."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_rank_step: int, ms_per_step: float) -> float:
    """Weak scaling: every rank moves the same bytes per step; the job's time
    per step is the slowest rank's."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------- inputs


def make_inputs(n_layers: int):
    st = workloads.structure(CFG)
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        layers = list(ex.map(lambda l: workloads.make_layer(CFG, l, st=st), range(n_layers)))
    return st, layers


# ---------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


# ---------------------------------------------------------------- GPU arm


def run_gpu(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import fp8_quantized_paged_gb300 as kvq

    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    st, layers = make_inputs(LAYERS)
    stream = torch.cuda.current_stream()

    def up(a, pin=False):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(a)
        return t.pin_memory() if pin else t.to(dev)

    slots = up(st.slot_mapping)
    bt = up(st.block_tables)
    sl = up(st.seq_lens)
    L = []
    for lay in layers:
        L.append(dict(k=up(lay.k), v=up(lay.v), q=up(lay.q), qs=up(lay.q_scale), ks=up(lay.k_scale),
                      vs=up(lay.v_scale),
                      kc=kvq.new_cache(st.num_blocks, HKV, DH, kvq.KVQ_FMT_E4M3, dev),
                      vc=kvq.new_cache(st.num_blocks, HKV, DH, kvq.KVQ_FMT_E4M3, dev),
                      out=torch.empty((1, HQ, DH), dtype=torch.bfloat16, device=dev)))
    ws = kvq.new_workspace(1, HQ, HKV, DH, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    E4, PH = kvq.KVQ_FMT_E4M3, kvq.KVQ_SCALE_PER_HEAD
    launches_per_step = LAYERS * 2  # one write and one decode kernel per layer

    def writes():
        for x in L:
            kvq.kvq_write(x["k"], x["v"], slots, x["kc"], x["vc"], x["ks"], x["vs"], PH, E4,
                          dev_status=status)

    def decodes(flags=0):
        for x in L:
            kvq.kvq_decode_attn(x["q"], x["kc"], x["vc"], bt, sl, x["qs"], x["ks"], x["vs"], PH,
                                E4, 0, ws, x["out"], dev_status=status, flags=flags)

    # eager warm-up (first calls configure the kernels), then one CUDA graph
    # for the 32 writes and one for the 32 decodes: the step replays both.
    for _ in range(max(args.warmup, 3)):
        writes()
        decodes()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    g_write, g_decode = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    g_decode_ready = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_write):
        writes()
    with torch.cuda.graph(g_decode):
        decodes()
    # The same decodes allowed to start before the previous layer's kernels end
    # (the caches, tables and lengths are complete before the decode graph).
    with torch.cuda.graph(g_decode_ready):
        decodes(kvq.KVQ_CACHE_READY)
    # The FP8-domain query mode: Q quantized with its per-head scale, QK^T on
    # FP8 codes.
    decodes(kvq.KVQ_Q_FP8)
    g_decode_qf8 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_decode_qf8):
        decodes(kvq.KVQ_Q_FP8)
    # Per-head scale calibration of every layer's K/V (into scratch scales).
    cal_k = torch.empty(HKV, dtype=torch.float32, device=dev)
    cal_v = torch.empty(HKV, dtype=torch.float32, device=dev)

    def calibrations():
        for x in L:
            kvq.kvq_calibrate_scales(x["k"], x["v"], cal_k, cal_v, PH, E4, dev_status=status)

    calibrations()
    g_calib = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_calib):
        calibrations()
    # Prefix-hit prefill on layer 0's cache: the last PREFILL_Q tokens are
    # queries over the 32768 cached ones (4 calls per graph replay).
    pf_q = torch.randn((PREFILL_Q, HQ, DH), device=dev).to(torch.bfloat16)
    pf_out = torch.empty_like(pf_q)
    pf_cu = torch.tensor([0, PREFILL_Q], dtype=torch.int32, device=dev)

    def prefills():
        for _ in range(4):
            kvq.kvq_prefill_attn(pf_q, pf_cu, PREFILL_Q, L[0]["kc"], L[0]["vc"], bt, sl,
                                 L[0]["ks"], L[0]["vs"], PH, E4, 0, pf_out, dev_status=status)

    prefills()
    g_prefill = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_prefill):
        prefills()
    # The unfused path the fused decode replaces: every layer's FP8 caches
    # dequantized into one bf16 scratch pair, then the bf16 decode over it.
    kb = torch.empty(L[0]["kc"].shape, dtype=torch.bfloat16, device=dev)
    vb = torch.empty(L[0]["vc"].shape, dtype=torch.bfloat16, device=dev)

    def unfused():
        for x in L:
            kvq.kvq_dequant_cache(x["kc"], kb, x["ks"], PH, E4)
            kvq.kvq_dequant_cache(x["vc"], vb, x["vs"], PH, E4)
            kvq.kvq_decode_attn(x["q"], kb, vb, bt, sl, None, None, None, 0, kvq.KVQ_FMT_BF16, 0,
                                ws, x["out"], dev_status=status)

    unfused()
    g_unfused = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_unfused):
        unfused()
    # Per-(token, head) scales: every layer's write into the same caches with
    # its scale caches beside them, then the decodes reading them.  Timed
    # after the per-head graphs (it rewrites the caches).
    for x in L:
        x["ksc"] = kvq.new_scale_cache(st.num_blocks, HKV, dev)
        x["vsc"] = kvq.new_scale_cache(st.num_blocks, HKV, dev)

    def writes_th():
        for x in L:
            kvq.kvq_write_token_head(x["k"], x["v"], slots, x["kc"], x["vc"], x["ksc"], x["vsc"],
                                     E4, dev_status=status)

    def decodes_th():
        for x in L:
            kvq.kvq_decode_attn(x["q"], x["kc"], x["vc"], bt, sl, None, x["ksc"], x["vsc"],
                                kvq.KVQ_SCALE_PER_TOKEN_HEAD, E4, 0, ws, x["out"],
                                dev_status=status)

    g_write_th, g_decode_th = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_write_th):
        writes_th()
    with torch.cuda.graph(g_decode_th):
        decodes_th()
    stream = torch.cuda.current_stream()

    def step(_timed=False):
        g_write.replay()
        g_decode.replay()

    def timed_replays(fn, n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def rank_max(x):
        return max_over_ranks(x, world, dev)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    # ---- device-resident timed region: whole steps, then each graph alone
    barrier()
    with ClockSampler(torch.cuda.current_device()) as clk:
        total_ms = timed_replays(step, args.steps)
        write_total = timed_replays(g_write.replay, args.steps)
        decode_total = timed_replays(g_decode.replay, args.steps)
        ready_total = timed_replays(g_decode_ready.replay, args.steps)
        qf8_total = timed_replays(g_decode_qf8.replay, args.steps)
        calib_total = timed_replays(g_calib.replay, args.steps)
        prefill_total = timed_replays(g_prefill.replay, args.steps)
        unfused_total = timed_replays(g_unfused.replay, args.steps)
        g_write_th.replay()  # the caches now hold per-token-head codes
        g_decode_th.replay()
        write_th_total = timed_replays(g_write_th.replay, args.steps)
        decode_th_total = timed_replays(g_decode_th.replay, args.steps)
    barrier()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    ms_step = rank_max(total_ms) / args.steps
    write_ms = rank_max(write_total) / args.steps
    decode_ms = rank_max(decode_total) / args.steps
    ready_ms = rank_max(ready_total) / args.steps
    qf8_ms = rank_max(qf8_total) / args.steps
    calib_ms = rank_max(calib_total) / args.steps
    write_th_us = rank_max(write_th_total) / args.steps * 1e3 / LAYERS
    prefill_us = rank_max(prefill_total) / args.steps * 1e3 / 4
    decode_th_us = rank_max(decode_th_total) / args.steps * 1e3 / LAYERS
    unfused_us = rank_max(unfused_total) / args.steps * 1e3 / LAYERS

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(args, kvq, torch, dist, dev, st, layers, L, ws, status, world, barrier,
                  rank_max)
    # ---- the other workloads' layers (not part of the step)
    configs = None
    if not args.no_configs:
        with ClockSampler(torch.cuda.current_device()) as clk_cfg:
            configs = run_configs(kvq, torch, dev, measured_peaks()[0], max(5, args.steps // 5))
        configs["clocks"] = clk_cfg.summary()

    peak, peak_src = measured_peaks()
    write_launch_us = write_ms * 1e3 / LAYERS
    decode_launch_us = decode_ms * 1e3 / LAYERS
    w_ach = write_bytes(SEQ) / (write_launch_us * 1e-6) / 1e9
    d_ach = decode_bytes(SEQ) / (decode_launch_us * 1e-6) / 1e9
    ready_launch_us = ready_ms * 1e3 / LAYERS
    r_ach = decode_bytes(SEQ) / (ready_launch_us * 1e-6) / 1e9
    qf8_launch_us = qf8_ms * 1e3 / LAYERS
    q_ach = decode_bytes(SEQ) / (qf8_launch_us * 1e-6) / 1e9
    calib_launch_us = calib_ms * 1e3 / LAYERS
    c_ach = SEQ * 2 * HKV * DH * 2 / (calib_launch_us * 1e-6) / 1e9  # bf16 K and V read once

    def roof(name, ach, per_launch_bytes):
        return {"kernel": name, "bound": "hbm", "achieved": round(ach, 1), "peak": peak,
                "unit": "GB/s", "frac": round(ach / peak, 4), "peak_source": peak_src,
                "algorithmic_bytes_per_launch": per_launch_bytes,
                "traffic": recorded_traffic(name)}

    dominant = "kvq_write" if write_ms >= decode_ms else "kvq_decode_attn"
    res = {
        "metric": METRIC,
        "value": round(whole_job_gbs(world, STEP_BYTES, ms_step), 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3 cache, f16 MMA / f32 accumulate",
        "data": "synthetic (seeded N(0,1) bf16 K/V/Q, per-head amax/448 scales)",
        "config": dict(WORKLOAD, parallelism=f"replicas x{world}" if world > 1 else "1 GPU"),
        "decode_attn": {"gbs": round(d_ach, 1), "frac_of_peak": round(d_ach / peak, 4),
                        "us_per_layer": round(decode_launch_us, 2),
                        "kv_tok_s": round(SEQ / (decode_launch_us * 1e-6), 0)},
        "decode_attn_cache_ready": {"gbs": round(r_ach, 1), "frac_of_peak": round(r_ach / peak, 4),
                                    "us_per_layer": round(ready_launch_us, 2),
                                    "flags": "KVQ_CACHE_READY"},
        "decode_attn_q_fp8": {"gbs": round(q_ach, 1), "frac_of_peak": round(q_ach / peak, 4),
                              "us_per_layer": round(qf8_launch_us, 2), "flags": "KVQ_Q_FP8"},
        "kv_calibrate": {"gbs": round(c_ach, 1), "frac_of_peak": round(c_ach / peak, 4),
                         "us_per_layer": round(calib_launch_us, 2),
                         "what": "per-head amax scales of one layer's 32768 bf16 K/V tokens"},
        "prefill_attn": {
            "tflops": round(prefill_flops(PREFILL_Q, SEQ) / (prefill_us * 1e-6) / 1e12, 1),
            "us_per_call": round(prefill_us, 1),
            "frac_of_bf16_peak": round(prefill_flops(PREFILL_Q, SEQ) / (prefill_us * 1e-6) / 1e12
                                       / measured_tflops(), 4),
            "what": "prefix-hit prefill of layer 0: last 2048 of 32768 tokens as causal queries "
                    "(Hq=32, Hkv=8, dh=128, FP8 E4M3), tcgen05 f16 MMA, accumulators in TMEM"},
        "kv_write_token_head": {
            "gbs": round(write_bytes_token_head(SEQ) / (write_th_us * 1e-6) / 1e9, 1),
            "frac_of_peak": round(write_bytes_token_head(SEQ) / (write_th_us * 1e-6) / 1e9 / peak, 4),
            "us_per_layer": round(write_th_us, 2),
            "what": "kvq_write_token_head: per-(token, head) amax scales stored beside the pages"},
        "decode_attn_token_head": {
            "gbs": round(decode_bytes_token_head(SEQ) / (decode_th_us * 1e-6) / 1e9, 1),
            "frac_of_peak": round(decode_bytes_token_head(SEQ) / (decode_th_us * 1e-6) / 1e9 / peak, 4),
            "us_per_layer": round(decode_th_us, 2),
            "what": "decode reading the per-(token, head) scale caches"},
        "kv_write": {"gbs": round(w_ach, 1), "frac_of_peak": round(w_ach / peak, 4),
                     "us_per_layer": round(write_launch_us, 2),
                     "tok_s": round(SEQ / (write_launch_us * 1e-6), 0)},
        "kv_tok_s": round(world * SEQ * LAYERS / (decode_ms * 1e-3), 0),
        "roofline": roof(dominant, w_ach if dominant == "kvq_write" else d_ach,
                         write_bytes(SEQ) if dominant == "kvq_write" else decode_bytes(SEQ)),
        "roofline_decode": roof("kvq_decode_attn", d_ach, decode_bytes(SEQ)),
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "decode_unfused_ablation": {
            "us_per_layer": round(unfused_us, 2),
            "vs_fused": round(unfused_us / (decode_ms * 1e3 / LAYERS), 3),
            "hbm_bytes_per_layer": unfused_bytes(SEQ),
            "what": "kvq_dequant_cache of K and V into one bf16 scratch cache, then the bf16 "
                    "decode over it: FP8 read, bf16 written and read again (the scratch is "
                    "about the L2's size, so part of the re-read hits L2)"},
        "timing": "CUDA graphs (32 writes, 32 decodes) replayed; events on the replay stream; "
                  "per-kernel figures from replaying each graph alone; decode_attn_cache_ready "
                  "replays the 32 decodes with KVQ_CACHE_READY, decode_attn_q_fp8 with "
                  "KVQ_Q_FP8, kv_calibrate 32 scale calibrations, kv_write_token_head and "
                  "decode_attn_token_head the per-(token, head) scale mode, "
                  "decode_unfused_ablation 32 dequant + bf16 decode layers (none part of the "
                  "step)",
        "clocks": clk.summary(),
    }
    if configs is not None:
        res["configs"] = configs
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(layers[0], st, args.cpu_seconds)
    return res


def run_e2e(args, kvq, torch, dist, dev, st, layers, L, ws, status, world, barrier,
            rank_max):
    """Host buffers in, host result out: per step, copy every layer's K/V/Q from
    pinned host memory (copy stream, one event per layer), run the same calls,
    read the outputs back.  A layer's next copy waits only for the kernels of
    the previous step that read its buffers, so the copy stream never idles
    behind a whole step."""
    hk = [torch.from_numpy(np.ascontiguousarray(l.k).view(np.int16)).pin_memory() for l in layers]
    hv = [torch.from_numpy(np.ascontiguousarray(l.v).view(np.int16)).pin_memory() for l in layers]
    hq = [torch.from_numpy(np.ascontiguousarray(l.q).view(np.int16)).pin_memory() for l in layers]
    hslot = torch.from_numpy(st.slot_mapping).pin_memory()
    hout = torch.empty((LAYERS, HQ, DH), dtype=torch.int16).pin_memory()
    slot_d = torch.empty_like(hslot, device=dev)
    bt = torch.from_numpy(st.block_tables).to(dev)
    sl = torch.from_numpy(st.seq_lens).to(dev)
    comp = torch.cuda.current_stream()
    copies = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]  # layers alternate
    E4, PH = kvq.KVQ_FMT_E4M3, kvq.KVQ_SCALE_PER_HEAD
    ready = [torch.cuda.Event() for _ in range(LAYERS)]
    written = [torch.cuda.Event() for _ in range(LAYERS)]   # layer's K/V consumed
    decoded = [torch.cuda.Event() for _ in range(LAYERS)]   # layer's Q consumed
    for i in range(LAYERS):
        written[i].record(comp)
        decoded[i].record(comp)
    h2d = sum(x.numel() * 2 for x in hk + hv + hq) + hslot.numel() * 8
    d2h = hout.numel() * 2

    def copy_in():
        with torch.cuda.stream(copies[0]):
            copies[0].wait_event(written[LAYERS - 1])  # every write of the last step read the slots
            slot_d.copy_(hslot, non_blocking=True)
        for i, x in enumerate(L):
            cs = copies[i % 2]
            with torch.cuda.stream(cs):
                cs.wait_event(written[i])
                x["k"].view(torch.int16).copy_(hk[i], non_blocking=True)
                x["v"].view(torch.int16).copy_(hv[i], non_blocking=True)
                cs.wait_event(decoded[i])
                x["q"].view(torch.int16).copy_(hq[i], non_blocking=True)
                ready[i].record(cs)

    def step():
        copy_in()
        for i, x in enumerate(L):
            comp.wait_event(ready[i])
            kvq.kvq_write(x["k"], x["v"], slot_d, x["kc"], x["vc"], x["ks"], x["vs"], PH, E4,
                          dev_status=status)
            written[i].record(comp)
        for i, x in enumerate(L):
            kvq.kvq_decode_attn(x["q"], x["kc"], x["vc"], bt, sl, None, x["ks"], x["vs"], PH, E4,
                                0, ws, x["out"], dev_status=status)
            decoded[i].record(comp)
        for i, x in enumerate(L):
            hout[i].copy_(x["out"][0].view(torch.int16), non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    n = max(2, min(args.steps, args.e2e_steps))
    barrier()
    t = time.perf_counter()
    for _ in range(n):
        step()
    torch.cuda.synchronize()
    el = rank_max(time.perf_counter() - t)
    # the host-to-device copies alone (both streams, no kernels): the bound of this number
    for _ in range(2):
        copy_in()
    torch.cuda.synchronize()
    t = time.perf_counter()
    for _ in range(n):
        copy_in()
    torch.cuda.synchronize()
    el_h2d = rank_max(time.perf_counter() - t)
    return {"value": round(whole_job_gbs(world, STEP_BYTES, el * 1e3 / n), 1), "unit": "GB/s",
            "ms_per_step": round(el * 1e3 / n, 3), "steps": n,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "copy_streams": len(copies),
            "h2d_gbs": round(world * h2d * n / el_h2d / 1e9, 1),
            "h2d_only_ms_per_step": round(el_h2d * 1e3 / n, 3),
            "what": "per step: every layer's K/V/Q copied from pinned host memory on two copy "
                    "streams (layers alternate), the 32 writes and 32 decodes, the outputs read "
                    "back; h2d_gbs times the same copies alone"}


# ---------------------------------------------------------------- the other workloads

L2_BYTES = 129 * 1024 * 1024


def layer_bytes(st, Hq, Hkv, dh, fmt, gran, window):
    """Algorithmic bytes of one layer's write (every token) and decode (the
    attended tokens of every sequence): as write_bytes / decode_bytes, with the
    layer's own shape, cache element size and window."""
    elem = 2 if fmt == workloads.BF16 else 1
    lens = st.seq_lens.astype(np.int64)
    B = len(lens)
    lo = np.where((window > 0) & (lens > window), lens - window, 0)
    attended = int((lens - lo).sum())
    pages = int(((lens + BS - 1) // BS - lo // BS).sum())
    tokens = int(lens.sum())
    nsc = 0 if fmt == workloads.BF16 else 2 * (Hkv if gran == workloads.PER_HEAD else 1)
    write = tokens * (2 * Hkv * dh * 2 + 2 * Hkv * dh * elem + 8)
    decode = (attended * 2 * Hkv * dh * elem + B * Hq * dh * 2 * 2 + pages * 4 + B * 4 + nsc * 4)
    return write, decode, attended, tokens


def run_configs(kvq, torch, dev, peak, steps):
    """Workloads 2, 3 (E4M3 and E5M2) and 5 (an FP8 layer and a bf16 window
    layer), one layer each: its write of every token and its decode, each as a
    CUDA graph over enough copies of the caches that one replay moves more than
    4x the L2 (the next call never finds its pages in L2), replayed `steps`
    times.  Lengths, block tables, shapes, formats and scale granularities are
    the workloads'; the seeded bf16 K/V/Q are drawn on the device in each
    workload's recipe (N(0,1); workload 2 with four x10 outlier channels per KV
    head in K, workload 3 with per-head standard deviations log-uniform in
    [0.1, 10]) and the scales computed from them by kvq_calibrate_scales
    (amax / the format's largest value), since only timings come out of it."""
    cases = [("workload2_llama8b_e4m3", 2, 0, workloads.E4M3),
             ("workload3_per_head_e4m3", 3, 0, workloads.E4M3),
             ("workload3_per_head_e5m2", 3, 0, workloads.E5M2),
             ("workload5_fp8_layer", 5, 2, workloads.E4M3),
             ("workload5_bf16_window_layer", 5, 3, workloads.E4M3)]
    stream = torch.cuda.current_stream()
    out = {}
    structures = {}
    for name, cfg, layer, fmt3 in cases:
        st = structures.setdefault(cfg, workloads.structure(cfg))
        Hq, Hkv, dh = workloads.SHAPES[cfg]
        fmt, gran, window = workloads.layer_format(cfg, layer, fmt3)
        wb, db, attended, tokens = layer_bytes(st, Hq, Hkv, dh, fmt, gran, window)
        B = len(st.seq_lens)
        elem = 2 if fmt == workloads.BF16 else 1
        kv = tokens * 2 * Hkv * dh * elem
        n = max(1, -(-4 * L2_BYTES // kv))
        gen = torch.Generator(device=dev)
        gen.manual_seed(1000 * cfg + layer)
        k = torch.randn((tokens, Hkv, dh), generator=gen, device=dev)
        v = torch.randn((tokens, Hkv, dh), generator=gen, device=dev)
        if cfg == 2:
            for h in range(Hkv):
                ch = torch.randperm(dh, generator=gen, device=dev)[:4]
                k[:, h, ch] *= 10.0
        elif cfg == 3:
            lo_, hi_ = np.log(0.1), np.log(10.0)
            sk = torch.exp(lo_ + (hi_ - lo_) * torch.rand(Hkv, generator=gen, device=dev))
            sv = torch.exp(lo_ + (hi_ - lo_) * torch.rand(Hkv, generator=gen, device=dev))
            k *= sk[None, :, None]
            v *= sv[None, :, None]
        k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
        q = torch.randn((B, Hq, dh), generator=gen, device=dev).to(torch.bfloat16)
        nsc = Hkv if gran == workloads.PER_HEAD else 1
        ks = torch.ones(nsc, dtype=torch.float32, device=dev)
        vs = torch.ones(nsc, dtype=torch.float32, device=dev)
        if fmt != workloads.BF16:
            kvq.kvq_calibrate_scales(k, v, ks, vs, gran, fmt)
        slots = torch.from_numpy(st.slot_mapping).to(dev)
        bt = torch.from_numpy(st.block_tables).to(dev)
        sl = torch.from_numpy(st.seq_lens).to(dev)
        caches = [(kvq.new_cache(st.num_blocks, Hkv, dh, fmt, dev),
                   kvq.new_cache(st.num_blocks, Hkv, dh, fmt, dev)) for _ in range(n)]
        ws = kvq.new_workspace(B, Hq, Hkv, dh, dev)
        o = torch.empty((B, Hq, dh), dtype=torch.bfloat16, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)

        def writes():
            for kc, vc in caches:
                kvq.kvq_write(k, v, slots, kc, vc, ks, vs, gran, fmt, dev_status=status)

        def decodes():
            for kc, vc in caches:
                kvq.kvq_decode_attn(q, kc, vc, bt, sl, None, ks, vs, gran, fmt, window, ws, o,
                                    dev_status=status)

        writes()
        decodes()
        torch.cuda.synchronize()
        gw, gd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(gw):
            writes()
        with torch.cuda.graph(gd):
            decodes()

        def timed(g):
            for _ in range(3):
                g.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(steps):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) * 1e3 / (steps * n)

        w_us, d_us = timed(gw), timed(gd)
        assert int(status.item()) == 0, f"{name}: device status {int(status.item())}"
        w_gbs, d_gbs = wb / (w_us * 1e-6) / 1e9, db / (d_us * 1e-6) / 1e9
        out[name] = {
            "workload": cfg, "layer": layer, "seqs": B, "tokens": tokens,
            "cache": {workloads.E4M3: "fp8_e4m3", workloads.E5M2: "fp8_e5m2",
                      workloads.BF16: "bf16"}[fmt],
            "scales": "per-head" if gran == workloads.PER_HEAD else "per-tensor",
            "window": window, "cache_copies_rotated": n,
            "decode_attn": {"us_per_layer": round(d_us, 2), "gbs": round(d_gbs, 1),
                            "frac_of_peak": round(d_gbs / peak, 4),
                            "kv_tok_s": round(attended / (d_us * 1e-6), 0),
                            "algorithmic_bytes": db},
            "kv_write": {"us_per_layer": round(w_us, 2), "gbs": round(w_gbs, 1),
                         "frac_of_peak": round(w_gbs / peak, 4),
                         "tok_s": round(tokens / (w_us * 1e-6), 0), "algorithmic_bytes": wb}}
        del caches, k, v, q, gw, gd
        torch.cuda.synchronize()
    return out


# ---------------------------------------------------------------- CPU oracle


def oracle_sample_step(lay, st, n_write_tokens, heads):
    """One bounded sample of the workload on the CPU oracle: quantize-and-scatter
    the first n_write_tokens tokens of the layer, and decode `heads` query heads
    over the layer's full 32768-token cache.  Returns algorithmic bytes."""
    import oracle
    K = np.zeros((st.num_blocks, HKV, BS, DH), np.uint8)
    V = np.zeros_like(K)
    # the decode reads a fully written cache: write every token once (untimed
    # by the caller only in the sense that it is counted as write bytes)
    oracle.write(lay.k[:n_write_tokens], lay.v[:n_write_tokens], st.slot_mapping[:n_write_tokens],
                 K, V, lay.k_scale, lay.v_scale, lay.gran, lay.fmt)
    pairs = np.array([[0, h] for h in heads], np.int32)
    oracle.decode_attn(lay.q, K, V, st.block_tables, st.seq_lens, lay.k_scale, lay.v_scale,
                       lay.gran, lay.fmt, pairs=pairs)
    return write_bytes(n_write_tokens) + decode_bytes(SEQ, len(heads))


def cpu_baseline(lay, st, seconds):
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    done_bytes, t0, reps = 0, time.perf_counter(), 0
    while True:
        done_bytes += oracle_sample_step(lay, st, SEQ, range(HQ))
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    return {"value": round(done_bytes / el / 1e9, 3), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{reps} x one layer of the workload (write 32768 tokens, decode 32 heads "
                      f"over 32768 tokens), float64 attention, OpenMP on {cores} threads, "
                      f"{el:.1f} s"}


def run_reference(args):
    """The oracle as the reference arm, on the host cores."""
    import oracle
    oracle.build()
    st = workloads.structure(CFG)
    lay = workloads.make_layer(CFG, 0, st=st)
    cores = oracle.max_threads()
    n_tok, heads = 4096, range(4)  # bounded per-step sample
    for _ in range(max(args.warmup, 1)):
        oracle_sample_step(lay, st, n_tok, heads)
    t = time.perf_counter()
    tot = 0
    for _ in range(args.steps):
        tot += oracle_sample_step(lay, st, n_tok, heads)
    el = time.perf_counter() - t
    v = round(tot / el / 1e9, 4)
    sample = (f"per step: write 4096 tokens of one layer and decode 4 query heads over the "
              f"32768-token cache (float64 oracle, OpenMP on {cores} threads)")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": 0,
            "steps": args.steps, "warmup": max(args.warmup, 1),
            "ms_per_step": round(el * 1e3 / args.steps, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": WORKLOAD,
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- main


def run_ncu_case(case: str):
    """A few launches of one kernel for ncu captures (ncu flushes the caches
    before each captured launch): 'decode' and 'write' run one FP8 layer of
    the mixed skip-layer batch (128 sequences, about 0.9 GB of FP8 cache),
    'decode_long' and 'write_long' one layer of the long-context workload
    (32768 tokens: 128 MiB of bf16 K/V in, 64 MiB of FP8 cache); on that
    layer 'write_th_long' / 'decode_th_long' use per-(token, head) scales,
    'calib_long' calibrates per-head scales and 'prefill_long' runs the
    bench's prefix-hit prefill (the last 2048 tokens as queries)."""
    import torch

    import fp8_quantized_paged_gb300 as kvq
    cfg, layer = (4, 0) if case.endswith("_long") else (5, 2)
    lay = workloads.make_layer(cfg, layer)
    st = lay.st
    dev = torch.device("cuda:0")

    def up(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    k, v, q = up(lay.k), up(lay.v), up(lay.q)
    slots, bt, sl = up(st.slot_mapping), up(st.block_tables), up(st.seq_lens)
    ks, vs = up(lay.k_scale), up(lay.v_scale)
    kc = kvq.new_cache(st.num_blocks, lay.Hkv, lay.dh, lay.fmt, dev)
    vc = kvq.new_cache(st.num_blocks, lay.Hkv, lay.dh, lay.fmt, dev)
    ws = kvq.new_workspace(lay.B, lay.Hq, lay.Hkv, lay.dh, dev)
    out = torch.empty((lay.B, lay.Hq, lay.dh), dtype=torch.bfloat16, device=dev)
    token_head = "_th" in case
    n_write = 3 if case.startswith("write") else 1
    if token_head:
        ksc = kvq.new_scale_cache(st.num_blocks, lay.Hkv, dev)
        vsc = kvq.new_scale_cache(st.num_blocks, lay.Hkv, dev)
        for _ in range(n_write):
            kvq.kvq_write_token_head(k, v, slots, kc, vc, ksc, vsc, lay.fmt)
        ks, vs, gran = ksc, vsc, kvq.KVQ_SCALE_PER_TOKEN_HEAD
    else:
        gran = lay.gran
        for _ in range(n_write):
            kvq.kvq_write(k, v, slots, kc, vc, ks, vs, lay.gran, lay.fmt)
    for _ in range(3 if case.startswith("decode") else 0):
        kvq.kvq_decode_attn(q, kc, vc, bt, sl, None, ks, vs, gran, lay.fmt, lay.window, ws, out)
    if case == "calib_long":
        cal_k = torch.empty(lay.Hkv, dtype=torch.float32, device=dev)
        cal_v = torch.empty(lay.Hkv, dtype=torch.float32, device=dev)
        for _ in range(3):
            kvq.kvq_calibrate_scales(k, v, cal_k, cal_v, kvq.KVQ_SCALE_PER_HEAD, lay.fmt)
    if case == "prefill_long":
        nq = 2048
        pq = torch.randn((nq, lay.Hq, lay.dh), device=dev).to(torch.bfloat16)
        pout = torch.empty_like(pq)
        cu = torch.tensor([0, nq], dtype=torch.int32, device=dev)
        for _ in range(2):
            kvq.kvq_prefill_attn(pq, cu, nq, kc, vc, bt, sl, ks, vs, lay.gran, lay.fmt, 0, pout)
    torch.cuda.synchronize()
    print(json.dumps({"ncu_case": case, "workload": cfg, "layer": layer,
                      "kv_tokens": int(st.seq_lens.sum()), "decode_bytes": int(st.seq_lens.sum()) * 2048}))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-layer lines of workloads 2, 3 and 5")
    ap.add_argument("--ncu-case", choices=["decode", "write", "decode_long", "write_long",
                                           "write_th_long", "decode_th_long", "calib_long",
                                           "prefill_long"], default=None,
                    help="run a few launches of one kernel for an ncu capture, then exit")
    args = ap.parse_args()
    if args.ncu_case:
        run_ncu_case(args.ncu_case)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    res = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
