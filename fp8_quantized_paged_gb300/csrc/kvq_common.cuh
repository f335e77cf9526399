// kvq_common.cuh -- shared device helpers of libkvq (sm_103a).
//
// Thin inline-PTX wrappers: mbarrier, TMA tile loads, warp-level MMA and the
// FP8 <-> f16 / f32 conversions.  Written for Blackwell (sm_103a) only.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

#define KVQ_DEVI __device__ __forceinline__

namespace kvq {

// Upper bound on the polls of one mbarrier wait (each poll is a try_wait
// that itself suspends for a hardware-chosen time).  A wait that exhausts it
// reports KVQ_DEV_WAIT_TIMEOUT instead of hanging.
// (A build may lower it with -DKVQ_MAX_POLLS, as the tests' timeout build does.)
#ifndef KVQ_MAX_POLLS
#define KVQ_MAX_POLLS (1u << 22)
#endif
constexpr uint32_t kMaxPolls = KVQ_MAX_POLLS;

KVQ_DEVI uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

KVQ_DEVI void flag_status(uint32_t* st, uint32_t bit) {
  if (st) atomicOr(st, bit);
}

// Internal consistency guards: an index that should be in range by
// construction is checked anyway; a failed guard sets bit 16 + id of the
// status word and the access is skipped.
KVQ_DEVI bool guard(bool ok, uint32_t* st, int id) {
  if (!ok) flag_status(st, KVQ_DEV_INTERNAL | (1u << (16 + id)));
  return ok;
}

// ------------------------------------------------------------------ mbarrier

KVQ_DEVI void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

KVQ_DEVI void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

KVQ_DEVI void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

KVQ_DEVI void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

KVQ_DEVI bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test for completion of the phase of the given parity.
KVQ_DEVI bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of the given parity; false when it ran out.
KVQ_DEVI bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kMaxPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// ------------------------------------------------------------------ PDL
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel on the stream drains;
// it must wait for that kernel's completion (and memory) before touching any
// data another kernel may have written.
KVQ_DEVI void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
KVQ_DEVI void pdl_allow_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ TMA

KVQ_DEVI void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

KVQ_DEVI void tma_load_2d(void* dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// An L2 policy that marks the lines a load brings in as first to evict: for
// data read once (a stream that would otherwise push everything else out).
KVQ_DEVI uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

KVQ_DEVI void tma_load_2d_hint(void* dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

KVQ_DEVI void tma_load_3d(void* dst, const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2,
                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Untiled bulk copy global -> shared, completion counted in bytes on bar.
// Both addresses 16-byte aligned, bytes a multiple of 16.
KVQ_DEVI void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Orders this thread's earlier generic-proxy accesses (and what it has
// acquired from other threads) before its later async-proxy accesses.
KVQ_DEVI void fence_proxy_async() { asm volatile("fence.proxy.async;" ::: "memory"); }
KVQ_DEVI void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
KVQ_DEVI void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ MMA (m16n8k16, fp32 accumulate)

KVQ_DEVI void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

KVQ_DEVI void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// m16n8k32 with 8-bit float operands, A and B both in format FMT.
template <int FMT>
KVQ_DEVI void mma_fp8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if (FMT == KVQ_FMT_E4M3)
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e5m2.e5m2.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ conversions

// Two FP8 codes (low byte -> low half) to f16x2.  Exact: every E4M3 and E5M2
// value is representable in binary16.
template <int FMT>
KVQ_DEVI uint32_t fp8x2_to_f16x2(uint16_t two) {
  uint32_t r;
  if (FMT == KVQ_FMT_E4M3)
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  else
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(r) : "h"(two));
  return r;
}

// Four FP8 codes of one word to two f16x2 (bytes 0,1 -> lo; bytes 2,3 -> hi).
template <int FMT>
KVQ_DEVI void fp8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if (FMT == KVQ_FMT_E4M3)
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
  else
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e5m2x2 %0, a;\n\tcvt.rn.f16x2.e5m2x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// Two binary32 values to two FP8 codes, round to nearest even, saturating
// finite overflow and +-inf to +-max.  lo -> low byte.
template <int FMT>
KVQ_DEVI uint16_t f32x2_to_fp8x2(float lo, float hi) {
  uint16_t r;
  if (FMT == KVQ_FMT_E4M3)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two binary32 values to f16x2 / bf16x2 (round to nearest even); lo -> low half.
KVQ_DEVI uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

KVQ_DEVI uint32_t f32x2_to_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

KVQ_DEVI float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
KVQ_DEVI float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

KVQ_DEVI float f16lo_to_f32(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
KVQ_DEVI float f16hi_to_f32(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

KVQ_DEVI uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

KVQ_DEVI float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Largest finite magnitude among bf16 values, two at a time, as signed
// 16-bit keys: key = (|x| bits) + 0x80 maps the finite magnitudes
// (0 .. 0x7F7F) onto 0x80 .. 0x7FFF in their order and +-inf / NaN
// (0x7F80 .. 0x7FFF) onto negative values, so a running max.s16x2 that
// starts at the key of 0 skips them.  No carry crosses the halves (a key is
// at most 0x807F).  mag_of_key16 turns the larger half back into the
// magnitude's bits.
constexpr uint32_t kMagKey0 = 0x00800080u;  // both halves: the key of 0

KVQ_DEVI uint32_t max_s16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.s16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

KVQ_DEVI uint32_t max_key16(uint32_t acc, const uint4& a, const uint4& b) {
  acc = max_s16x2(acc, (a.x & 0x7FFF7FFFu) + kMagKey0);
  acc = max_s16x2(acc, (a.y & 0x7FFF7FFFu) + kMagKey0);
  acc = max_s16x2(acc, (a.z & 0x7FFF7FFFu) + kMagKey0);
  acc = max_s16x2(acc, (a.w & 0x7FFF7FFFu) + kMagKey0);
  acc = max_s16x2(acc, (b.x & 0x7FFF7FFFu) + kMagKey0);
  acc = max_s16x2(acc, (b.y & 0x7FFF7FFFu) + kMagKey0);
  acc = max_s16x2(acc, (b.z & 0x7FFF7FFFu) + kMagKey0);
  acc = max_s16x2(acc, (b.w & 0x7FFF7FFFu) + kMagKey0);
  return acc;
}

// bf16 bits of the larger of the two halves' magnitudes (both halves of a
// running max are keys >= 0x80), placed in the high half: a binary32 value
KVQ_DEVI uint32_t mag_of_key16(uint32_t acc) {
  return (max(acc & 0xFFFFu, acc >> 16) - 0x80u) << 16;
}

}  // namespace kvq
