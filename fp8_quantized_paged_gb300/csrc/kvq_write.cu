// kvq_write.cu -- quantize-and-scatter into the paged FP8 cache, and the
// unfused path's separate dequant kernel.
//
// "10.4 KV Cache quantization: INT8, KIVI 2-bit, FP8 KV", section 10.4.5:
// the cache stores cast_fp8(K / sK); section 10.4.2: the inefficient path
// runs an independent dequant kernel that writes a 16-bit KV back to HBM.
//
// Both kernels are HBM streams.  One thread owns 16 contiguous elements of
// one (token, KV head) row: two 16-byte bf16 loads per tensor, one 16-byte
// FP8 store (or two 16-byte bf16 stores), so a warp moves whole 128-byte
// lines.  Grids are a multiple of the SM count with a grid-stride loop.
#include <cuda_fp16.h>

#include "kvq_common.cuh"
#include "kvq_host.h"

namespace kvq {

struct WriteParams {
  const uint16_t* k;
  const uint16_t* v;
  int64_t token_stride;
  const int64_t* slots;
  int64_t num_tokens;
  int hkv;
  int dh;
  void* kc;
  void* vc;
  int64_t capacity;  // num_blocks * block_size
  int bs;
  const float* ks;
  const float* vs;
  int per_head;
  uint32_t* status;
  int64_t in_elems;     // extent of k / v in elements
  int64_t cache_elems;  // elements of one cache tensor
};

// x / s, correctly rounded (IEEE binary32), for a scale s whose reciprocal
// r = RN(1/s) and the residuals below stay normal (s in [2^-80, 2^80]): one
// product and one fused residual correction (Markstein's iteration)
// q0 = RN(x r), e = RN(x - q0 s), q = RN(q0 + e r).  Exhaustively checked
// against IEEE division for every bf16 significand and every binary32 scale
// significand.  e == 0 means q0 is exact (this also keeps the sign of zero);
// |q0| >= 2^20 saturates every FP8 format, so q0 is kept there (and an
// infinite or NaN x passes through).  Quotients too small for the residual to
// stay normal encode to a signed FP8 zero either way.
KVQ_DEVI float div_by_scale(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  const float e = __fmaf_rn(-q0, s, x);
  return (e == 0.f || !(fabsf(q0) < 1048576.f)) ? q0 : __fmaf_rn(e, r, q0);
}

KVQ_DEVI bool scale_is_nice(float s) { return s >= 0x1p-80f && s <= 0x1p80f; }

// Sixteen bf16 values (two uint4) -> sixteen FP8 codes: binary32 IEEE
// quotient x / s (round to nearest even, no flush to zero), then the
// saturating RNE conversion to FP8.
template <int FMT>
KVQ_DEVI uint4 quantize16(const uint4& a, const uint4& b, float s, float r, bool fast) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float x[4] = {bf16lo_to_f32(w[2 * i]), bf16hi_to_f32(w[2 * i]), bf16lo_to_f32(w[2 * i + 1]),
                  bf16hi_to_f32(w[2 * i + 1])};
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = fast ? div_by_scale(x[j], s, r) : __fdiv_rn(x[j], s);
    o[i] = static_cast<uint32_t>(f32x2_to_fp8x2<FMT>(x[0], x[1])) |
           (static_cast<uint32_t>(f32x2_to_fp8x2<FMT>(x[2], x[3])) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One thread per 16-element chunk of one (token, KV head) row.  The K/V
// loads do not depend on the slot, so they are issued before it is checked.
template <int FMT>
__global__ void __launch_bounds__(256) write_kernel(const WriteParams p) {
  pdl_allow_next();
  pdl_wait();  // k, v, slots may come from the previous kernel
  const int chunks = p.dh >> 4;
  const int64_t units = p.num_tokens * p.hkv * chunks;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
       u += stride) {
    const int c = static_cast<int>(u % chunks);
    const int64_t th = u / chunks;
    const int h = static_cast<int>(th % p.hkv);
    const int64_t t = th / p.hkv;
    const int64_t src = t * p.token_stride + static_cast<int64_t>(h) * p.dh + c * 16;
    if (!guard(src >= 0 && src + 16 <= p.in_elems, p.status, 7)) continue;
    const uint4* ksrc = reinterpret_cast<const uint4*>(p.k + src);
    const uint4* vsrc = reinterpret_cast<const uint4*>(p.v + src);
    const uint4 ka = __ldcs(ksrc), kb = __ldcs(ksrc + 1);
    const uint4 va = __ldcs(vsrc), vb = __ldcs(vsrc + 1);
    const int64_t slot = __ldg(p.slots + t);
    if (slot < 0) continue;  // padding token
    if (slot >= p.capacity) {
      if (h == 0 && c == 0) flag_status(p.status, KVQ_DEV_BAD_SLOT);
      continue;
    }
    const int64_t blk = slot / p.bs, off = slot - blk * p.bs;
    const int64_t dst = ((blk * p.hkv + h) * p.bs + off) * p.dh + c * 16;
    if (!guard(dst >= 0 && dst + 16 <= p.cache_elems, p.status, 8)) continue;
    if (FMT == KVQ_FMT_BF16) {
      uint4* kd = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.kc) + dst);
      uint4* vd = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.vc) + dst);
      kd[0] = ka;
      kd[1] = kb;
      vd[0] = va;
      vd[1] = vb;
    } else {
      const float sk = __ldg(p.ks + (p.per_head ? h : 0));
      const float sv = __ldg(p.vs + (p.per_head ? h : 0));
      const bool fast = scale_is_nice(sk) && scale_is_nice(sv);
      *reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.kc) + dst) =
          quantize16<FMT>(ka, kb, sk, __frcp_rn(sk), fast);
      *reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.vc) + dst) =
          quantize16<FMT>(va, vb, sv, __frcp_rn(sv), fast);
    }
  }
}

struct DequantParams {
  const uint8_t* src;
  uint16_t* dst;
  int64_t units;        // 16-element chunks in the cache
  int chunks_per_head;  // block_size * head_dim / 16
  int hkv;
  const float* scale;
  int per_head;
};

// Sixteen FP8 codes -> sixteen bf16: exact FP8 -> f16 -> f32, one binary32
// product with the head's scale, RNE to bf16.
template <int FMT>
__global__ void __launch_bounds__(256) dequant_kernel(const DequantParams p) {
  pdl_allow_next();
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < p.units;
       u += stride) {
    const int h = static_cast<int>((u / p.chunks_per_head) % p.hkv);
    const float s = __ldg(p.scale + (p.per_head ? h : 0));
    const uint4 c = __ldcs(reinterpret_cast<const uint4*>(p.src) + u);
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = fp8x2_to_f16x2<FMT>(static_cast<uint16_t>(w[i] & 0xFFFFu));
      const uint32_t hi = fp8x2_to_f16x2<FMT>(static_cast<uint16_t>(w[i] >> 16));
      o[2 * i] = f32x2_to_bf16x2(__fmul_rn(f16lo_to_f32(lo), s), __fmul_rn(f16hi_to_f32(lo), s));
      o[2 * i + 1] =
          f32x2_to_bf16x2(__fmul_rn(f16lo_to_f32(hi), s), __fmul_rn(f16hi_to_f32(hi), s));
    }
    uint4* d = reinterpret_cast<uint4*>(p.dst) + 2 * u;
    d[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// One work unit per thread while the grid stays under 64 waves of the SMs;
// beyond that the kernels loop (grid-stride).
static int grid_for(int64_t units, int threads) {
  const int64_t need = (units + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8 * 64;
  return static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
}

}  // namespace kvq

using namespace kvq;

extern "C" int kvq_write(const void* k, const void* v, int64_t token_stride,
                         const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                         int head_dim, void* k_cache, void* v_cache, int64_t num_blocks,
                         int block_size, const float* k_scale, int k_scale_len,
                         const float* v_scale, int v_scale_len, int scale_granularity, int fmt,
                         uint32_t* dev_status, kvq_stream_t stream) {
  if (fmt < KVQ_FMT_BF16 || fmt > KVQ_FMT_E5M2) return KVQ_ERR_ARG;
  if (scale_granularity != KVQ_SCALE_PER_TENSOR && scale_granularity != KVQ_SCALE_PER_HEAD)
    return KVQ_ERR_ARG;
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return KVQ_ERR_ARG;
  if (!k_cache || !v_cache) return KVQ_ERR_NULL;
  if (num_tokens > 0 && (!k || !v || !slot_mapping)) return KVQ_ERR_NULL;
  if (head_dim != 64 && head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (block_size != 16) return KVQ_ERR_UNSUPPORTED;
  if (token_stride < static_cast<int64_t>(num_kv_heads) * head_dim) return KVQ_ERR_SHAPE;
  if (token_stride % 8 != 0) return KVQ_ERR_ALIGN;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return KVQ_ERR_ALIGN;
  if (fmt != KVQ_FMT_BF16) {
    if (!k_scale || !v_scale) return KVQ_ERR_NULL;
    const int want = scale_granularity == KVQ_SCALE_PER_HEAD ? num_kv_heads : 1;
    if (k_scale_len != want || v_scale_len != want) return KVQ_ERR_SHAPE;
  }
  if (num_blocks > (INT64_MAX / 16) / (static_cast<int64_t>(num_kv_heads) * head_dim))
    return KVQ_ERR_SHAPE;
  if (num_tokens == 0) return KVQ_OK;

  WriteParams p;
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.token_stride = token_stride;
  p.slots = slot_mapping;
  p.num_tokens = num_tokens;
  p.hkv = num_kv_heads;
  p.dh = head_dim;
  p.kc = k_cache;
  p.vc = v_cache;
  p.capacity = num_blocks * block_size;
  p.bs = block_size;
  p.ks = k_scale;
  p.vs = v_scale;
  p.per_head = scale_granularity == KVQ_SCALE_PER_HEAD;
  p.status = dev_status;
  p.in_elems = (num_tokens - 1) * token_stride + static_cast<int64_t>(num_kv_heads) * head_dim;
  p.cache_elems = num_blocks * num_kv_heads * block_size * head_dim;
  const int64_t units = num_tokens * num_kv_heads * (head_dim / 16);
  const int grid = grid_for(units, 256);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (fmt) {
    case KVQ_FMT_E4M3: e = launch_pdl(write_kernel<KVQ_FMT_E4M3>, dim3(grid), dim3(256), 0, s, p); break;
    case KVQ_FMT_E5M2: e = launch_pdl(write_kernel<KVQ_FMT_E5M2>, dim3(grid), dim3(256), 0, s, p); break;
    default: e = launch_pdl(write_kernel<KVQ_FMT_BF16>, dim3(grid), dim3(256), 0, s, p); break;
  }
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

extern "C" int kvq_dequant_cache(const void* src, void* dst_bf16, int64_t num_blocks,
                                 int num_kv_heads, int block_size, int head_dim,
                                 const float* scale, int scale_len, int scale_granularity,
                                 int fmt, kvq_stream_t stream) {
  if (fmt != KVQ_FMT_E4M3 && fmt != KVQ_FMT_E5M2) return KVQ_ERR_UNSUPPORTED;
  if (scale_granularity != KVQ_SCALE_PER_TENSOR && scale_granularity != KVQ_SCALE_PER_HEAD)
    return KVQ_ERR_ARG;
  if (num_blocks < 0 || num_kv_heads <= 0) return KVQ_ERR_ARG;
  if (!src || !dst_bf16 || !scale) return KVQ_ERR_NULL;
  if (head_dim != 64 && head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (block_size != 16) return KVQ_ERR_UNSUPPORTED;
  if (!aligned16(src) || !aligned16(dst_bf16)) return KVQ_ERR_ALIGN;
  const int want = scale_granularity == KVQ_SCALE_PER_HEAD ? num_kv_heads : 1;
  if (scale_len != want) return KVQ_ERR_SHAPE;
  if (num_blocks == 0) return KVQ_OK;
  DequantParams p;
  p.src = static_cast<const uint8_t*>(src);
  p.dst = static_cast<uint16_t*>(dst_bf16);
  p.chunks_per_head = block_size * head_dim / 16;
  p.units = num_blocks * num_kv_heads * p.chunks_per_head;
  p.hkv = num_kv_heads;
  p.scale = scale;
  p.per_head = scale_granularity == KVQ_SCALE_PER_HEAD;
  const int grid = grid_for(p.units, 256);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e =
      fmt == KVQ_FMT_E4M3
          ? launch_pdl(dequant_kernel<KVQ_FMT_E4M3>, dim3(grid), dim3(256), 0, s, p)
          : launch_pdl(dequant_kernel<KVQ_FMT_E5M2>, dim3(grid), dim3(256), 0, s, p);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
