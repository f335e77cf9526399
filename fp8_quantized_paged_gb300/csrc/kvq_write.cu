// kvq_write.cu -- quantize-and-scatter into the paged FP8 cache, and the
// unfused path's separate dequant kernel.
//
// "10.4 KV Cache quantization: INT8, KIVI 2-bit, FP8 KV", section 10.4.5:
// the cache stores cast_fp8(K / sK); section 10.4.2: the inefficient path
// runs an independent dequant kernel that writes a 16-bit KV back to HBM.
//
// With per-(token, KV head) scales ("10.4 KV Cache quantization", section
// 10.4.3, per-token granularity) the write derives each row's scale from the
// row itself, s = amax / fmt_max over its finite values (1 if 0), stores it
// in a binary32 scale cache [num_blocks][Hkv][16] beside the pages and
// quantizes the row with it.
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
  int64_t capacity;  // num_blocks * 16 (block_size is 16)
  const float* ks;
  const float* vs;
  int per_head;
  float* ksc;  // per-(token, head) scale caches [num_blocks][Hkv][16] (token-head mode)
  float* vsc;
  uint32_t* status;
  int64_t in_elems;     // extent of k / v in elements
  int64_t cache_elems;  // elements of one cache tensor
};

// Per-head constants of the quantizing division x / s.  For s in
// [2^-80, 2^80] the quotient comes from the reciprocal r = RN(1/s) and one
// fused residual correction (Markstein's iteration): q0 = RN(x r),
// e = RN(x - q0 s), q = RN(q0 + e r) -- the IEEE binary32 quotient for every
// bf16 significand and every binary32 scale significand (checked
// exhaustively), on the packed f32x2 pipes two elements at a time.  Inputs
// first go through a bf16x2 clamp to +-L, L = 2^20 s rounded toward zero
// (L >= 2^19 s): every |x| > L saturates the FP8 format and so does L itself,
// infinities turn into +-L and NaN stays NaN, so q0, e and q stay finite.
// The one sign the residual form can lose is that of a zero quotient from
// x = -0; the FP8 sign bit is therefore OR-ed in from the bf16 sign bit
// (equal to the quotient's sign everywhere else).  Quotients too small for
// the residual to stay normal encode to a signed FP8 zero either way.
struct HeadScale {
  float2 r2, ns2;  // (r, r), (-s, -s)
  uint32_t L2;  // bf16x2 (L, L)
  float s;
  bool fast;
};

KVQ_DEVI HeadScale head_scale(float s) {
  HeadScale h;
  h.s = s;
  h.fast = s >= 0x1p-80f && s <= 0x1p80f;
  const float r = __frcp_rn(s);
  h.r2 = make_float2(r, r);
  h.ns2 = make_float2(-s, -s);
  uint16_t L;
  asm("cvt.rz.bf16.f32 %0, %1;" : "=h"(L) : "f"(h.fast ? s * 1048576.f : 0.f));
  h.L2 = static_cast<uint32_t>(L) * 0x10001u;
  return h;
}

// sign(x) * min(|x|, L) on both halves (L positive), NaN propagated.
KVQ_DEVI uint32_t bf16x2_clamp(uint32_t w, uint32_t L2) {
  uint32_t d;
  asm("min.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(w), "r"(L2));
  return d;
}

// Two bf16 (one word) -> two FP8 codes (low byte = low element).
template <int FMT>
KVQ_DEVI uint32_t quantize2(uint32_t w, const HeadScale& h) {
  float2 q;
  if (h.fast) {
    const uint32_t c = bf16x2_clamp(w, h.L2);
    const float2 x = make_float2(bf16lo_to_f32(c), bf16hi_to_f32(c));
    const float2 q0 = __fmul2_rn(x, h.r2);
    const float2 e = __ffma2_rn(q0, h.ns2, x);
    q = __ffma2_rn(e, h.r2, q0);
  } else {
    q = make_float2(__fdiv_rn(bf16lo_to_f32(w), h.s), __fdiv_rn(bf16hi_to_f32(w), h.s));
  }
  return f32x2_to_fp8x2<FMT>(q.x, q.y);
}

// Sixteen bf16 values (two uint4) -> sixteen FP8 codes: binary32 quotient
// x / s, then the saturating RNE conversion to FP8; signs from the inputs.
template <int FMT>
KVQ_DEVI uint4 quantize16(const uint4& a, const uint4& b, const HeadScale& h) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t codes = prmt(quantize2<FMT>(w[2 * i], h), quantize2<FMT>(w[2 * i + 1], h), 0x5410u);
    const uint32_t signs = prmt(w[2 * i], w[2 * i + 1], 0x7531u);
    o[i] = codes | (signs & 0x80808080u);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Scale of one (token, KV head) row held by CH consecutive lanes (aligned to
// CH in the warp; mask = those lanes): the largest finite magnitude of the
// row over the format's largest finite value (binary32 division), or 1 when
// that is 0.
template <int CH>
KVQ_DEVI float row_amax(const uint4& a, const uint4& b, uint32_t mask) {
  uint32_t am = mag_of_key16(max_key16(kMagKey0, a, b));
#pragma unroll
  for (int off = 1; off < CH; off <<= 1) am = max(am, __shfl_xor_sync(mask, am, off));
  return __uint_as_float(am);
}

template <int FMT>
KVQ_DEVI float scale_of_amax(float amax) {
  const float q = __fdiv_rn(amax, FMT == KVQ_FMT_E4M3 ? 448.f : 57344.f);
  return q > 0.f ? q : 1.f;
}

// The K and V row scales' division constants: one half of the row's lanes
// derives K's, the other half V's (a correctly rounded division and
// reciprocal each), and the halves swap them.
template <int FMT, int CH>
KVQ_DEVI void row_scales(const uint4 (&k)[2], const uint4 (&v)[2], uint32_t mask, HeadScale& hk,
                         HeadScale& hv) {
  const float ak = row_amax<CH>(k[0], k[1], mask), av = row_amax<CH>(v[0], v[1], mask);
  const bool k_half = (threadIdx.x & (CH / 2)) == 0;
  const HeadScale h = head_scale(scale_of_amax<FMT>(k_half ? ak : av));
  HeadScale o;
  o.s = __shfl_xor_sync(mask, h.s, CH / 2);
  const float r = __shfl_xor_sync(mask, h.r2.x, CH / 2);
  o.L2 = __shfl_xor_sync(mask, h.L2, CH / 2);
  o.fast = o.s >= 0x1p-80f && o.s <= 0x1p80f;
  o.r2 = make_float2(r, r);
  o.ns2 = make_float2(-o.s, -o.s);
  hk = k_half ? h : o;
  hv = k_half ? o : h;
}

// One thread per 16-element chunk (h, c) of the (token, KV head) rows.  The
// grid's thread count is a multiple of the Hkv * DH/16 chunks of a token, so
// a thread keeps its chunk (and its head's scales) and strides over tokens;
// the next token's K/V and slot loads are issued before the current token is
// converted.
// TS: per-(token, head) scales, computed by the CH lanes of each row.
template <int FMT, int DH, bool TS>
__global__ void __launch_bounds__(256, 3) write_kernel(const WriteParams p) {
  constexpr int CH = DH / 16;
  pdl_allow_next();
  pdl_wait();  // k, v, slots may come from the previous kernel
  const int row_units = p.hkv * CH;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int rem = static_cast<int>(gtid % row_units);
  const int h = rem / CH;
  const int64_t tstride = nthreads / row_units;
  int64_t t = gtid / row_units;
  if (t >= p.num_tokens) return;
  HeadScale hk, hv;
  // the CH lanes of this thread's row (a token's rows are whole, aligned
  // lane groups: the block is a multiple of Hkv * CH threads, or of 256)
  const uint32_t row_mask = (CH == 8 ? 0xFFu : 0xFu) << (threadIdx.x & 31 & ~(CH - 1));
  if (FMT != KVQ_FMT_BF16 && !TS) {
    hk = head_scale(__ldg(p.ks + (p.per_head ? h : 0)));
    hv = head_scale(__ldg(p.vs + (p.per_head ? h : 0)));
  }
  auto load = [&](int64_t tt, uint4 (&kk)[2], uint4 (&vv)[2], int64_t& slot) {
    const int64_t src = tt * p.token_stride + rem * 16;
    if (guard(src >= 0 && src + 16 <= p.in_elems, p.status, 7)) {
      const uint4* ks = reinterpret_cast<const uint4*>(p.k + src);
      const uint4* vs = reinterpret_cast<const uint4*>(p.v + src);
      kk[0] = __ldcs(ks);
      kk[1] = __ldcs(ks + 1);
      vv[0] = __ldcs(vs);
      vv[1] = __ldcs(vs + 1);
      slot = __ldg(p.slots + tt);
    } else {
      slot = -1;
    }
  };
  uint4 k[2], v[2];
  int64_t slot;
  load(t, k, v, slot);
  while (true) {
    const int64_t tn = t + tstride;
    uint4 kn[2], vn[2];
    int64_t sn = -1;
    if (tn < p.num_tokens) load(tn, kn, vn, sn);
    if (TS)  // every lane of the row takes part, whatever its slot
      row_scales<FMT, CH>(k, v, row_mask, hk, hv);
    if (slot >= p.capacity) {
      if (rem == 0) flag_status(p.status, KVQ_DEV_BAD_SLOT);
    } else if (slot >= 0) {  // a negative slot is a padding token
      const int64_t dst = (((slot >> 4) * p.hkv + h) * 16 + (slot & 15)) * DH + (rem % CH) * 16;
      if (guard(dst >= 0 && dst + 16 <= p.cache_elems, p.status, 8)) {
        if (FMT == KVQ_FMT_BF16) {
          uint4* kd = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.kc) + dst);
          uint4* vd = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.vc) + dst);
          kd[0] = k[0];
          kd[1] = k[1];
          vd[0] = v[0];
          vd[1] = v[1];
        } else {
          *reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.kc) + dst) = quantize16<FMT>(k[0], k[1], hk);
          *reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.vc) + dst) = quantize16<FMT>(v[0], v[1], hv);
          if (TS && rem % CH == 0) {
            const int64_t row = ((slot >> 4) * p.hkv + h) * 16 + (slot & 15);
            p.ksc[row] = hk.s;
            p.vsc[row] = hv.s;
          }
        }
      }
    }
    if (tn >= p.num_tokens) break;
    t = tn;
    k[0] = kn[0];
    k[1] = kn[1];
    v[0] = vn[0];
    v[1] = vn[1];
    slot = sn;
  }
}

struct DequantParams {
  const uint8_t* src;
  uint16_t* dst;
  int64_t units;        // 16-element chunks in the cache
  int chunks_per_head;  // block_size * head_dim / 16
  int hkv;
  const float* scale;
  int gran;  // kvq_gran: [1], [Hkv] or [num_blocks][Hkv][16] scales
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
    // the token row of chunk u is u / (chunks per row), chunks_per_head / 16
    const int64_t si = p.gran == KVQ_SCALE_PER_TOKEN_HEAD ? u / (p.chunks_per_head / 16)
                                                          : (p.gran == KVQ_SCALE_PER_HEAD ? h : 0);
    const float s = __ldg(p.scale + si);
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

// Grid of a streaming kernel: one work unit per thread while that stays
// under 64 waves of the SMs; beyond that the kernel loops (grid-stride).
static int grid_for(int64_t units, int threads) {
  const int64_t need = (units + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8 * 64;
  return static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
}

// Shape checks and launch shared by the two write entry points.
static int write_common(const void* k, const void* v, int64_t token_stride,
                        const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                        int head_dim, void* k_cache, void* v_cache, int64_t num_blocks,
                        int block_size, int fmt, WriteParams& p, bool token_scales,
                        uint32_t* dev_status, kvq_stream_t stream) {
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
  if (num_blocks > (INT64_MAX / 16) / (static_cast<int64_t>(num_kv_heads) * head_dim))
    return KVQ_ERR_SHAPE;
  if (num_tokens == 0) return KVQ_OK;

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
  p.status = dev_status;
  p.in_elems = (num_tokens - 1) * token_stride + static_cast<int64_t>(num_kv_heads) * head_dim;
  p.cache_elems = num_blocks * num_kv_heads * block_size * head_dim;
  int grid = 0, block = 0;
  token_row_shape(num_tokens, num_kv_heads * (head_dim / 16), 3, grid, block);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  const dim3 gd(grid), bd(block);
#define KVQ_WRITE_LAUNCH(F, D)                                                              \
  (token_scales ? launch_pdl(write_kernel<F, D, true>, gd, bd, 0, s, p)                     \
                : launch_pdl(write_kernel<F, D, false>, gd, bd, 0, s, p))
  if (head_dim == 128) {
    switch (fmt) {
      case KVQ_FMT_E4M3: e = KVQ_WRITE_LAUNCH(KVQ_FMT_E4M3, 128); break;
      case KVQ_FMT_E5M2: e = KVQ_WRITE_LAUNCH(KVQ_FMT_E5M2, 128); break;
      default: e = launch_pdl(write_kernel<KVQ_FMT_BF16, 128, false>, gd, bd, 0, s, p); break;
    }
  } else {
    switch (fmt) {
      case KVQ_FMT_E4M3: e = KVQ_WRITE_LAUNCH(KVQ_FMT_E4M3, 64); break;
      case KVQ_FMT_E5M2: e = KVQ_WRITE_LAUNCH(KVQ_FMT_E5M2, 64); break;
      default: e = launch_pdl(write_kernel<KVQ_FMT_BF16, 64, false>, gd, bd, 0, s, p); break;
    }
  }
#undef KVQ_WRITE_LAUNCH
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
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
  if (fmt != KVQ_FMT_BF16 && num_kv_heads > 0) {
    if (!k_scale || !v_scale) return KVQ_ERR_NULL;
    const int want = scale_granularity == KVQ_SCALE_PER_HEAD ? num_kv_heads : 1;
    if (k_scale_len != want || v_scale_len != want) return KVQ_ERR_SHAPE;
  }
  WriteParams p = {};
  p.ks = k_scale;
  p.vs = v_scale;
  p.per_head = scale_granularity == KVQ_SCALE_PER_HEAD;
  return write_common(k, v, token_stride, slot_mapping, num_tokens, num_kv_heads, head_dim,
                      k_cache, v_cache, num_blocks, block_size, fmt, p, false, dev_status,
                      stream);
}

extern "C" int kvq_write_token_head(const void* k, const void* v, int64_t token_stride,
                                    const int64_t* slot_mapping, int64_t num_tokens,
                                    int num_kv_heads, int head_dim, void* k_cache, void* v_cache,
                                    int64_t num_blocks, int block_size, float* k_scale_cache,
                                    float* v_scale_cache, int fmt, uint32_t* dev_status,
                                    kvq_stream_t stream) {
  if (fmt < KVQ_FMT_BF16 || fmt > KVQ_FMT_E5M2) return KVQ_ERR_ARG;
  if (fmt == KVQ_FMT_BF16) return KVQ_ERR_UNSUPPORTED;
  if (!k_scale_cache || !v_scale_cache) return KVQ_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(k_scale_cache) & 15u) ||
      (reinterpret_cast<uintptr_t>(v_scale_cache) & 15u))
    return KVQ_ERR_ALIGN;
  WriteParams p = {};
  p.ksc = k_scale_cache;
  p.vsc = v_scale_cache;
  return write_common(k, v, token_stride, slot_mapping, num_tokens, num_kv_heads, head_dim,
                      k_cache, v_cache, num_blocks, block_size, fmt, p, true, dev_status, stream);
}

extern "C" int kvq_dequant_cache(const void* src, void* dst_bf16, int64_t num_blocks,
                                 int num_kv_heads, int block_size, int head_dim,
                                 const float* scale, int scale_len, int scale_granularity,
                                 int fmt, kvq_stream_t stream) {
  if (fmt != KVQ_FMT_E4M3 && fmt != KVQ_FMT_E5M2) return KVQ_ERR_UNSUPPORTED;
  if (scale_granularity != KVQ_SCALE_PER_TENSOR && scale_granularity != KVQ_SCALE_PER_HEAD &&
      scale_granularity != KVQ_SCALE_PER_TOKEN_HEAD)
    return KVQ_ERR_ARG;
  if (num_blocks < 0 || num_kv_heads <= 0) return KVQ_ERR_ARG;
  if (!src || !dst_bf16 || !scale) return KVQ_ERR_NULL;
  if (head_dim != 64 && head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (block_size != 16) return KVQ_ERR_UNSUPPORTED;
  if (!aligned16(src) || !aligned16(dst_bf16)) return KVQ_ERR_ALIGN;
  const int64_t want = scale_granularity == KVQ_SCALE_PER_TOKEN_HEAD
                           ? num_blocks * num_kv_heads * block_size
                           : (scale_granularity == KVQ_SCALE_PER_HEAD ? num_kv_heads : 1);
  if (scale_len != want) return KVQ_ERR_SHAPE;
  if (num_blocks == 0) return KVQ_OK;
  DequantParams p;
  p.src = static_cast<const uint8_t*>(src);
  p.dst = static_cast<uint16_t*>(dst_bf16);
  p.chunks_per_head = block_size * head_dim / 16;
  p.units = num_blocks * num_kv_heads * p.chunks_per_head;
  p.hkv = num_kv_heads;
  p.scale = scale;
  p.gran = scale_granularity;
  const int grid = grid_for(p.units, 256);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e =
      fmt == KVQ_FMT_E4M3
          ? launch_pdl(dequant_kernel<KVQ_FMT_E4M3>, dim3(grid), dim3(256), 0, s, p)
          : launch_pdl(dequant_kernel<KVQ_FMT_E5M2>, dim3(grid), dim3(256), 0, s, p);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
