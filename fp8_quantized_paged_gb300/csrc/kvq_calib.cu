// kvq_calib.cu -- per-tensor or per-KV-head FP8 scales from the data.
//
// "vLLM FP8 quantized KV cache guide", scale calibration, way two: the
// scales are estimated from statistics of the K/V activations (there by a
// calibration pass over a small data set).  The statistic here is the
// absolute maximum of the given tokens, and the scale maps it onto the
// format's largest finite value, s = amax / fmt_max (448 for E4M3, 57344
// for E5M2), so quantizing those tokens with s never saturates.
//
// Three kernels: a reduction, one thread per 16-element chunk of a (token,
// head) row striding over tokens (signed 16-bit max of keys of the bf16
// magnitudes, two at a time, four tokens in flight), lanes of a head combined by shuffles and one atomicMax per head
// and warp on the magnitude's bit pattern (non-negative floats order like
// unsigned integers), after a one-block kernel has zeroed those words; then
// a finalize kernel that turns the maxima into scales in place.
#include "kvq_common.cuh"
#include "kvq_host.h"

namespace kvq {

struct CalibParams {
  const uint16_t* k;
  const uint16_t* v;
  int64_t token_stride;
  int64_t num_tokens;
  int hkv;
  int per_head;
  uint32_t* kmax;  // [1] or [Hkv]: bit patterns of the running maxima (start at 0)
  uint32_t* vmax;
  int64_t in_elems;  // extent of k / v in elements
  uint32_t* status;
};

constexpr int kCalibTokens = 4;     // tokens a thread has in flight per step
constexpr int kCalibBlocksPerSM = 3;

template <int DH>
__global__ void __launch_bounds__(256, kCalibBlocksPerSM) calib_kernel(const CalibParams p) {
  constexpr int CH = DH / 16;  // chunks of a head row; divides 32
  pdl_allow_next();
  pdl_wait();  // k, v may come from the previous kernel
  const int row_units = p.hkv * CH;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int rem = static_cast<int>(gtid % row_units);
  const int h = rem / CH;
  const int64_t tstride = nthreads / row_units;
  uint32_t mk = kMagKey0, mv = kMagKey0;  // two 16-bit magnitude keys each
  // kCalibTokens tokens per step, their 16-byte loads issued together (the
  // kernel is bound by load latency: the more bytes in flight the better)
  for (int64_t t = gtid / row_units; t < p.num_tokens; t += kCalibTokens * tstride) {
    uint4 a[kCalibTokens][4];
    bool ok[kCalibTokens];
#pragma unroll
    for (int i = 0; i < kCalibTokens; ++i) {
      const int64_t tt = t + i * tstride;
      const int64_t src = tt * p.token_stride + rem * 16;
      ok[i] = tt < p.num_tokens && guard(src >= 0 && src + 16 <= p.in_elems, p.status, 9);
      const uint4* ks = reinterpret_cast<const uint4*>(p.k + (ok[i] ? src : 0));
      const uint4* vs = reinterpret_cast<const uint4*>(p.v + (ok[i] ? src : 0));
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      a[i][0] = ok[i] ? __ldcs(ks) : z;
      a[i][1] = ok[i] ? __ldcs(ks + 1) : z;
      a[i][2] = ok[i] ? __ldcs(vs) : z;
      a[i][3] = ok[i] ? __ldcs(vs + 1) : z;
    }
#pragma unroll
    for (int i = 0; i < kCalibTokens; ++i) {
      mk = max_key16(mk, a[i][0], a[i][1]);
      mv = max_key16(mv, a[i][2], a[i][3]);
    }
  }
  // every thread takes part (those without tokens contribute 0): the CH
  // lanes of a head are consecutive, as the block is a multiple of Hkv * CH
  uint32_t ak = mag_of_key16(mk), av = mag_of_key16(mv);
#pragma unroll
  for (int off = 1; off < CH; off <<= 1) {
    ak = max(ak, __shfl_xor_sync(0xFFFFFFFFu, ak, off));
    av = max(av, __shfl_xor_sync(0xFFFFFFFFu, av, off));
  }
  if ((threadIdx.x & (CH - 1)) == 0 && (ak | av)) {
    const int i = p.per_head ? h : 0;
    if (ak) atomicMax(p.kmax + i, ak);
    if (av) atomicMax(p.vmax + i, av);
  }
}

// The maxima words (the scale arrays themselves) start at zero.  A kernel
// rather than a memset, so that the chain of three launches overlaps by
// programmatic dependent launch; it waits for the kernel before it, which
// may still read the previous scales.
__global__ void calib_zero(uint32_t* kbits, uint32_t* vbits, int n) {
  pdl_allow_next();
  pdl_wait();
  for (int i = threadIdx.x; i < 2 * n; i += blockDim.x) (i < n ? kbits[i] : vbits[i - n]) = 0u;
}

// In place: scale = amax / fmt_max (binary32, round to nearest even); 1.0
// where that is 0 (no finite non-zero value, or a quotient that underflows).
__global__ void calib_finalize(uint32_t* kbits, uint32_t* vbits, int n, float fmt_max) {
  pdl_allow_next();
  pdl_wait();
  for (int i = threadIdx.x; i < 2 * n; i += blockDim.x) {
    uint32_t* b = i < n ? kbits + i : vbits + (i - n);
    const float amax = __uint_as_float(*b);
    const float q = __fdiv_rn(amax, fmt_max);
    *reinterpret_cast<float*>(b) = q > 0.f ? q : 1.f;
  }
}

}  // namespace kvq

using namespace kvq;

extern "C" int kvq_calibrate_scales(const void* k, const void* v, int64_t token_stride,
                                    int64_t num_tokens, int num_kv_heads, int head_dim,
                                    int scale_granularity, int fmt, float* k_scale, float* v_scale,
                                    uint32_t* dev_status, kvq_stream_t stream) {
  if (fmt != KVQ_FMT_E4M3 && fmt != KVQ_FMT_E5M2) return KVQ_ERR_UNSUPPORTED;
  if (scale_granularity != KVQ_SCALE_PER_TENSOR && scale_granularity != KVQ_SCALE_PER_HEAD)
    return KVQ_ERR_ARG;
  if (num_tokens < 0 || num_kv_heads <= 0) return KVQ_ERR_ARG;
  if (!k_scale || !v_scale) return KVQ_ERR_NULL;
  if (num_tokens > 0 && (!k || !v)) return KVQ_ERR_NULL;
  if (head_dim != 64 && head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (token_stride < static_cast<int64_t>(num_kv_heads) * head_dim) return KVQ_ERR_SHAPE;
  if (token_stride % 8 != 0) return KVQ_ERR_ALIGN;
  if ((num_tokens > 0 && (!aligned16(k) || !aligned16(v))) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
    return KVQ_ERR_ALIGN;
  const int n = scale_granularity == KVQ_SCALE_PER_HEAD ? num_kv_heads : 1;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_pdl(calib_zero, dim3(1), dim3(256), 0, s,
                             reinterpret_cast<uint32_t*>(k_scale), reinterpret_cast<uint32_t*>(v_scale), n);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  if (num_tokens > 0) {
    CalibParams p;
    p.k = static_cast<const uint16_t*>(k);
    p.v = static_cast<const uint16_t*>(v);
    p.token_stride = token_stride;
    p.num_tokens = num_tokens;
    p.hkv = num_kv_heads;
    p.per_head = scale_granularity == KVQ_SCALE_PER_HEAD;
    p.kmax = reinterpret_cast<uint32_t*>(k_scale);
    p.vmax = reinterpret_cast<uint32_t*>(v_scale);
    p.in_elems = (num_tokens - 1) * token_stride + static_cast<int64_t>(num_kv_heads) * head_dim;
    p.status = dev_status;
    int grid = 0, block = 0;
    token_row_shape(num_tokens, num_kv_heads * (head_dim / 16), kCalibBlocksPerSM, grid, block);
    e = head_dim == 128 ? launch_pdl(calib_kernel<128>, dim3(grid), dim3(block), 0, s, p)
                        : launch_pdl(calib_kernel<64>, dim3(grid), dim3(block), 0, s, p);
    if (e != cudaSuccess) return KVQ_ERR_CUDA;
  }
  const float fmt_max = fmt == KVQ_FMT_E4M3 ? 448.f : 57344.f;
  e = launch_pdl(calib_finalize, dim3(1), dim3(256), 0, s, reinterpret_cast<uint32_t*>(k_scale),
                 reinterpret_cast<uint32_t*>(v_scale), n, fmt_max);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
