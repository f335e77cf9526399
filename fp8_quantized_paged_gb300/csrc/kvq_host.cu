// kvq_host.cu -- host helpers of libkvq: device properties, the
// kv_cache_dtype parser, the skip-layer rule, status strings.
//
// The parser and the skip rule restate the configuration surface of the
// "vLLM FP8 quantized KV cache guide" (kv_cache_dtype values and the
// fp8 -> fp8_e4m3 alias; kv_cache_dtype_skip_layers taking either the
// attention type "sliding_window" or layer indices; a skipped layer falls
// back to the model dtype).
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstring>

#include "../../include/kvq.h"
#include "kvq_host.h"

namespace kvq {

void token_row_shape(int64_t num_tokens, int row_units, int blocks_per_sm, int& grid, int& block) {
  int g_mult = 1;
  if (row_units <= 256) {
    block = (256 / row_units) * row_units;
  } else {
    block = 256;
    int a = row_units, b = 256;
    while (b) {
      const int t = a % b;
      a = b;
      b = t;
    }
    g_mult = row_units / a;  // row_units / gcd(row_units, 256)
  }
  const int64_t threads = num_tokens * row_units;  // one per chunk
  int64_t need = (threads + block - 1) / block;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * blocks_per_sm;
  if (need > cap) need = cap;
  need = (need + g_mult - 1) / g_mult * g_mult;
  grid = static_cast<int>(need > 0 ? need : g_mult);
}

int device_sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace kvq

extern "C" int kvq_parse_dtype(const char* s) {
  if (!s) return KVQ_ERR_NULL;
  if (!std::strcmp(s, "fp8") || !std::strcmp(s, "fp8_e4m3")) return KVQ_FMT_E4M3;
  if (!std::strcmp(s, "fp8_e5m2")) return KVQ_FMT_E5M2;
  if (!std::strcmp(s, "auto") || !std::strcmp(s, "bfloat16") || !std::strcmp(s, "bf16"))
    return KVQ_FMT_BF16;
  return KVQ_ERR_UNSUPPORTED;
}

extern "C" int kvq_layer_fmt(int fmt, int layer_idx, int is_sliding, const char* const* skip,
                             int n_skip) {
  if (fmt < KVQ_FMT_BF16 || fmt > KVQ_FMT_E5M2 || layer_idx < 0 || n_skip < 0) return KVQ_ERR_ARG;
  if (n_skip > 0 && !skip) return KVQ_ERR_NULL;
  char idx[16];
  std::snprintf(idx, sizeof idx, "%d", layer_idx);
  for (int i = 0; i < n_skip; ++i) {
    if (!skip[i]) return KVQ_ERR_NULL;
    if (is_sliding && !std::strcmp(skip[i], "sliding_window")) return KVQ_FMT_BF16;
    if (!std::strcmp(skip[i], idx)) return KVQ_FMT_BF16;
  }
  return fmt;
}

extern "C" const char* kvq_status_string(int status) {
  switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_NULL: return "a required pointer is NULL";
    case KVQ_ERR_SHAPE: return "inconsistent sizes or scale length";
    case KVQ_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case KVQ_ERR_UNSUPPORTED: return "unsupported head_dim, block_size, group size, format or flag";
    case KVQ_ERR_WORKSPACE: return "workspace too small";
    case KVQ_ERR_CUDA: return "CUDA launch error";
    case KVQ_ERR_ARG: return "invalid argument";
    default: return "unknown status";
  }
}

extern "C" int kvq_version(void) { return 100; }
