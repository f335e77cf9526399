// kvq_static.cu -- decode attention for callers that cannot allocate device
// memory.
//
// kvq_decode_attn needs a device workspace from its caller.  Some callers
// have no way to provide one: a C plugin that a host program loads and hands
// only input and output pointers, with no allocator of its own to call, or
// a serving loop that has fixed its device-memory plan at start-up and may
// not call cudaMalloc on the decode path (cudaMalloc can block until the
// device is idle).  kvq_decode_attn_static serves them from a scratch array
// that lives in this library's device image instead.
//
// The array is a file-scope __device__ variable of KVQ_STATIC_SCRATCH_BYTES
// bytes.  Every GPU on which the library's device code is loaded holds it
// until the process exits.  Host code cannot use the array's name as a
// device address, so the first call on each device looks the address up
// with cudaGetSymbolAddress while that device is current, and keeps it.
#include <cuda_runtime.h>

#include "../../include/kvq.h"
#include "kvq_host.h"

namespace {

constexpr size_t kScratchBytes = KVQ_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

kvq::DeviceOnce g_once;
void* g_scratch_ptr[kMaxDevices];

// The array's device address on the current device dev, looked up (with dev
// current) until a lookup succeeds; nullptr while none has.
void* scratch_of(int dev) {
  const bool ok = g_once.run(dev, [dev] {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return false;
    g_scratch_ptr[dev] = p;
    return true;
  });
  return ok ? g_scratch_ptr[dev] : nullptr;
}

}  // namespace

extern "C" int kvq_decode_attn_static(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* seq_lens, int num_seqs, int num_q_heads,
                                      int num_kv_heads, int head_dim, int64_t num_blocks,
                                      int block_size, const float* q_scale, int q_scale_len,
                                      const float* k_scale, int k_scale_len,
                                      const float* v_scale, int v_scale_len,
                                      int scale_granularity, int fmt, int sliding_window,
                                      unsigned flags, void* out, uint32_t* dev_status,
                                      kvq_stream_t stream) {
  const int dev = kvq::current_device();
  if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
  // Sizes whose workspace would not fit the array are refused up front.
  const size_t need =
      kvq_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, 0);
  if (need > kScratchBytes) return KVQ_ERR_WORKSPACE;
  void* scratch = scratch_of(dev);
  if (!scratch) return KVQ_ERR_CUDA;
  // The array's counters are zero at load, and every completed call leaves
  // them zero (kvq_decode_static_reset clears them after a timeout); the
  // rest is overwritten before it is read.
  return kvq_decode_attn(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                         num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                         q_scale, q_scale_len, k_scale, k_scale_len, v_scale, v_scale_len,
                         scale_granularity, fmt, sliding_window, flags, scratch, kScratchBytes,
                         out, dev_status, stream);
}

extern "C" int kvq_decode_static_reset(kvq_stream_t stream) {
  const int dev = kvq::current_device();
  if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
  void* scratch = scratch_of(dev);
  if (!scratch) return KVQ_ERR_CUDA;
  // The counter table at the array's start: an asynchronous fill, no allocation.
  if (cudaMemsetAsync(scratch, 0, KVQ_WS_COUNTER_BYTES, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return KVQ_ERR_CUDA;
  return KVQ_OK;
}
