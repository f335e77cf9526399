// kvq_decode.cu -- entry points of the paged decode attention: argument
// checks, the plan of the launch (grid, workspace layout, tensor maps) and
// the dispatch to the kernel variants, which kvq_decode_variant.cu compiles
// once per cache format and head size.
#include <atomic>
#include <mutex>

#include "kvq_decode.cuh"

namespace kvq {

extern template int launch<KVQ_FMT_E4M3, 128>(const DecodeParams&, const CUtensorMap&,
                                              const CUtensorMap&, cudaStream_t);
extern template int launch<KVQ_FMT_E4M3, 64>(const DecodeParams&, const CUtensorMap&,
                                             const CUtensorMap&, cudaStream_t);
extern template int launch<KVQ_FMT_E5M2, 128>(const DecodeParams&, const CUtensorMap&,
                                              const CUtensorMap&, cudaStream_t);
extern template int launch<KVQ_FMT_E5M2, 64>(const DecodeParams&, const CUtensorMap&,
                                             const CUtensorMap&, cudaStream_t);
extern template int launch<KVQ_FMT_BF16, 128>(const DecodeParams&, const CUtensorMap&,
                                              const CUtensorMap&, cudaStream_t);
extern template int launch<KVQ_FMT_BF16, 64>(const DecodeParams&, const CUtensorMap&,
                                             const CUtensorMap&, cudaStream_t);
#ifndef KVQ_DECODE_TC
#define KVQ_DECODE_TC 0
#endif
#ifndef KVQ_DECODE_BLK
#define KVQ_DECODE_BLK 0
#endif
namespace dtc {
// The tensor-core kernels of the FP8 caches at head size 128 (kvq_decode_tc.cu).
template <int FMT>
int launch_tc(const DecodeParams&, const CUtensorMap&, const CUtensorMap&, cudaStream_t);
extern template int launch_tc<KVQ_FMT_E4M3>(const DecodeParams&, const CUtensorMap&,
                                            const CUtensorMap&, cudaStream_t);
extern template int launch_tc<KVQ_FMT_E5M2>(const DecodeParams&, const CUtensorMap&,
                                            const CUtensorMap&, cudaStream_t);
constexpr int kCtasPerSmTc = KVQ_DTC_CTAS_PER_SM;  // CTAs per SM of the tensor-core grid
// The launch's shared memory fits the device (a large batch's plan may not).
bool fits_tc(int G, int B, int Hkv);
// Cluster size of the per-segment variant for this batch, or 0 (split).
template <int FMT>
int choose_clu(int G, int B, int Hkv, int max_blocks);
extern template int choose_clu<KVQ_FMT_E4M3>(int, int, int, int);
extern template int choose_clu<KVQ_FMT_E5M2>(int, int, int, int);
}  // namespace dtc

namespace dtb {
// The whole-block tensor-core kernel (kvq_decode_blk.cu): FP8 caches, head
// size 128, four query heads per KV head, KV heads in groups of eight.
template <int FMT>
int launch_blk(const DecodeParams&, const CUtensorMap&, const CUtensorMap&, bool, cudaStream_t);
extern template int launch_blk<KVQ_FMT_E4M3>(const DecodeParams&, const CUtensorMap&,
                                             const CUtensorMap&, bool, cudaStream_t);
extern template int launch_blk<KVQ_FMT_E5M2>(const DecodeParams&, const CUtensorMap&,
                                             const CUtensorMap&, bool, cudaStream_t);
// The launch's shared memory (with the plan of B sequences) fits the device.
bool fits_blk(int B, int Hkv);
}  // namespace dtb

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Tensor map of one cache tensor viewed as 2D: rows of head_dim elements
// (num_blocks * Hkv * 16 rows).  One box is box_rows rows (a page of one KV
// head, or a block of eight) by at most 128 bytes, swizzled so that the
// decode kernels' fragment reads are free of bank conflicts and the tensor
// cores read the 128-byte rows directly; a 256-byte bf16 row takes two
// boxes (x = 0 and x = 64).
static bool make_cache_map(CUtensorMap* m, const void* base, int fmt, int dh, uint64_t rows,
                           int box_rows = kBS) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const int elem = fmt == KVQ_FMT_BF16 ? 2 : 1;
  const int row_bytes = dh * elem;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(dh), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(row_bytes > 128 ? 128 / elem : dh),
                             static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[2] = {1, 1};
  const CUtensorMapSwizzle sw =
      row_bytes >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const CUresult r =
      enc(m, elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
          const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

#ifdef KVQ_TEST_HOOKS
// Test builds only: the stream position CTA 0's producer withholds (-1: none).
static std::atomic<int> g_withhold{-1};
#endif

}  // namespace kvq

using namespace kvq;

#ifdef KVQ_TEST_HOOKS
// Test builds only (not declared in kvq.h): make the next decodes withhold the
// copy of CTA 0's page at stream position `position` (-1: none), so that a
// bounded wait runs out and reports KVQ_DEV_WAIT_TIMEOUT.
extern "C" __attribute__((visibility("default"))) void kvq_test_withhold_page(int position) {
  g_withhold.store(position);
}
#endif

extern "C" size_t kvq_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                            int head_dim, int num_sms) {
  if (num_seqs <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads)
    return 0;
  if (head_dim != 64 && head_dim != 128) return 0;
  if (num_sms <= 0) num_sms = device_sm_count();
  if (num_sms <= 0) return 0;
  const int G = num_q_heads / num_kv_heads;
  return ws_layout(num_seqs, G, num_kv_heads, head_dim, kCtasPerSM * num_sms).total;
}

extern "C" int kvq_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* seq_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int64_t num_blocks,
                               int block_size, const float* q_scale, int q_scale_len,
                               const float* k_scale, int k_scale_len, const float* v_scale,
                               int v_scale_len, int scale_granularity, int fmt,
                               int sliding_window, unsigned flags, void* workspace,
                               size_t workspace_bytes, void* out, uint32_t* dev_status,
                               kvq_stream_t stream) {
  if (fmt < KVQ_FMT_BF16 || fmt > KVQ_FMT_E5M2) return KVQ_ERR_ARG;
  if (scale_granularity != KVQ_SCALE_PER_TENSOR && scale_granularity != KVQ_SCALE_PER_HEAD &&
      scale_granularity != KVQ_SCALE_PER_TOKEN_HEAD)
    return KVQ_ERR_ARG;
  if (flags & ~(KVQ_Q_FP8 | KVQ_CACHE_READY)) return KVQ_ERR_ARG;
  const bool q_fp8 = (flags & KVQ_Q_FP8) != 0;
  if (q_fp8 && fmt == KVQ_FMT_BF16) return KVQ_ERR_UNSUPPORTED;
  if (q_fp8 && !q_scale) return KVQ_ERR_NULL;
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0 || sliding_window < 0)
    return KVQ_ERR_ARG;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !workspace || !out)
    return KVQ_ERR_NULL;
  if (head_dim != 64 && head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (block_size != kBS) return KVQ_ERR_UNSUPPORTED;
  if (num_q_heads % num_kv_heads) return KVQ_ERR_SHAPE;
  const int G = num_q_heads / num_kv_heads;
  if (G > kMaxGroup || num_kv_heads > kMaxKvHeads) return KVQ_ERR_UNSUPPORTED;
  if (num_seqs > kMaxSeqs || num_seqs * num_kv_heads > kMaxSegments) return KVQ_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_seqs) * (max_blocks_per_seq + kPieceCost) * num_kv_heads >=
      (int64_t(1) << 31))
    return KVQ_ERR_UNSUPPORTED;
  if (num_blocks * num_kv_heads * kBS >= (int64_t(1) << 31)) return KVQ_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return KVQ_ERR_ALIGN;
  const bool token_scales = scale_granularity == KVQ_SCALE_PER_TOKEN_HEAD;
  if (fmt != KVQ_FMT_BF16) {
    if (!k_scale || !v_scale) return KVQ_ERR_NULL;
    const int64_t want = token_scales ? num_blocks * num_kv_heads * kBS
                                      : (scale_granularity == KVQ_SCALE_PER_HEAD ? num_kv_heads : 1);
    if (k_scale_len != want || v_scale_len != want) return KVQ_ERR_SHAPE;
    if (token_scales && (!aligned16(k_scale) || !aligned16(v_scale))) return KVQ_ERR_ALIGN;
  }
  if (q_scale) {
    const bool ok = token_scales ? (q_scale_len == 1 || q_scale_len == num_q_heads)
                                 : q_scale_len == (scale_granularity == KVQ_SCALE_PER_HEAD ? num_q_heads : 1);
    if (!ok) return KVQ_ERR_SHAPE;
  }
  const int sms = device_sm_count();
  if (sms <= 0) return KVQ_ERR_CUDA;
  const int64_t max_units = static_cast<int64_t>(num_seqs) * max_blocks_per_seq * num_kv_heads;
  // The tcgen05 kernel (one CTA per SM) serves FP8 caches at head size 128
  // with per-tensor or per-head scales when KVQ_DECODE_TC is set at build
  // time; by default every call runs the warp-MMA kernel, which times faster.
  const bool use_tc = KVQ_DECODE_TC && fmt != KVQ_FMT_BF16 && head_dim == 128 && !token_scales &&
                      dtc::fits_tc(G, num_seqs, num_kv_heads);
  // With KVQ_DECODE_BLK set at build time, FP8 caches at head size 128 with
  // per-tensor or per-head scales, four query heads per KV head and KV heads
  // in groups of eight run on the whole-block tensor-core kernel (one CTA per
  // SM); by default the warp-MMA kernel serves them, which times faster.
  const bool use_blk = KVQ_DECODE_BLK && !use_tc && fmt != KVQ_FMT_BF16 && head_dim == 128 && !token_scales &&
                       G == 4 && num_kv_heads % kMaxHT == 0 && dtb::fits_blk(num_seqs, num_kv_heads);
  int ctas = use_blk ? sms : (use_tc ? dtc::kCtasPerSmTc * sms : kCtasPerSM * sms);
  // Under KVQ_CACHE_READY this grid's CTAs take the slots that the previous
  // call's CTAs free as they exit, and prefetch their first pages there; the
  // CTAs still merging a split segment hold a slot each to the end.  With few
  // (sequence, KV head) segments (each split over four or more CTAs) every
  // segment has such a merger, so the grid leaves that many slots to them:
  // otherwise its last CTAs would start only after the merges, with nothing
  // prefetched, and finish last.
  const int64_t segments = static_cast<int64_t>(num_seqs) * num_kv_heads;
  if ((flags & KVQ_CACHE_READY) && !use_blk && !use_tc && 4 * segments <= ctas)
    ctas -= static_cast<int>(segments);
  const int P = static_cast<int>(std::min<int64_t>(ctas, use_blk ? max_units / kMaxHT : max_units));
  const WsLayout wl = ws_layout(num_seqs, G, num_kv_heads, head_dim, kCtasPerSM * sms);
  if (workspace_bytes < wl.total) return KVQ_ERR_WORKSPACE;

  DecodeParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.max_blocks = max_blocks_per_seq;
  p.B = num_seqs;
  p.Hq = num_q_heads;
  p.Hkv = num_kv_heads;
  p.G = G;
  p.window = sliding_window;
  p.num_blocks = num_blocks;
  p.ks = fmt == KVQ_FMT_BF16 ? nullptr : k_scale;
  p.vs = fmt == KVQ_FMT_BF16 ? nullptr : v_scale;
  p.per_head = scale_granularity == KVQ_SCALE_PER_HEAD;
  p.ts = token_scales && fmt != KVQ_FMT_BF16;
  p.P = P;
  p.early = (flags & KVQ_CACHE_READY) ? 1 : 0;
  p.qs = q_fp8 ? q_scale : nullptr;
  p.q_per_head = q_scale && q_scale_len == num_q_heads && num_q_heads > 1;
  p.logit_scale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(head_dim)));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.ws_cnt = reinterpret_cast<uint32_t*>(ws + wl.cnt);
  p.ws_ml = reinterpret_cast<float*>(ws + wl.ml);
  p.ws_o = reinterpret_cast<float*>(ws + wl.o);
  p.out = static_cast<uint16_t*>(out);
  p.status = dev_status;
  p.rows = num_blocks * num_kv_heads * kBS;
  p.n_slots = static_cast<int64_t>(kMaxHT) * kCtasPerSM * sms + static_cast<int64_t>(num_seqs) * num_kv_heads;

  const uint64_t rows = static_cast<uint64_t>(num_blocks) * num_kv_heads * kBS;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  p.clu = 0;
  p.ncl = 0;
#ifdef KVQ_TEST_HOOKS
  p.withhold = g_withhold.load();
#else
  p.withhold = -1;
#endif
  if (use_blk) {
    CUtensorMap bk, bv;
    if (!make_cache_map(&bk, k_cache, fmt, head_dim, rows, kMaxHT * kBS) ||
        !make_cache_map(&bv, v_cache, fmt, head_dim, rows, kMaxHT * kBS))
      return KVQ_ERR_CUDA;
    // Few segments split over many CTAs each: merge them all at once after a
    // grid barrier; otherwise the CTA completing a segment merges it.
    const int64_t nseg = static_cast<int64_t>(num_seqs) * (num_kv_heads / kMaxHT);
    const bool grid_merge = P > 8 * nseg;
    return fmt == KVQ_FMT_E4M3 ? dtb::launch_blk<KVQ_FMT_E4M3>(p, bk, bv, grid_merge, s)
                               : dtb::launch_blk<KVQ_FMT_E5M2>(p, bk, bv, grid_merge, s);
  }
  CUtensorMap tk, tv;
  if (!make_cache_map(&tk, k_cache, fmt, head_dim, rows) ||
      !make_cache_map(&tv, v_cache, fmt, head_dim, rows))
    return KVQ_ERR_CUDA;
  if (use_tc) {
    p.clu = fmt == KVQ_FMT_E4M3
                ? dtc::choose_clu<KVQ_FMT_E4M3>(G, num_seqs, num_kv_heads, max_blocks_per_seq)
                : dtc::choose_clu<KVQ_FMT_E5M2>(G, num_seqs, num_kv_heads, max_blocks_per_seq);
    return fmt == KVQ_FMT_E4M3 ? dtc::launch_tc<KVQ_FMT_E4M3>(p, tk, tv, s)
                               : dtc::launch_tc<KVQ_FMT_E5M2>(p, tk, tv, s);
  }
  switch (fmt) {
    case KVQ_FMT_E4M3:
      return head_dim == 128 ? launch<KVQ_FMT_E4M3, 128>(p, tk, tv, s)
                             : launch<KVQ_FMT_E4M3, 64>(p, tk, tv, s);
    case KVQ_FMT_E5M2:
      return head_dim == 128 ? launch<KVQ_FMT_E5M2, 128>(p, tk, tv, s)
                             : launch<KVQ_FMT_E5M2, 64>(p, tk, tv, s);
    default:
      return head_dim == 128 ? launch<KVQ_FMT_BF16, 128>(p, tk, tv, s)
                             : launch<KVQ_FMT_BF16, 64>(p, tk, tv, s);
  }
}
