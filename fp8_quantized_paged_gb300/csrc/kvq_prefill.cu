// kvq_prefill.cu -- prefill / prefix-hit attention over the paged cache.
//
// "10.4 KV Cache quantization: INT8, KIVI 2-bit, FP8 KV", section 10.4.2:
// prefill, decode and prefix-hit paths read the same compressed cache, with
// the dequantization fused into QK and PV.  Sequence b holds L_b tokens, the
// last n_b of them new; query token j of the chunk sits at position
// pos = L_b - n_b + j and attends causally to the cached tokens [lo, pos]
// (lo from the sliding window), the earlier ones being a cached prefix.
//
// Work decomposition: one CTA per (sequence, KV head, tile of 64 query rows);
// a row is a (query token, query head of the group) pair, so a tile holds
// 64 / G tokens.  Later tiles attend to more tokens and are launched first.
//   warp 4 (producer): lane s owns ring slot s and issues the TMA loads of
//   the K and V pages of positions s, s + S, ... of the tile's page range.
//   warps 0-3 (consumers): 16 rows each; every warp reads every page into
//   registers and frees the slot (the empty barrier counts four arrivals).
//   QK: Q is the m16n8k16 A operand (bf16 -> f16, exact in f16's normal
//   range), the K page the B operand (two 8-token n-tiles; FP8 -> f16 exact),
//   the head dims permuted alike on both sides so that a lane reads its K
//   bytes contiguously.  The causal and window masks apply per row; the
//   online softmax is in the log2 domain with sK folded into the logit scale
//   and a lazy rescale of O.  PV: the probabilities (f16; for the bf16 cache
//   bf16 high and low parts, two MMAs) are the A operand as they leave the
//   accumulators, the V page the B operand, head dim n of n-tile nt at
//   g * DH/8 + nt.
#include <mutex>

#include "kvq_decode.cuh"

namespace kvq {

constexpr int kPfRows = 16 * kConsumerWarps;  // query rows per CTA

struct PrefillParams {
  const uint16_t* q;         // [total_q][Hq][DH]
  const int32_t* cu_q;       // [B + 1]
  const int32_t* block_tables;
  const int32_t* seq_lens;
  int max_blocks;
  int B, Hq, Hkv, G;
  int window;
  int tiles;                 // query tiles per sequence
  int tpc;                   // query tiles per CTA (the tcgen05 kernel: 1 or 2)
  int64_t num_blocks;
  int64_t rows;              // rows of the cache tensor maps
  int64_t total_q;
  const float* ks;           // [1], [Hkv], or the scale caches [num_blocks][Hkv][16] (ts)
  const float* vs;
  int per_head;
  int ts;                    // per-(token, KV head) scales
  const float* qs;           // KVQ_Q_FP8: query scales, [1] or [Hq]; else null
  int q_per_head;
  float logit_scale;         // log2(e) / sqrt(dh)
  uint16_t* out;             // [total_q][Hq][DH]
  uint32_t* status;
};

template <int FMT, int DH>
struct PfSmem {
  using C = Cfg<FMT, DH>;
  static constexpr int S = C::kStages < 32 ? C::kStages : 32;  // one producer lane per slot
  static constexpr size_t ring = 0;
  static constexpr size_t bars = ring + static_cast<size_t>(S) * C::kSlot;  // full[S], empty[S]
  static constexpr size_t flags = bars + 2 * S * sizeof(uint64_t);          // bad[S], abort, last[S]
  static constexpr size_t total = flags + (2 * S + 1) * sizeof(uint32_t) + 1024;
};

// Q rows g and g + 8 of the warp as m16n8k16 A fragments: step kk holds dims
// t * DH/4 + 4kk + {0, 1} (a0 row g, a1 row g+8) and + {2, 3} (a2, a3),
// f16 for the FP8 caches, bf16 as is for the bf16 cache; absent rows zero.
template <int FMT, int DH>
KVQ_DEVI void prefill_q_fragments(const PrefillParams& p, int64_t row_g, int64_t row_g8, int t,
                                  uint32_t (&qa)[DH / 16][4]) {
  uint32_t w[2][DH / 8];
  const int64_t rows[2] = {row_g, row_g8};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const bool ok = rows[r] >= 0 &&
                    guard(rows[r] < p.total_q * p.Hq, p.status, 11);
    const uint4* src = reinterpret_cast<const uint4*>(p.q + (ok ? rows[r] : 0) * DH + t * (DH / 4));
#pragma unroll
    for (int i = 0; i < DH / 32; ++i) {
      const uint4 v = ok ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
      w[r][4 * i] = v.x; w[r][4 * i + 1] = v.y; w[r][4 * i + 2] = v.z; w[r][4 * i + 3] = v.w;
    }
  }
#pragma unroll
  for (int kk = 0; kk < DH / 16; ++kk) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint32_t lo = w[r][2 * kk], hi = w[r][2 * kk + 1];  // dims +{0,1}, +{2,3}
      if (FMT == KVQ_FMT_BF16) {
        qa[kk][r] = lo;
        qa[kk][2 + r] = hi;
      } else {
        qa[kk][r] = f32x2_to_f16x2(bf16lo_to_f32(lo), bf16hi_to_f32(lo));
        qa[kk][2 + r] = f32x2_to_f16x2(bf16lo_to_f32(hi), bf16hi_to_f32(hi));
      }
    }
  }
}

template <int FMT, int DH>
__global__ void __launch_bounds__(kThreads, 2)
    prefill_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  using C = Cfg<FMT, DH>;
  using SL = PfSmem<FMT, DH>;
  using R = PageRegs<FMT, DH>;
  constexpr int S = SL::S;
  constexpr int NT = DH / 8;  // PV n-tiles
  constexpr bool BF = FMT == KVQ_FMT_BF16;
  static_assert(S <= 32, "one producer lane per ring slot");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem + SL::ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SL::bars);
  uint64_t* empty = full + S;
  uint32_t* bad_s = reinterpret_cast<uint32_t*>(smem + SL::flags);
  volatile uint32_t* abort_flag = bad_s + S;
  int32_t* last_s = reinterpret_cast<int32_t*>(bad_s + S + 1);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < S) {
    mbar_init(&full[tid], 1);
    mbar_init(&empty[tid], kConsumerWarps);
    last_s[tid] = -1;
    fence_mbar_init();
  } else if (tid == S) {
    *abort_flag = 0u;
  }
  if (warp == kConsumerWarps && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  pdl_wait();  // q, caches, tables and lengths may come from the previous kernel
  pdl_allow_next();

  const int b = blockIdx.z, gkv = blockIdx.y;
  const int tile = p.tiles - 1 - static_cast<int>(blockIdx.x);  // longest tiles first
  const int TQ = kPfRows / p.G;                                    // query tokens per tile
  const int q0 = __ldg(p.cu_q + b);
  const int n = __ldg(p.cu_q + b + 1) - q0;
  const int j0 = tile * TQ;
  // a chunk longer than the grid covers (max_q_len): its later rows stay unwritten
  if (blockIdx.x == 0 && gkv == 0 && tid == 0 && n > p.tiles * TQ)
    flag_status(p.status, KVQ_DEV_BAD_QLEN);
  if (n <= 0 || j0 >= n) return;  // the whole CTA: nothing of this sequence here
  const int j1 = min(n, j0 + TQ);
  const int L = __ldg(p.seq_lens + b);
  const bool len_ok = L >= n && L <= p.max_blocks * kBS;
  __syncthreads();  // barriers initialised
  if (!len_ok) {
    if (tile == 0 && gkv == 0 && tid == 0) flag_status(p.status, KVQ_DEV_BAD_SEQLEN);
    // zero this tile's output rows of this KV head's query heads
    for (int i = tid; i < (j1 - j0) * p.G * DH; i += kThreads) {
      const int r = i / DH, d = i - r * DH;
      const int64_t orow = static_cast<int64_t>(q0 + j0 + r / p.G) * p.Hq + gkv * p.G + r % p.G;
      if (guard(orow >= 0 && orow < p.total_q * p.Hq, p.status, 12)) p.out[orow * DH + d] = 0;
    }
    return;
  }
  const int base = L - n;                        // position of query token 0
  const int pos_first = base + j0, pos_last = base + j1 - 1;
  const int p_begin = window_lo(p.window, pos_first + 1) / kBS;
  const int npages = pos_last / kBS - p_begin + 1;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane < S) {
      int it = 0;
      for (int i = lane; i < npages; i += S, ++it) {
        if (it > 0 && !wait_or_abort(&empty[lane], static_cast<uint32_t>((it - 1) & 1), abort_flag)) {
          if (!*abort_flag) {
            *abort_flag = 1u;
            flag_status(p.status, KVQ_DEV_WAIT_TIMEOUT);
          }
          break;
        }
        const int col = p_begin + i;
        int blk = -1;
        if (guard(col >= 0 && col < p.max_blocks, p.status, 13))
          blk = __ldg(p.block_tables + static_cast<int64_t>(b) * p.max_blocks + col);
        const bool bad = blk < 0 || blk >= p.num_blocks;
        if (bad) flag_status(p.status, KVQ_DEV_BAD_BLOCK);
        int32_t row = ((bad ? 0 : blk) * p.Hkv + gkv) * kBS;
        bool skip = bad;
        if (!guard(row >= 0 && row + kBS <= p.rows, p.status, 14)) {
          row = 0;
          skip = true;
        }
        bad_s[lane] = skip ? 1u : 0u;
        uint8_t* dst = ring + lane * C::kSlot;
        mbar_arrive_expect_tx(&full[lane], C::kSlot);
        // K and V pages are read by every query tile of the sequence: keep the
        // default L2 policy (they are re-read by the other tiles' CTAs).
        if (C::kRow > 128) {
          tma_load_2d(dst, &tmk, 0, row, &full[lane]);
          tma_load_2d(dst + C::kPage / 2, &tmk, 64, row, &full[lane]);
          tma_load_2d(dst + C::kPage, &tmv, 0, row, &full[lane]);
          tma_load_2d(dst + C::kPage + C::kPage / 2, &tmv, 64, row, &full[lane]);
        } else {
          tma_load_2d(dst, &tmk, 0, row, &full[lane]);
          tma_load_2d(dst + C::kPage, &tmv, 0, row, &full[lane]);
        }
        last_s[lane] = i;
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3;
    // this lane's rows: tile rows 16 warp + g and + 8 -> (token, head)
    int jr[2], pos[2], lo[2];
    int64_t qrow[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int tr = 16 * warp + g + 8 * r;
      jr[r] = j0 + tr / p.G;
      const bool live = jr[r] < j1;
      pos[r] = live ? base + jr[r] : -1;  // a missing row attends to nothing
      lo[r] = live ? window_lo(p.window, pos[r] + 1) : 0;
      qrow[r] = live ? static_cast<int64_t>(q0 + jr[r]) * p.Hq + gkv * p.G + tr % p.G : -1;
    }
    // the warp's rows span positions [wlo, whi]
    const int wr_first = 16 * warp, wr_last = 16 * warp + 15;
    const int wj_first = j0 + wr_first / p.G;
    const int wj_last = min(j1 - 1, j0 + wr_last / p.G);
    const int whi = base + wj_last;
    const int wlo = window_lo(p.window, base + wj_first + 1);
    const bool warp_live = wj_first < j1;

    uint32_t qa[DH / 16][4];
    prefill_q_fragments<FMT, DH>(p, qrow[0], qrow[1], t, qa);
    const float sk = BF ? 1.f : __ldg(p.ks + (p.per_head ? gkv : 0));
    const float sv = BF ? 1.f : __ldg(p.vs + (p.per_head ? gkv : 0));
    const float lscale = sk * p.logit_scale;

    float o[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    bool aborted = false;

    for (int i = 0; i < npages; ++i) {
      const int slot = i % S;
      const uint32_t par = static_cast<uint32_t>((i / S) & 1);
      const bool ok = !aborted && wait_or_abort(&full[slot], par, abort_flag);
      if (!__all_sync(kFull, ok)) {
        if (!aborted && lane == 0 && !*abort_flag) {
          *abort_flag = 1u;
          flag_status(p.status, KVQ_DEV_WAIT_TIMEOUT);
        }
        aborted = true;
        break;
      }
      const int tok0 = (p_begin + i) * kBS;
      const bool bad = bad_s[slot] != 0u;
      const bool needed = warp_live && !bad && tok0 <= whi && tok0 + kBS > wlo;
      R pr;
      if (needed) {
        const uint32_t kp = smem_u32(ring + slot * C::kSlot);
        // V rows of tokens past the sequence are zeroed (they may hold
        // anything, and p = 0 would not clear a NaN)
        load_page<FMT, DH>(kp, kp + C::kPage, g, t, tok0, 0, L, false, pr);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (!needed) continue;

      // ---- S = Q K^T, two n-tiles of 8 tokens
      float s[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const uint32_t* kw = nt ? pr.k1 : pr.k0;  // token rows g (+ 8)
          if (BF) {
            mma_bf16(s[nt], qa[kk], kw[2 * kk], kw[2 * kk + 1]);
          } else {
            uint32_t b0, b1;
            fp8x4_to_f16x2x2<FMT>(kw[kk], b0, b1);
            mma_f16(s[nt], qa[kk], b0, b1);
          }
        }
      }
      // ---- mask, online softmax (rows g: c0, c1; g + 8: c2, c3)
      float x[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int kpos = tok0 + 8 * nt + 2 * t + (c & 1);
          const int r = c >> 1;
          const bool valid = kpos >= lo[r] && kpos <= pos[r];
          x[nt][c] = valid ? s[nt][c] * lscale : -INFINITY;
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float mx = fmaxf(fmaxf(x[0][2 * r], x[0][2 * r + 1]), fmaxf(x[1][2 * r], x[1][2 * r + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
        if (mx > m[r] + kRescaleThreshold) {  // same decision on the row's four lanes
          const float a = (m[r] == -INFINITY) ? 0.f : fast_exp2(m[r] - mx);
          l[r] *= a;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            o[nt][2 * r] *= a;
            o[nt][2 * r + 1] *= a;
          }
          m[r] = mx;
        }
      }
      float pv[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float mr = m[c >> 1];
          pv[nt][c] = (x[nt][c] == -INFINITY) ? 0.f : fast_exp2(x[nt][c] - mr);
          l[c >> 1] += pv[nt][c];
        }
      // ---- O += P V: P (16 rows x 16 tokens) as the A operand
      uint32_t pa[4], pl[4];  // pl: the bf16 remainders p - bf16(p) (bf16 cache)
      if (BF) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x0 = pv[i >> 1][2 * (i & 1)], x1 = pv[i >> 1][2 * (i & 1) + 1];
          pa[i] = f32x2_to_bf16x2(x0, x1);
          pl[i] = f32x2_to_bf16x2(x0 - bf16lo_to_f32(pa[i]), x1 - bf16hi_to_f32(pa[i]));
        }
      } else {
        pa[0] = f32x2_to_f16x2(pv[0][0], pv[0][1]);
        pa[1] = f32x2_to_f16x2(pv[0][2], pv[0][3]);
        pa[2] = f32x2_to_f16x2(pv[1][0], pv[1][1]);
        pa[3] = f32x2_to_f16x2(pv[1][2], pv[1][3]);
      }
      // V rows held: v[0] token 2t, v[1] 2t + 8, v[2] 2t + 1, v[3] 2t + 9
#pragma unroll
      for (int w = 0; w < R::VB / 4; ++w) {
        if (BF) {  // word w: dims g*DH/8 + 2w, +1 -> n-tiles 2w, 2w + 1; P as hi + lo
          const uint32_t b00 = prmt(pr.v[0][w], pr.v[2][w], 0x5410u);
          const uint32_t b01 = prmt(pr.v[1][w], pr.v[3][w], 0x5410u);
          const uint32_t b10 = prmt(pr.v[0][w], pr.v[2][w], 0x7632u);
          const uint32_t b11 = prmt(pr.v[1][w], pr.v[3][w], 0x7632u);
          mma_bf16(o[2 * w], pa, b00, b01);
          mma_bf16(o[2 * w], pl, b00, b01);
          mma_bf16(o[2 * w + 1], pa, b10, b11);
          mma_bf16(o[2 * w + 1], pl, b10, b11);
        } else {  // word w: dims g*DH/8 + 4w .. +3 -> n-tiles 4w .. 4w + 3
          uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
          fp8x4_to_f16x2x2<FMT>(prmt(pr.v[0][w], pr.v[2][w], 0x5140u), a0, a1);
          fp8x4_to_f16x2x2<FMT>(prmt(pr.v[1][w], pr.v[3][w], 0x5140u), c0, c1);
          fp8x4_to_f16x2x2<FMT>(prmt(pr.v[0][w], pr.v[2][w], 0x7362u), a2, a3);
          fp8x4_to_f16x2x2<FMT>(prmt(pr.v[1][w], pr.v[3][w], 0x7362u), c2, c3);
          mma_f16(o[4 * w], pa, a0, c0);
          mma_f16(o[4 * w + 1], pa, a1, c1);
          mma_f16(o[4 * w + 2], pa, a2, c2);
          mma_f16(o[4 * w + 3], pa, a3, c3);
        }
      }
    }

    // ---- normalise and store: lane holds, per row, dims (2t) DH/8 + nt and
    // (2t + 1) DH/8 + nt for every n-tile nt
    if (!aborted) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        l[r] += __shfl_xor_sync(kFull, l[r], 1);
        l[r] += __shfl_xor_sync(kFull, l[r], 2);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (qrow[r] < 0 || !guard(qrow[r] < p.total_q * p.Hq, p.status, 15)) continue;
        const float f = l[r] > 0.f ? sv / l[r] : 0.f;
        uint16_t* dst = p.out + qrow[r] * DH;
#pragma unroll
        for (int c = 0; c < 2; ++c) {  // the runs at (2t + c) DH/8
          uint32_t packed[NT / 2];
#pragma unroll
          for (int nt = 0; nt < NT; nt += 2)
            packed[nt / 2] = f32x2_to_bf16x2(o[nt][2 * r + c] * f, o[nt + 1][2 * r + c] * f);
          uint4* d4 = reinterpret_cast<uint4*>(dst + (2 * t + c) * (DH / 8));
#pragma unroll
          for (int v = 0; v < NT / 8; ++v)
            d4[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        }
      }
    }
  }
  __syncthreads();
  // After an abort, wait (bounded) for copies still in flight before exit.
  if (*abort_flag && tid == 0) {
    for (int s = 0; s < S; ++s)
      if (last_s[s] >= 0) mbar_wait(&full[s], static_cast<uint32_t>((last_s[s] / S) & 1));
  }
}

}  // namespace kvq

#include "kvq_prefill_tc.cuh"

namespace kvq {

static PFN_cuTensorMapEncodeTiled_v12000 pf_encode_fn() {
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

// The decode's tensor map of one cache tensor (rows of head_dim elements,
// 16-row boxes of at most 128 bytes, swizzled alike).
static bool pf_cache_map(CUtensorMap* m, const void* base, int fmt, int dh, uint64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = pf_encode_fn();
  if (!enc) return false;
  const int elem = fmt == KVQ_FMT_BF16 ? 2 : 1;
  const int row_bytes = dh * elem;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(dh), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(row_bytes > 128 ? 128 / elem : dh), kBS};
  const cuuint32_t es[2] = {1, 1};
  const CUtensorMapSwizzle sw =
      row_bytes >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return enc(m, elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
             const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, int DH>
static int prefill_launch(const PrefillParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                          cudaStream_t s) {
  constexpr size_t smem = PfSmem<FMT, DH>::total;
  static DeviceOnce once;  // the kernel's attributes, once per device (again after a failure)
  if (!once.run(current_device(), [] {
        return cudaFuncSetAttribute(prefill_kernel<FMT, DH>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem)) == cudaSuccess &&
               cudaFuncSetAttribute(prefill_kernel<FMT, DH>,
                                    cudaFuncAttributePreferredSharedMemoryCarveout,
                                    cudaSharedmemCarveoutMaxShared) == cudaSuccess;
      }))
    return KVQ_ERR_CUDA;
  const dim3 grid(p.tiles, p.Hkv, p.B), block(kThreads);
  if (launch_pdl(prefill_kernel<FMT, DH>, grid, block, smem, s, p, tk, tv) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// The FP8 caches' prefill on the tcgen05 tensor cores (two tiles of 128
// query rows a CTA).
template <int FMT, int DH>
static int prefill_tc_launch(PrefillParams p, int max_q_len, const CUtensorMap& tk,
                             const CUtensorMap& tv, cudaStream_t s) {
  constexpr size_t smem = tc::Layout<DH, false>::total, smem_ts = tc::Layout<DH, true>::total;
  static DeviceOnce once;  // the kernels' attribute, once per device (again after a failure)
  if (!once.run(current_device(), [] {
        return cudaFuncSetAttribute(tc::prefill_tc_kernel<FMT, DH, false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem)) == cudaSuccess &&
               cudaFuncSetAttribute(tc::prefill_tc_kernel<FMT, DH, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem_ts)) == cudaSuccess;
      }))
    return KVQ_ERR_CUDA;
  const int TQ = tc::kRows / p.G;
  p.tiles = (max_q_len + TQ - 1) / TQ;
  // Two tiles a CTA share each converted key block and take about 1.15
  // times one tile's time per block (measured: 2 x 4 x 128 query rows per
  // KV head over 32768 keys, 607 against 526 us): pairs only when that
  // saves waves of CTAs (one CTA per SM).
  const int sms = device_sm_count();
  if (sms <= 0) return KVQ_ERR_CUDA;
  const int64_t cta1 = static_cast<int64_t>(p.tiles) * p.Hkv * p.B;
  const int64_t cta2 = static_cast<int64_t>((p.tiles + tc::kTiles - 1) / tc::kTiles) * p.Hkv * p.B;
  const int64_t waves1 = (cta1 + sms - 1) / sms, waves2 = (cta2 + sms - 1) / sms;
  p.tpc = 8 * waves2 < 7 * waves1 ? tc::kTiles : 1;
  const dim3 grid((p.tiles + p.tpc - 1) / p.tpc, p.Hkv, p.B), block(tc::kThreadsTc);
  const cudaError_t e =
      p.ts ? launch_pdl(tc::prefill_tc_kernel<FMT, DH, true>, grid, block, smem_ts, s, p, tk, tv)
           : launch_pdl(tc::prefill_tc_kernel<FMT, DH, false>, grid, block, smem, s, p, tk, tv);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq

using namespace kvq;

extern "C" int kvq_prefill_attn(const void* q, const int32_t* cu_q_lens, int64_t num_q_tokens,
                                int max_q_len, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* seq_lens, int num_seqs, int num_q_heads,
                                int num_kv_heads, int head_dim, int64_t num_blocks,
                                int block_size, const float* q_scale, int q_scale_len,
                                const float* k_scale, int k_scale_len, const float* v_scale,
                                int v_scale_len, int scale_granularity, int fmt,
                                int sliding_window, unsigned flags, void* out,
                                uint32_t* dev_status, kvq_stream_t stream) {
  if (fmt < KVQ_FMT_BF16 || fmt > KVQ_FMT_E5M2) return KVQ_ERR_ARG;
  if (scale_granularity != KVQ_SCALE_PER_TENSOR && scale_granularity != KVQ_SCALE_PER_HEAD &&
      scale_granularity != KVQ_SCALE_PER_TOKEN_HEAD)
    return KVQ_ERR_ARG;
  if (flags & ~KVQ_Q_FP8) return KVQ_ERR_ARG;
  const bool token_scales = scale_granularity == KVQ_SCALE_PER_TOKEN_HEAD;
  const bool q_fp8 = (flags & KVQ_Q_FP8) != 0;
  // per-(token, head) scales and the FP8-domain query exist for the FP8 caches only
  if ((token_scales || q_fp8) && fmt == KVQ_FMT_BF16) return KVQ_ERR_ARG;
  if (q_fp8 && !q_scale) return KVQ_ERR_NULL;
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0 || sliding_window < 0 || num_q_tokens < 0 || max_q_len < 0)
    return KVQ_ERR_ARG;
  if (!q || !cu_q_lens || !k_cache || !v_cache || !block_tables || !seq_lens || !out)
    return KVQ_ERR_NULL;
  if (head_dim != 64 && head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (block_size != kBS) return KVQ_ERR_UNSUPPORTED;
  if (num_q_heads % num_kv_heads) return KVQ_ERR_SHAPE;
  const int G = num_q_heads / num_kv_heads;
  if (G > kMaxGroup || (G & (G - 1))) return KVQ_ERR_UNSUPPORTED;  // 1, 2, 4 or 8
  if (num_seqs > 65535 || num_kv_heads > 65535) return KVQ_ERR_UNSUPPORTED;
  if (num_blocks * num_kv_heads * kBS >= (int64_t(1) << 31)) return KVQ_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks_per_seq) * kBS >= (int64_t(1) << 30))
    return KVQ_ERR_UNSUPPORTED;
  if (num_q_tokens * num_q_heads >= (int64_t(1) << 40)) return KVQ_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u) || (reinterpret_cast<uintptr_t>(cu_q_lens) & 3u))
    return KVQ_ERR_ALIGN;
  if (fmt != KVQ_FMT_BF16) {
    if (!k_scale || !v_scale) return KVQ_ERR_NULL;
    const int64_t want = token_scales ? num_blocks * num_kv_heads * kBS
                                      : (scale_granularity == KVQ_SCALE_PER_HEAD ? num_kv_heads : 1);
    if (k_scale_len != want || v_scale_len != want) return KVQ_ERR_SHAPE;
    if (token_scales && (!aligned16(k_scale) || !aligned16(v_scale))) return KVQ_ERR_ALIGN;
  }
  if (q_fp8 && q_scale_len != 1 && q_scale_len != num_q_heads) return KVQ_ERR_SHAPE;
  if (num_q_tokens == 0 || max_q_len == 0) return KVQ_OK;
  const int TQ = kPfRows / G;
  const int64_t tiles = (static_cast<int64_t>(max_q_len) + TQ - 1) / TQ;
  if (tiles > (int64_t(1) << 31) - 1) return KVQ_ERR_UNSUPPORTED;

  PrefillParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.cu_q = cu_q_lens;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.max_blocks = max_blocks_per_seq;
  p.B = num_seqs;
  p.Hq = num_q_heads;
  p.Hkv = num_kv_heads;
  p.G = G;
  p.window = sliding_window;
  p.tiles = static_cast<int>(tiles);
  p.tpc = 1;
  p.num_blocks = num_blocks;
  p.rows = num_blocks * num_kv_heads * kBS;
  p.total_q = num_q_tokens;
  p.ks = fmt == KVQ_FMT_BF16 ? nullptr : k_scale;
  p.vs = fmt == KVQ_FMT_BF16 ? nullptr : v_scale;
  p.per_head = scale_granularity == KVQ_SCALE_PER_HEAD;
  p.ts = token_scales ? 1 : 0;
  p.qs = q_fp8 ? q_scale : nullptr;
  p.q_per_head = q_fp8 && q_scale_len == num_q_heads && num_q_heads > 1;
  p.logit_scale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(head_dim)));
  p.out = static_cast<uint16_t*>(out);
  p.status = dev_status;

  CUtensorMap tk, tv;
  const uint64_t rows = static_cast<uint64_t>(p.rows);
  if (!pf_cache_map(&tk, k_cache, fmt, head_dim, rows) ||
      !pf_cache_map(&tv, v_cache, fmt, head_dim, rows))
    return KVQ_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (fmt) {
    case KVQ_FMT_E4M3:
      return head_dim == 128 ? prefill_tc_launch<KVQ_FMT_E4M3, 128>(p, max_q_len, tk, tv, s)
                             : prefill_tc_launch<KVQ_FMT_E4M3, 64>(p, max_q_len, tk, tv, s);
    case KVQ_FMT_E5M2:
      return head_dim == 128 ? prefill_tc_launch<KVQ_FMT_E5M2, 128>(p, max_q_len, tk, tv, s)
                             : prefill_tc_launch<KVQ_FMT_E5M2, 64>(p, max_q_len, tk, tv, s);
    default:
      return head_dim == 128 ? prefill_launch<KVQ_FMT_BF16, 128>(p, tk, tv, s)
                             : prefill_launch<KVQ_FMT_BF16, 64>(p, tk, tv, s);
  }
}
