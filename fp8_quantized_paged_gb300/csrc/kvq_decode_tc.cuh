// kvq_decode_tc.cuh -- paged GQA decode attention over the FP8 caches on the
// 5th-generation tensor cores: QK^T and PV as tcgen05 MMAs straight on the
// FP8 pages, accumulators in tensor memory.  Head size 128, per-tensor or
// per-KV-head scales, the bf16 query or the FP8-domain query.
//
// "10.4 KV Cache quantization: INT8, KIVI 2-bit, FP8 KV", section 10.4.2:
// P = softmax(Q K^T / sqrt(dh) + mask), O = P V^, on the efficient path that
// reads the compressed KV once and feeds QK, PV and an online softmax
// directly; section 10.4.5: K^ = cast_float(K_fp8) * sK.  sK goes into the
// logit scale and sV onto the normalised output, so the MMAs work on the
// cache's codes as they arrive.
//
// Work decomposition: the persistent grid and the cost-balanced split of the
// KV-head pages among the CTAs are those of kvq_decode.cuh (same plan, same
// partial-state workspace, same in-kernel merge by the CTA that completes a
// segment).  Inside a CTA the pages of one (sequence, KV head) piece go in
// tiles of up to 8 pages (128 tokens):
//   warp 4 (producer): block ids of 4 tiles at once (one page per lane), TMA
//     loads of each tile's K and V pages into a ring of tile stages (the
//     128-byte-swizzled page boxes, 8 pages = one 128-row operand).
//   warp 5 (MMA): allocates the tensor memory; one lane issues per tile
//     S^T = K Q^T (M = 128 tokens, N = query pieces of the group's heads,
//     K = 128 dims in 4 steps of 32) and, once the tile's probabilities are
//     in shared memory, O^T += V^T P^T (M = 128 dims with V as the MN-major
//     A operand -- the page layout itself --, N = probability pieces of the
//     heads, K = 128 tokens), completions signalled by tcgen05.commit.
//   warps 0-3 (softmax; thread r = token r of a tile = TMEM lane r): the
//     logits from S, the causal/window and page masks, an online softmax in
//     the log2 domain with one running maximum per head shared by the CTA
//     (lazily raised: only when a tile exceeds it by 2^8), the probabilities
//     into a P^T tile; at a piece's end thread d reads row d of O^T (dim d).
// Precision.  The tensor cores take 8-bit operands, so the bf16 query goes in
// as three E4M3 pieces of a per-head power-of-two scaling 2^a q (exact for
// every element within 2^18 of the head's largest) and the probabilities
// p <= 2^8 as four E4M3 pieces p1 + p2/16 + p3/256 + p4/4096 (each piece the
// nearest code to 16 x the remaining residual, about 2^-16 relative, the
// error below 2^-21 absolute); the pieces accumulate in separate fp32 columns
// and are summed with their powers of two.  Under KVQ_Q_FP8 the query is one
// piece: its codes in the cache's format, scaled by q_scale.
// Every wait is bounded; a timeout sets KVQ_DEV_WAIT_TIMEOUT, the roles stop
// at the same named barriers, and the CTA waits (bounded) for its copies and
// MMAs in flight before it frees the tensor memory.
#pragma once

#include "kvq_decode.cuh"
#include "kvq_tc.cuh"

namespace kvq {
namespace dtc {

using namespace tc;

constexpr int kDH = 128;                      // head size of this kernel
constexpr int kTilePages = 8;                 // pages per tile
constexpr int kTileTok = kTilePages * kBS;    // 128 tokens: the M of S^T, the K of PV
constexpr int kPageB = kBS * kDH;             // bytes of one FP8 page (2 KB)
constexpr int kHalf = kTilePages * kPageB;    // K (or V) pages of one tile, 16 KB
constexpr int kStageB = 2 * kHalf;            // one ring stage: K then V
constexpr int kThreadsD = 224;  // warps 0-3 softmax, 4 producer, 5 QK^T issuer, 6 PV issuer
constexpr int kSoftThreads = 128;
#ifndef KVQ_DTC_STAGES
#define KVQ_DTC_STAGES 4
#endif
constexpr int kNst = KVQ_DTC_STAGES;
constexpr int kCtasPerSmD = KVQ_DTC_CTAS_PER_SM;
constexpr int kQPieces = 3;
constexpr int kPPieces = 4;
constexpr int kCluMax = 16;  // largest cluster of the per-segment (cluster) variant
constexpr uint32_t kSoftBar = 1;  // named barrier of the 128 softmax threads

// Shared memory and tensor memory of the variant for groups of up to GW
// query heads (GW = 4 or 8).
template <int GW>
struct DLay {
  static constexpr int NS = GW <= 4 ? 16 : 32;       // S^T columns (query pieces x heads)
  static constexpr int NO = kPPieces * GW;           // O^T columns (probability pieces x heads)
  static constexpr uint32_t kCols = GW <= 4 ? 64 : 128;  // 2 NS + NO, rounded to a power of 2
  static constexpr size_t ring = 0;
  static constexpr size_t qbuf = ring + static_cast<size_t>(kNst) * kStageB;  // [2][NS][128]
  static constexpr size_t qBytes = static_cast<size_t>(NS) * 128;
  static constexpr size_t pbuf = qbuf + 2 * qBytes;                           // [kNst][NO][128]
  static constexpr size_t pBytes = static_cast<size_t>(NO) * 128;
  static constexpr size_t bars = pbuf + kNst * pBytes;
  // full[kNst], empty[kNst], sfull[2], sfree[2], pfull[kNst], qfull[2], fin, mcopy, pvfin
  static constexpr int kBars = 3 * kNst + 9;
  static constexpr size_t misc = bars + kBars * sizeof(uint64_t);
  // misc u32: np[kNst], bad[kNst], issued[kNst], abort, tmem, merge, u0, u1, qexp[2][8], mcopy issued
  static constexpr int kMiscWords = 3 * kNst + 5 + 16 + 1;
  static constexpr size_t red = (misc + kMiscWords * 4 + 15) & ~size_t(15);
  // red: warp maxima [4][8], warp sums [4][8], plan scan scratch [8]
  static constexpr size_t plan = red + (2 * 32 + 8) * 4;
  __host__ __device__ static size_t plan_end(int B, int Hkv) {
    return (plan + (3 * static_cast<size_t>(B) + 2) * 4 + 2 * static_cast<size_t>(Hkv) * 4 + 15) &
           ~size_t(15);
  }
  __host__ __device__ static size_t total(int B, int Hkv) { return plan_end(B, Hkv) + 1024; }
  // cluster variant: the leader's merge area after the plan, (m, l) [kCluMax][GW]
  // then o [kCluMax][GW][kDH]
  static constexpr size_t mgBytes = static_cast<size_t>(kCluMax) * GW * (8 + kDH * 4);
  __host__ __device__ static size_t total_clu(int B, int Hkv) {
    return plan_end(B, Hkv) + mgBytes + 1024;
  }
};

KVQ_DEVI uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
KVQ_DEVI uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
KVQ_DEVI void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
KVQ_DEVI void st_cluster_v2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
KVQ_DEVI void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
KVQ_DEVI void cluster_wait_acquire() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Byte offset of byte c of row r in a 128-byte-swizzled tile.
KVQ_DEVI uint32_t sw_off(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((((c >> 4) ^ (r & 7))) << 4) + (c & 15));
}

// The pieces of the CTA's page range [u0, u1): piece = the part of one
// (sequence, KV head) segment in the range, tile = up to 8 of its pages.
struct TileIt {
  int64_t u, u1;  // the current piece starts at unit u
  int b, gkv, pages, p0, n;  // its segment (b, gkv) of `pages` pages; pages [p0, p0 + n) of it
  int pp, np;     // the tile: pages [pp, pp + np) of the piece
  int piece, t;   // piece and tile counters of the CTA
  bool valid;

  KVQ_DEVI void piece_at(const int32_t* seq_off, int B, int Hkv) {
    b = find_seq(seq_off, B, u);
    pages = (seq_off[b + 1] - seq_off[b]) / Hkv;
    const int r = static_cast<int>(u - seq_off[b]);
    gkv = pages > 0 ? r / pages : 0;
    p0 = r - gkv * pages;
    n = static_cast<int>((u1 - u) < (pages - p0) ? (u1 - u) : (pages - p0));
    pp = 0;
    np = n < kTilePages ? n : kTilePages;
    valid = pages > 0 && n > 0;
  }
  KVQ_DEVI void start(const int32_t* seq_off, int B, int Hkv, int64_t u0_, int64_t u1_) {
    u = u0_;
    u1 = u1_;
    piece = 0;
    t = 0;
    valid = u < u1;
    if (valid) piece_at(seq_off, B, Hkv);
  }
  KVQ_DEVI bool first() const { return pp == 0; }
  KVQ_DEVI bool last() const { return pp + np == n; }
  KVQ_DEVI void next(const int32_t* seq_off, int B, int Hkv) {
    ++t;
    if (pp + np < n) {
      pp += np;
      np = (n - pp) < kTilePages ? (n - pp) : kTilePages;
      return;
    }
    u += n;
    ++piece;
    valid = u < u1;
    if (valid) piece_at(seq_off, B, Hkv);
  }
};

KVQ_DEVI float pow2i(int a) { return __int_as_float((a + 127) << 23); }  // -126 <= a <= 127

// Two E4M3 codes (low byte first) back to binary32.
KVQ_DEVI void dec_e4m3x2(uint32_t two, float& lo, float& hi) {
  const uint32_t h = fp8x2_to_f16x2<KVQ_FMT_E4M3>(static_cast<uint16_t>(two));
  lo = f16lo_to_f32(h);
  hi = f16hi_to_f32(h);
}

// The four E4M3 pieces of two probabilities a, b in [0, 2^8]: codes c[k]
// (low byte a, high byte b) with a = d1 + d2/16 + d3/256 + d4/4096 + e.  Each
// residual a - d is exact in binary32 (d is the nearest code to a, within a
// factor of two of it or zero), and times 16 stays exact.
KVQ_DEVI void p_pieces(float a, float b, uint32_t (&c)[kPPieces]) {
#pragma unroll
  for (int k = 0; k < kPPieces; ++k) {
    c[k] = f32x2_to_fp8x2<KVQ_FMT_E4M3>(a, b);
    if (k + 1 < kPPieces) {
      float da, db;
      dec_e4m3x2(c[k], da, db);
      a = (a - da) * 16.f;
      b = (b - db) * 16.f;
    }
  }
}

// Q of one segment into a Q^T tile (the B operand of S^T = K Q^T): threads
// 0 .. 16 G - 1, 16 per head, 8 dims each.  bf16 query: rows 3h + k hold the
// pieces of 2^a_h q_h (a_h into qexp[h]); FP8-domain query: row h holds
// enc(q_h / sQ_h).  raw: the thread's 8 bf16 values, loaded earlier.
template <int FMT, bool QF8>
KVQ_DEVI void write_q_tile(const DecodeParams& p, int gkv, const uint4& raw, uint32_t qaddr,
                           int32_t* qexp, int tid) {
  const int h = tid >> 4, sub = tid & 15;
  const bool active = h < p.G;  // inactive lanes still take part in the shuffles
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  float x[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = active ? bf16lo_to_f32(w[i]) : 0.f;
    x[2 * i + 1] = active ? bf16hi_to_f32(w[i]) : 0.f;
  }
  const uint32_t chunk_off = static_cast<uint32_t>((sub & 1) * 8);
  if (QF8) {
    if (!active) return;
    const float sq = __ldg(p.qs + (p.q_per_head ? gkv * p.G + h : 0));
    uint32_t c[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t lo = f32x2_to_fp8x2<FMT>(__fdiv_rn(x[4 * j], sq), __fdiv_rn(x[4 * j + 1], sq));
      const uint32_t hi =
          f32x2_to_fp8x2<FMT>(__fdiv_rn(x[4 * j + 2], sq), __fdiv_rn(x[4 * j + 3], sq));
      c[j] = lo | (hi << 16);
    }
    const int row = h;
    sts64(qaddr + row * 128 + ((((sub >> 1) ^ (row & 7))) << 4) + chunk_off, c[0], c[1]);
    return;
  }
  // per-head power of two: 2^a max|q| in [128, 256)
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
  int a = 0;
  if (amax > 0.f) {
    const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127;  // subnormal: -127
    a = 7 - e;
    a = a > 126 ? 126 : (a < -126 ? -126 : a);
  }
  if (!active) return;
  if (sub == 0) qexp[h] = a;
  const float sc = pow2i(a);
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = x[i] * sc;  // exact: a power of two, no overflow
#pragma unroll
  for (int k = 0; k < kQPieces; ++k) {
    uint32_t c[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t lo = f32x2_to_fp8x2<KVQ_FMT_E4M3>(y[4 * j], y[4 * j + 1]);
      const uint32_t hi = f32x2_to_fp8x2<KVQ_FMT_E4M3>(y[4 * j + 2], y[4 * j + 3]);
      c[j] = lo | (hi << 16);
      if (k + 1 < kQPieces) {
        float d0, d1, d2, d3;
        dec_e4m3x2(lo, d0, d1);
        dec_e4m3x2(hi, d2, d3);
        y[4 * j] = (y[4 * j] - d0) * 16.f;
        y[4 * j + 1] = (y[4 * j + 1] - d1) * 16.f;
        y[4 * j + 2] = (y[4 * j + 2] - d2) * 16.f;
        y[4 * j + 3] = (y[4 * j + 3] - d3) * 16.f;
      }
    }
    const int row = kQPieces * h + k;
    sts64(qaddr + row * 128 + ((((sub >> 1) ^ (row & 7))) << 4) + chunk_off, c[0], c[1]);
  }
}

// Raw bf16 query words of thread tid (head tid / 16, dims 8 (tid % 16) ..)
// for segment (b, gkv).
KVQ_DEVI uint4 load_q8(const DecodeParams& p, int b, int gkv, int tid) {
  const int h = tid >> 4, sub = tid & 15;
  if (h >= p.G) return make_uint4(0u, 0u, 0u, 0u);
  const int64_t qrow = static_cast<int64_t>(b) * p.Hq + gkv * p.G + h;
  if (!guard(b >= 0 && b < p.B && qrow < static_cast<int64_t>(p.B) * p.Hq, p.status, 12))
    return make_uint4(0u, 0u, 0u, 0u);
  return reinterpret_cast<const uint4*>(p.q + qrow * kDH)[sub];
}

// 128-thread reduction helpers of the softmax warps (named barrier kSoftBar).
KVQ_DEVI void soft_bar() { asm volatile("bar.sync %0, %1;" ::"n"(kSoftBar), "n"(kSoftThreads) : "memory"); }

KVQ_DEVI bool soft_bar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "n"(kSoftBar), "n"(kSoftThreads)
      : "memory");
  return r != 0;
}

// CLU: one cluster of p.clu CTAs per (sequence, KV head) segment, CTA k of it
// taking the k-th of p.clu equal parts of the segment's pages; the parts'
// states are merged in the leader CTA's shared memory (distributed shared
// memory, a cluster barrier) instead of through the global workspace.
template <int FMT, bool QF8, int GW, bool CLU>
__global__ void __launch_bounds__(kThreadsD, 1)
    decode_tc_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
  using Lo = DLay<GW>;
  constexpr int NS = Lo::NS, NO = Lo::NO;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lo::bars);
  // Stage s holds tile t = s (mod kNst): its K and V pages and its P^T
  // tile.  The P^T tile is free whenever the stage has landed again (its
  // previous reader, PV(t - kNst), completed before the stage was reloaded).
  uint64_t* full = bars;             // [kNst] tile landed (TMA bytes)
  uint64_t* empty = bars + kNst;     // [kNst] PV of the stage's tile done (commit)
  uint64_t* pfull = bars + 2 * kNst; // [kNst] P^T tile written (4 warp arrivals)
  uint64_t* sfull = bars + 3 * kNst; // [2] S^T buffer written (commit)
  uint64_t* sfree = sfull + 2;       // [2] S^T buffer read (4 warp arrivals)
  uint64_t* qfull = sfull + 4;       // [2] Q^T tile written (4 warp arrivals)
  uint64_t* fin = sfull + 6;         // every QK^T MMA done (commit)
  uint64_t* mcopy = sfull + 7;       // the bulk copy of a segment's pieces for its merge
  uint64_t* pvfin = sfull + 8;       // every PV MMA done (commit)
  // A parity wait for phase k is sound only while the barrier has completed
  // k or k + 1 phases: every waiter waits each barrier's phases in order, and
  // a barrier's next phase needs the waiter's own later progress.
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lo::misc);
  volatile uint32_t* st_np = misc;                 // [kNst] pages of the staged tile
  volatile uint32_t* st_bad = misc + kNst;         // [kNst] masked pages (bit i = page i)
  int32_t* issued = reinterpret_cast<int32_t*>(misc + 2 * kNst);  // [kNst] last tile issued
  volatile uint32_t* abort_flag = misc + 3 * kNst;
  volatile uint32_t* tmem_slot = misc + 3 * kNst + 1;
  volatile uint32_t* merge_s = misc + 3 * kNst + 2;
  int32_t* ub = reinterpret_cast<int32_t*>(misc + 3 * kNst + 3);    // [2] u0, u1
  int32_t* qexp = reinterpret_cast<int32_t*>(misc + 3 * kNst + 5);  // [2][8]
  volatile uint32_t* mcopy_s = misc + 3 * kNst + 21;                // merge copy issued
  float* red_m = reinterpret_cast<float*>(smem + Lo::red);          // [4][8]
  float* red_l = red_m + 32;                                        // [4][8]
  int32_t* warp_tot = reinterpret_cast<int32_t*>(red_l + 32);       // [8]
  int32_t* seq_off = reinterpret_cast<int32_t*>(smem + Lo::plan);   // [B+1]
  int32_t* len_s = seq_off + p.B + 1;                               // [B]
  int32_t* vseq_off = len_s + p.B;                                  // [B+1]
  float* sk_s = reinterpret_cast<float*>(vseq_off + p.B + 1);       // [Hkv]
  float* sv_s = sk_s + p.Hkv;                                       // [Hkv]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < kNst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&pfull[i], 4);
      issued[i] = -1;
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sfree[i], 4);
      mbar_init(&qfull[i], 4);
    }
    mbar_init(fin, 1);
    mbar_init(mcopy, 1);
    mbar_init(pvfin, 1);
    *abort_flag = 0u;
    *mcopy_s = 0u;
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  if (warp == 5) {
    tmem_alloc(const_cast<uint32_t*>(tmem_slot), Lo::kCols);
    tc_fence_before();
  }
  if (!p.early) {
    // The metadata this kernel reads first (lengths, scales, its share of the
    // block tables and of q) into L2 while the previous kernel drains: a
    // prefetch returns no data, so what that kernel still writes is read
    // after the wait as usual.
    if (warp == 4) {
      auto pf = [](const void* a) { asm volatile("prefetch.global.L2 [%0];" ::"l"(a)); };
      auto slice = [&](const void* base, int64_t bytes, int i) {
        const int64_t lines = (bytes + 127) >> 7;
        const int64_t l0 = lines * blockIdx.x / gridDim.x, l1 = lines * (blockIdx.x + 1) / gridDim.x;
        if (l0 + i < l1 && i < 8) pf(static_cast<const uint8_t*>(base) + ((l0 + i) << 7));
      };
      if (lane == 0) pf(p.seq_lens);
      if (lane == 1) pf(p.ks);
      if (lane == 2) pf(p.vs);
      if (lane == 3) pf(p.ws_cnt);
      if (lane >= 8 && lane < 16)
        slice(p.block_tables, static_cast<int64_t>(p.B) * p.max_blocks * 4, lane - 8);
      if (lane >= 16 && lane < 24) slice(p.q, static_cast<int64_t>(p.B) * p.Hq * kDH * 2, lane - 16);
    }
    pdl_wait();
    pdl_allow_next();
  }
  int64_t u0 = 0, u1 = 0;
  int Pe = 1;
  const int c = blockIdx.x;
  const uint32_t crank = CLU ? cluster_rank() : 0u;
  int seg_c = 0;  // the cluster's segment
  if (!CLU) {
    build_plan<true, kThreadsD>(p, seq_off, len_s, vseq_off, sk_s, sv_s, warp_tot);  // ends in __syncthreads
    const int64_t W = seq_off[p.B];
    Pe = static_cast<int>(W < p.P ? W : p.P);
  } else {  // the lengths and scales of the (few) sequences and heads
    for (int b = tid; b < p.B; b += kThreadsD) {
      const int raw = p.seq_lens[b];
      if ((raw < 0 || raw > p.max_blocks * kBS) && blockIdx.x == 0)
        flag_status(p.status, KVQ_DEV_BAD_SEQLEN);
      len_s[b] = (raw < 0 || raw > p.max_blocks * kBS) ? 0 : raw;
    }
    for (int h = tid; h < p.Hkv; h += kThreadsD) {
      sk_s[h] = p.ks[p.per_head ? h : 0];
      sv_s[h] = p.vs[p.per_head ? h : 0];
    }
    seg_c = static_cast<int>(blockIdx.x) / p.clu;
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const CostSplit cost_split(CLU ? 1 : vseq_off[p.B], Pe);
  if (!CLU) {
    if ((tid == 0 || tid == 32) && c < Pe)
      ub[tid >> 5] = pages_before(seq_off, vseq_off, p.B, p.Hkv, cost_split(c + (tid >> 5)));
    __syncthreads();
    u0 = c < Pe ? ub[0] : 0;
    u1 = c < Pe ? ub[1] : 0;
  }
  // The CTA's tiles, from its first one.
  auto first_tile = [&](TileIt& it) {
    if (!CLU) {
      it.start(seq_off, p.B, p.Hkv, u0, u1);
      return;
    }
    const int b = seg_c / p.Hkv, L = len_s[b];
    const int pages = L > 0 ? (L + kBS - 1) / kBS - first_page_of(p, L) : 0;
    const int k = static_cast<int>(crank);
    it.b = b;
    it.gkv = seg_c - b * p.Hkv;
    it.pages = pages;
    it.p0 = static_cast<int>(static_cast<int64_t>(pages) * k / p.clu);
    it.n = static_cast<int>(static_cast<int64_t>(pages) * (k + 1) / p.clu) - it.p0;
    it.u = 0;
    it.u1 = it.n;
    it.pp = 0;
    it.np = it.n < kTilePages ? it.n : kTilePages;
    it.piece = 0;
    it.t = 0;
    it.valid = it.n > 0;
  };

  auto fail = [&]() {
    if (!*abort_flag) {
      *abort_flag = 1u;
      flag_status(p.status, KVQ_DEV_WAIT_TIMEOUT);
    }
  };

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    // Lane i looks up page i % 8 of tile i / 8 of a group of 4 tiles; the
    // next group's ids are requested while this group's tiles are issued.
    struct Look {
      int row;    // cache row of the page (-1 masked out, -2 no page)
      bool lastp; // the page holds its sequence's newest token
    };
    auto look_issue = [&](TileIt g, int& col_blk, int& meta) {
      // meta: -2 no page; else (b << 1 | last) with the block id load in col_blk
      for (int k = 0; k < (lane >> 3) && g.valid; ++k) g.next(seq_off, p.B, p.Hkv);
      const int i = lane & 7;
      meta = -2;
      col_blk = -1;
      if (g.valid && i < g.np) {
        const int pg = g.p0 + g.pp + i;
        const int col = first_page_of(p, len_s[g.b]) + pg;
        const bool lastp = pg == g.pages - 1;
        if (guard(col >= 0 && col < p.max_blocks && g.gkv >= 0 && g.gkv < p.Hkv, p.status, 0))
          col_blk = p.block_tables[static_cast<int64_t>(g.b) * p.max_blocks + col];
        else
          col_blk = -1;
        meta = (g.gkv << 1) | (lastp ? 1 : 0);
      }
    };
    auto look_finish = [&](int col_blk, int meta) {
      Look l;
      l.lastp = meta >= 0 && (meta & 1);
      if (meta < 0) {
        l.row = -2;
        return l;
      }
      const int gkv = meta >> 1;
      bool bad = col_blk < 0 || col_blk >= p.num_blocks;
      if (bad) flag_status(p.status, KVQ_DEV_BAD_BLOCK);
      int32_t row = ((bad ? 0 : col_blk) * p.Hkv + gkv) * kBS;
      if (!bad && !guard(row >= 0 && row + kBS <= p.rows, p.status, 1)) bad = true;
      l.row = bad ? -1 : row;
      return l;
    };
    const uint64_t pol = l2_evict_first_policy();
    bool waited = !p.early;
    TileIt it;
    first_tile(it);
    TileIt grp = it;  // first tile of the next group to look up
    int nb_blk = -1, nb_meta = -2;
    if (grp.valid) look_issue(grp, nb_blk, nb_meta);
    Look cur{-2, false};
    for (; it.valid; it.next(seq_off, p.B, p.Hkv)) {
      const int t = it.t, s = t % kNst, q = t & 3;
      if (q == 0) cur = look_finish(nb_blk, nb_meta);  // the looked-up group
      const int my_row = __shfl_sync(kFull, cur.row, 8 * q + (lane & 7));
      const bool my_last = __shfl_sync(kFull, cur.lastp ? 1 : 0, 8 * q + (lane & 7)) != 0;
      const bool mine = (lane < 8) && lane < it.np;  // lane i issues page i of the tile
      if (!waited && __any_sync(kFull, mine && my_last)) {  // a newest-token page: wait first
        pdl_wait();
        waited = true;
      }
      bool ok = t < kNst ||
                wait_or_abort(&empty[s], static_cast<uint32_t>(((t / kNst) - 1) & 1), abort_flag);
      if (!__all_sync(kFull, ok) || *abort_flag) {
        if (lane == 0) fail();
        break;
      }
      const bool good = mine && my_row >= 0;
      const uint32_t badm = __ballot_sync(kFull, mine && my_row < 0) & 0xFFu;
      const uint32_t ngood = __popc(__ballot_sync(kFull, good));
      if (lane == 0) {
        st_np[s] = static_cast<uint32_t>(it.np);
        st_bad[s] = badm;
        issued[s] = t;
        if (ngood == 0)
          mbar_arrive(&full[s]);  // nothing to load: complete the phase by hand
        else
          mbar_arrive_expect_tx(&full[s], ngood * 2 * kPageB);
      }
      __syncwarp();
      if (good) {
        uint8_t* dst = smem + Lo::ring + static_cast<size_t>(s) * kStageB + lane * kPageB;
        tma_load_2d_hint(dst, &tmk, 0, my_row, &full[s], pol);
        tma_load_2d_hint(dst + kHalf, &tmv, 0, my_row, &full[s], pol);
      }
      if (q == 0) {  // request the next group's block ids
        for (int k = 0; k < 4 && grp.valid; ++k) grp.next(seq_off, p.B, p.Hkv);
        if (grp.valid) look_issue(grp, nb_blk, nb_meta);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ QK^T issuer
    // One lane issues S^T(t) = K_t Q^T as soon as tile t has landed and its
    // S buffer has been read.  (An MMA costs its issuing thread ~75 cycles,
    // so QK^T and PV have a thread each: neither waits behind the other.)
    if (lane == 0) {
      const uint32_t id_qk = idesc_f8(kTileTok, NS, tc_type(FMT), QF8 ? tc_type(FMT) : kTcE4M3,
                                      false, false);
      // descriptors of stage 0's K pages and of Q buffer 0; a 32-byte K step
      // adds 2 to the start address field, a stage kStageB / 16
      const uint64_t dk0 = sw128_desc(sbase + Lo::ring), dq0 = sw128_desc(sbase + Lo::qbuf);
      bool ok = true;
      TileIt it;
      first_tile(it);
      for (; it.valid && ok; it.next(seq_off, p.B, p.Hkv)) {
        const int t = it.t, s = t % kNst, sb = t & 1;
        if (it.first())
          ok = wait_or_abort(&qfull[it.piece & 1], static_cast<uint32_t>((it.piece >> 1) & 1),
                             abort_flag);
        if (ok && t >= 2)
          ok = wait_or_abort(&sfree[sb], static_cast<uint32_t>(((t >> 1) - 1) & 1), abort_flag);
        if (ok) ok = wait_or_abort(&full[s], static_cast<uint32_t>((t / kNst) & 1), abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dk = dk0 + static_cast<uint64_t>(s) * (kStageB >> 4);
        const uint64_t dq = dq0 + static_cast<uint64_t>(it.piece & 1) * (Lo::qBytes >> 4);
#pragma unroll
        for (int k = 0; k < kDH / 32; ++k) mma_f8_ss(tmem + sb * NS, dk + 2 * k, dq + 2 * k, id_qk, k > 0 ? 1u : 0u);
        mma_commit(&sfull[sb]);
      }
      if (!ok) fail();
      mma_commit(fin);  // completes when every MMA issued above has
      if (!mbar_wait(fin, 0u)) fail();
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------------------ PV issuer
    // One lane issues O^T += V_t^T P_t^T once the softmax has written P_t,
    // in tile order; its completion frees the stage (K, V and P^T tiles).
    if (lane == 0) {
      const uint32_t id_pv = idesc_f8(kDH, NO, tc_type(FMT), kTcE4M3, true, false);
      // V as the MN-major A operand: a 32-token K step is 4096 bytes (256 in
      // the address field); the P^T tile K-major like Q
      const uint64_t dv0 = sw128_desc(sbase + Lo::ring + kHalf, 16384, 1024);
      const uint64_t dp0 = sw128_desc(sbase + Lo::pbuf);
      bool ok = true;
      TileIt it;
      first_tile(it);
      for (; it.valid && ok; it.next(seq_off, p.B, p.Hkv)) {
        const int t = it.t, s = t % kNst;
        ok = wait_or_abort(&pfull[s], static_cast<uint32_t>((t / kNst) & 1), abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dv = dv0 + static_cast<uint64_t>(s) * (kStageB >> 4);
        const uint64_t dp = dp0 + static_cast<uint64_t>(s) * (Lo::pBytes >> 4);
#pragma unroll
        for (int k = 0; k < kTileTok / 32; ++k)
          mma_f8_ss(tmem + 2 * NS, dv + 256 * k, dp + 2 * k, id_pv, (k > 0 || !it.first()) ? 1u : 0u);
        mma_commit(&empty[s]);  // the stage (and its P^T tile) is free, O^T holds this tile
      }
      if (!ok) fail();
      mma_commit(pvfin);
      if (!mbar_wait(pvfin, 0u)) fail();
    }
    __syncwarp();
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int r = tid;  // token r of a tile = TMEM lane r; dim r of O^T
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    if (p.early) {  // q and every write wait for the previous kernel
      pdl_wait();
      pdl_allow_next();
    }
    // Sequences with nothing to attend to get a zero output row (CTAs share
    // them; in the cluster variant the leader's merge writes them).
    for (int b = blockIdx.x; !CLU && b < p.B; b += gridDim.x) {
      if (seq_off[b + 1] != seq_off[b]) continue;
      uint16_t* row = p.out + static_cast<int64_t>(b) * p.Hq * kDH;
      for (int i = r; i < p.Hq * kDH; i += kSoftThreads) row[i] = 0;
    }
    auto wait_w = [&](uint64_t* bar, uint32_t parity) {
      const bool w = __all_sync(kFull, wait_or_abort(bar, parity, abort_flag));
      if (!w && lane == 0) fail();
      return w;
    };
    bool ok = true;  // this warp's waits so far (the named barriers run regardless)
    TileIt it;
    first_tile(it);
    const bool no_tiles = !it.valid;
    // Q of the first piece now, the next one's raw words in flight
    TileIt nx = it;  // positioned at the next piece to get its Q
    uint4 qraw = make_uint4(0u, 0u, 0u, 0u);
    if (it.valid) {
      write_q_tile<FMT, QF8>(p, it.gkv, load_q8(p, it.b, it.gkv, r),
                             sbase + Lo::qbuf, qexp, r);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&qfull[0]);
      // advance nx to the second piece
      while (nx.valid && nx.piece == 0) nx.next(seq_off, p.B, p.Hkv);
      if (nx.valid) qraw = load_q8(p, nx.b, nx.gkv, r);
    }
    constexpr float kThr = kRescaleThreshold;
    float m[GW], l[GW], cq[GW];
    float sv = 1.f;
    int L = 0, lo = 0, fp = 0;
    for (; it.valid; it.next(seq_off, p.B, p.Hkv)) {
      const int t = it.t, s = t % kNst, sb = t & 1;
      if (it.first()) {
        soft_bar();  // qexp of this piece is written (by the Q writers)
        L = len_s[it.b];
        lo = window_lo(p, L);
        fp = lo / kBS;
        sv = sv_s[it.gkv];
        const float lk = sk_s[it.gkv] * p.logit_scale;
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          m[h] = -INFINITY;
          l[h] = 0.f;
          if (QF8)
            cq[h] = h < p.G ? lk * __ldg(p.qs + (p.q_per_head ? it.gkv * p.G + h : 0)) : 0.f;
          else
            cq[h] = h < p.G ? lk * pow2i(-qexp[(it.piece & 1) * 8 + h]) : 0.f;
        }
      }
      // ---- S^T row of token r
      if (ok) ok = wait_w(&full[s], static_cast<uint32_t>((t / kNst) & 1));  // stage flags
      if (ok) ok = wait_w(&sfull[sb], static_cast<uint32_t>((t >> 1) & 1));
      uint32_t sr[NS];
      if (ok) {
        tc_fence_after();
        __syncwarp();
        uint32_t a[16];
        tmem_ld16(tmem + lane_base + sb * NS, a);
#pragma unroll
        for (int i = 0; i < 16; ++i) sr[i] = a[i];
        if (NS > 16) {
          uint32_t b2[16];
          tmem_ld16(tmem + lane_base + sb * NS + 16, b2);
#pragma unroll
          for (int i = 0; i < 16 && 16 + i < NS; ++i) sr[16 + i] = b2[i];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfree[sb]);
      } else {
#pragma unroll
        for (int i = 0; i < NS; ++i) sr[i] = 0u;
      }
      const int pg = r >> 4;  // page of token r in the tile
      const uint32_t np = ok ? st_np[s] : 0u, bad = ok ? st_bad[s] : 0xFFu;
      const int pos = (fp + it.p0 + it.pp + pg) * kBS + (r & 15);
      const bool valid = pg < static_cast<int>(np) && !((bad >> pg) & 1u) && pos >= lo && pos < L;
      float x[GW];
#pragma unroll
      for (int h = 0; h < GW; ++h) {
        float v;
        if (QF8)
          v = __uint_as_float(sr[h]);
        else
          v = fmaf(__uint_as_float(sr[3 * h + 2]), 1.f / 256.f,
                   fmaf(__uint_as_float(sr[3 * h + 1]), 1.f / 16.f, __uint_as_float(sr[3 * h])));
        x[h] = (valid && h < p.G) ? v * cq[h] : -INFINITY;
      }
      // ---- running maxima: raised only when a tile exceeds them by 2^8
      bool need = false;
#pragma unroll
      for (int h = 0; h < GW; ++h) need |= x[h] > m[h] + kThr;
      if (soft_bar_or(need)) {
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          float v = x[h];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, off));
          if (lane == 0) red_m[warp * 8 + h] = v;
        }
        soft_bar();
        float alpha[GW];
        bool any_scale = false;
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          const float tm = fmaxf(fmaxf(red_m[h], red_m[8 + h]), fmaxf(red_m[16 + h], red_m[24 + h]));
          const float nm = tm > m[h] + kThr ? tm : m[h];
          alpha[h] = (m[h] == -INFINITY) ? 0.f : fast_exp2(m[h] - nm);
          any_scale |= nm != m[h] && m[h] != -INFINITY;  // O^T holds tiles of this piece
          m[h] = nm;
          l[h] *= alpha[h];  // m = -inf before: no token yet, l = 0
        }
        // O^T already holds earlier tiles of this piece: rescale its columns
        // once the last PV issued (tile t - 1) is done
        if (any_scale) {
          if (ok) ok = wait_w(&empty[(t - 1) % kNst], static_cast<uint32_t>(((t - 1) / kNst) & 1));
          if (ok) {
            tc_fence_after();
            const uint32_t ta = tmem + lane_base + 2 * NS;
#pragma unroll
            for (int c0 = 0; c0 < NO; c0 += 16) {
              uint32_t o[16];
              __syncwarp();
              tmem_ld16(ta + c0, o);
#pragma unroll
              for (int i = 0; i < 16; ++i)
                o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha[(c0 + i) / kPPieces]);
              tmem_st16(ta + c0, o);
            }
          }
        }
        soft_bar();  // red_m read by every thread before its next write
      }
      // ---- probabilities and their pieces
      float pr[GW];
#pragma unroll
      for (int h = 0; h < GW; ++h) {
        pr[h] = (x[h] == -INFINITY || m[h] == -INFINITY) ? 0.f : fast_exp2(x[h] - m[h]);
        l[h] += pr[h];
      }
      uint32_t pc[(GW + 1) / 2][kPPieces];
#pragma unroll
      for (int j = 0; j < (GW + 1) / 2; ++j)
        p_pieces(pr[2 * j], (2 * j + 1 < GW) ? pr[2 * j + 1] : 0.f, pc[j]);
      if (ok) {  // the stage's P^T tile (free: the stage has landed again)
        const uint32_t pt = sbase + Lo::pbuf + s * Lo::pBytes;
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          if (h < p.G) {
#pragma unroll
            for (int k = 0; k < kPPieces; ++k) {
              const int row = h * kPPieces + k;
              sts8(pt + sw_off(row, r), (pc[h >> 1][k] >> ((h & 1) * 8)) & 0xFFu);
            }
          }
        }
        if (!valid) {  // a masked token's V row may hold anything (p = 0 would not clear a NaN)
          const uint32_t vr = sbase + Lo::ring + s * kStageB + kHalf + pg * kPageB + (r & 15) * 128;
#pragma unroll
          for (int i = 0; i < 8; ++i) sts128(vr + 16 * i, 0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();  // P^T bytes and zeroed V rows -> the tensor core
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[s]);
      // ---- the next piece's Q once this piece has started
      if (it.first() && nx.valid) {
        write_q_tile<FMT, QF8>(p, nx.gkv, qraw, sbase + Lo::qbuf + (nx.piece & 1) * Lo::qBytes,
                               qexp + (nx.piece & 1) * 8, r);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&qfull[nx.piece & 1]);
        const int cur = nx.piece;
        while (nx.valid && nx.piece == cur) nx.next(seq_off, p.B, p.Hkv);
        if (nx.valid) qraw = load_q8(p, nx.b, nx.gkv, r);
      }
      if (!it.last()) continue;
      // ---- piece end: O^T row r (dim r) once PV(t) is done
      if (ok) ok = wait_w(&empty[s], static_cast<uint32_t>((t / kNst) & 1));
      float o[GW];
#pragma unroll
      for (int h = 0; h < GW; ++h) o[h] = 0.f;
      if (ok) {
        tc_fence_after();
        const uint32_t ta = tmem + lane_base + 2 * NS;
#pragma unroll
        for (int c0 = 0; c0 < NO; c0 += 16) {
          uint32_t v[16];
          __syncwarp();
          tmem_ld16(ta + c0, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = c0 + i, h = col / kPPieces, k = col % kPPieces;
            const float f = k == 0 ? 1.f : (k == 1 ? 1.f / 16.f : (k == 2 ? 1.f / 256.f : 1.f / 4096.f));
            o[h] = fmaf(__uint_as_float(v[i]), f, o[h]);
          }
        }
        tc_fence_before();
      }
      // denominators: sum of the 128 threads' partial sums
#pragma unroll
      for (int h = 0; h < GW; ++h) {
        float v = l[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
        if (lane == 0) red_l[warp * 8 + h] = v;
      }
      soft_bar();
      float Ls[GW];
#pragma unroll
      for (int h = 0; h < GW; ++h) Ls[h] = (red_l[h] + red_l[8 + h]) + (red_l[16 + h] + red_l[24 + h]);
      if (CLU) {  // this part's state into the leader's merge area
        const uint32_t mg = map_rank(sbase + static_cast<uint32_t>(Lo::plan_end(p.B, p.Hkv)), 0u);
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          if (h < p.G)
            st_cluster_f32(mg + kCluMax * GW * 8 + ((crank * GW + h) * kDH + r) * 4, o[h]);
          if (h == r && h < p.G) st_cluster_v2(mg + (crank * GW + h) * 8, m[h], Ls[h]);
        }
        soft_bar();  // red_l read by every thread before its next write
        continue;
      }
      const bool single = it.p0 == 0 && it.n == it.pages;
      const int64_t sigma = static_cast<int64_t>(it.b) * p.Hkv + it.gkv;
      if (single) {
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          if (h < p.G) {
            const float f = Ls[h] > 0.f ? sv / Ls[h] : 0.f;
            const int64_t oi = (static_cast<int64_t>(it.b) * p.Hq + it.gkv * p.G + h) * kDH + r;
            if (guard(oi >= 0 && oi < static_cast<int64_t>(p.B) * p.Hq * kDH, p.status, 3))
              p.out[oi] = static_cast<uint16_t>(f32x2_to_bf16x2(o[h] * f, 0.f) & 0xFFFFu);
          }
        }
        soft_bar();  // red_l read by every thread before its next write
        continue;
      }
      // ---- a split segment: publish this piece; the CTA completing the
      // segment merges its pieces
      const int64_t slot_idx = static_cast<int64_t>(blockIdx.x) + sigma;
      const bool slot_ok = guard(slot_idx >= 0 && slot_idx < p.n_slots, p.status, 4);
      if (slot_ok) {
#pragma unroll
        for (int h = 0; h < GW; ++h)
          if (h < p.G) p.ws_o[(slot_idx * p.G + h) * kDH + r] = o[h];
        if (r < p.G) {
          float mm = -INFINITY, ll = 0.f;
#pragma unroll
          for (int h = 0; h < GW; ++h)
            if (h == r) {
              mm = m[h];
              ll = Ls[h];
            }
          *reinterpret_cast<float2*>(p.ws_ml + (slot_idx * p.G + r) * 2) = make_float2(mm, ll);
        }
      }
      const int v_first = vseq_off[it.b] + it.gkv * (it.pages + kPieceCost) + kPieceCost;
      const int seg_lo = cost_split.cta_of(v_first);
      const int seg_n = cost_split.cta_of(v_first + it.pages - 1) - seg_lo + 1;
      soft_bar();  // every store of the piece before the arrival; red_l reads done
      const uint32_t obytes = static_cast<uint32_t>(seg_n) * p.G * kDH * 4;
      const uint32_t mlbytes = static_cast<uint32_t>(seg_n) * p.G * 8;
      if (r == 0) {
        // 0: not the last piece; 1: merge from global memory; 2: merge after
        // the CTA's last piece, its ring idle: the pieces' o vectors come in
        // with one bulk copy.  Decided once here, so that every thread takes
        // the same branch.
        uint32_t last = 0u;
        if (!*abort_flag && slot_ok) {
          const uint32_t prev = atom_add_acq_rel_gpu(p.ws_cnt + sigma, 1u);
          last = prev + 1 == static_cast<uint32_t>(seg_n) ? 1u : 0u;
        }
        if (last && it.u + it.n == it.u1 && !*abort_flag &&
            obytes + mlbytes + static_cast<uint32_t>(seg_n + 1) * GW * 4 <=
                static_cast<uint32_t>(kNst) * kStageB)
          last = 2u;
        *merge_s = last;
      }
      soft_bar();
      if (*merge_s) {
        // M = max m_c, w_c = 2^(m_c - M), O = sV sum w_c o_c / sum w_c l_c,
        // one running maximum per head (thread r: dim r of every head)
        const int64_t base = static_cast<int64_t>(seg_lo) + sigma;
        const bool mok = guard(seg_lo >= 0 && seg_n <= p.P && base + seg_n <= p.n_slots,
                               p.status, 5);
        float M[GW], acc[GW], Lt[GW];
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          M[h] = -INFINITY;
          acc[h] = 0.f;
          Lt[h] = 0.f;
        }
        // after the CTA's last piece the ring is idle: the pieces' states come
        // in with one bulk copy (o) and one load per thread (m, l)
        const bool staged = *merge_s == 2u && mok;
        if (staged) {
          float* so = reinterpret_cast<float*>(smem + Lo::ring);
          float2* sml = reinterpret_cast<float2*>(smem + Lo::ring + obytes);
          if (r == 0) {
            *mcopy_s = 1u;
            mbar_arrive_expect_tx(mcopy, obytes);
            fence_proxy_async_global();  // the pieces were acquired through the counter
            const uint8_t* src = reinterpret_cast<const uint8_t*>(p.ws_o + base * p.G * kDH);
            for (uint32_t off = 0; off < obytes; off += 16384)
              bulk_load(reinterpret_cast<uint8_t*>(so) + off, src + off,
                        obytes - off < 16384 ? obytes - off : 16384, mcopy);
          }
          const int nml = seg_n * p.G;
          // shared memory after the o vectors: (m, l) [seg_n][G], then the
          // weights [seg_n][GW] (a piece's heads contiguous), then l [GW]
          float* sw = reinterpret_cast<float*>(sml + nml);
          float* sL = sw + seg_n * GW;
          for (int i = r; i < nml; i += kSoftThreads)
            sml[i] = __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + base * p.G + i);
          soft_bar();  // (m, l) of every piece in shared memory
          // warp h < G: the head's maximum, weights and denominator over the pieces
          for (int h = warp; h < p.G; h += kSoftThreads / 32) {
            float mx = -INFINITY;
            for (int c2 = lane; c2 < seg_n; c2 += 32) mx = fmaxf(mx, sml[c2 * p.G + h].x);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
            float lsum = 0.f;
            for (int c2 = lane; c2 < seg_n; c2 += 32) {
              const float2 x = sml[c2 * p.G + h];
              const float w = x.x == -INFINITY ? 0.f : fast_exp2(x.x - mx);
              sw[c2 * GW + h] = w;
              lsum = fmaf(w, x.y, lsum);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(kFull, lsum, off);
            if (lane == 0) sL[h] = lsum;
          }
          soft_bar();
          const bool cok = __all_sync(kFull, mbar_wait(mcopy, 0u));
          if (!cok && lane == 0) fail();
          if (cok) {
            float a2[2][GW];
#pragma unroll
            for (int h = 0; h < GW; ++h) a2[0][h] = a2[1][h] = 0.f;
            int c2 = 0;
            for (; c2 + 1 < seg_n; c2 += 2) {
#pragma unroll
              for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int h = 0; h < GW; ++h)
                  if (h < p.G)
                    a2[j][h] = fmaf(sw[(c2 + j) * GW + h], so[((c2 + j) * p.G + h) * kDH + r], a2[j][h]);
            }
            if (c2 < seg_n) {
#pragma unroll
              for (int h = 0; h < GW; ++h)
                if (h < p.G) a2[0][h] = fmaf(sw[c2 * GW + h], so[(c2 * p.G + h) * kDH + r], a2[0][h]);
            }
#pragma unroll
            for (int h = 0; h < GW; ++h) {
              acc[h] = a2[0][h] + a2[1][h];
              Lt[h] = h < p.G ? sL[h] : 0.f;
            }
          }
        } else {
          constexpr int CH = GW <= 4 ? 4 : 2;  // pieces loaded together
          for (int c0 = 0; mok && c0 < seg_n; c0 += CH) {
            float2 mlv[CH][GW];
            float ov[CH][GW];
#pragma unroll
            for (int j = 0; j < CH; ++j)
#pragma unroll
              for (int h = 0; h < GW; ++h) {
                const bool in = c0 + j < seg_n && h < p.G;
                const int64_t sl = base + c0 + j;
                mlv[j][h] = in ? __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + sl * p.G + h)
                               : make_float2(-INFINITY, 0.f);
                ov[j][h] = in ? __ldcg(p.ws_o + (sl * p.G + h) * kDH + r) : 0.f;
              }
#pragma unroll
            for (int j = 0; j < CH; ++j)
#pragma unroll
              for (int h = 0; h < GW; ++h) {
                const float mc = mlv[j][h].x;
                if (mc == -INFINITY) continue;
                if (mc > M[h]) {
                  const float sc = M[h] == -INFINITY ? 0.f : fast_exp2(M[h] - mc);
                  acc[h] *= sc;
                  Lt[h] *= sc;
                  M[h] = mc;
                }
                const float w = fast_exp2(mc - M[h]);
                acc[h] = fmaf(w, ov[j][h], acc[h]);
                Lt[h] = fmaf(w, mlv[j][h].y, Lt[h]);
              }
          }
        }
        if (mok) {
#pragma unroll
          for (int h = 0; h < GW; ++h) {
            if (h < p.G) {
              const float f = Lt[h] > 0.f ? sv / Lt[h] : 0.f;
              const int64_t oi = (static_cast<int64_t>(it.b) * p.Hq + it.gkv * p.G + h) * kDH + r;
              if (guard(oi >= 0 && oi < static_cast<int64_t>(p.B) * p.Hq * kDH, p.status, 3))
                p.out[oi] = static_cast<uint16_t>(f32x2_to_bf16x2(acc[h] * f, 0.f) & 0xFFFFu);
            }
          }
        }
        if (r == 0) p.ws_cnt[sigma] = 0u;
      }
      soft_bar();  // merge_s read by every thread before its next write
    }
    if (CLU && no_tiles) {  // an empty part: m = -inf, l = 0, o = 0
      const uint32_t mg = map_rank(sbase + static_cast<uint32_t>(Lo::plan_end(p.B, p.Hkv)), 0u);
      for (int h = 0; h < p.G; ++h) st_cluster_f32(mg + kCluMax * GW * 8 + ((crank * GW + h) * kDH + r) * 4, 0.f);
      if (r < p.G) st_cluster_v2(mg + (crank * GW + r) * 8, -INFINITY, 0.f);
    }
    if (!ok) fail();
  }

  if (CLU) {
    // Every thread of every CTA arrives (release: this CTA's parts are in
    // the leader's shared memory); the leader waits for all of them and
    // merges the parts: M = max m_k, w_k = 2^(m_k - M),
    // O = sV sum w_k o_k / sum w_k l_k, thread r for dim r of every head.
    cluster_arrive_release();
    if (crank == 0) {
      cluster_wait_acquire();
      if (warp < 4) {
        const int r = tid;  // dim r
        const float2* ml = reinterpret_cast<const float2*>(smem + Lo::plan_end(p.B, p.Hkv));
        const float* mo = reinterpret_cast<const float*>(smem + Lo::plan_end(p.B, p.Hkv) + kCluMax * GW * 8);
        const int b = seg_c / p.Hkv, g = seg_c - b * p.Hkv;
        const float sv = sv_s[g];
        const int nk = p.clu;
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          if (h >= p.G) continue;
          float M = -INFINITY;
          for (int k = 0; k < nk; ++k) M = fmaxf(M, ml[k * GW + h].x);
          float acc0 = 0.f, acc1 = 0.f, l0 = 0.f, l1 = 0.f;
          int k = 0;
          for (; k + 1 < nk; k += 2) {
            const float2 x0 = ml[k * GW + h], x1 = ml[(k + 1) * GW + h];
            const float w0 = x0.x == -INFINITY ? 0.f : fast_exp2(x0.x - M);
            const float w1 = x1.x == -INFINITY ? 0.f : fast_exp2(x1.x - M);
            acc0 = fmaf(w0, mo[(k * GW + h) * kDH + r], acc0);
            acc1 = fmaf(w1, mo[((k + 1) * GW + h) * kDH + r], acc1);
            l0 = fmaf(w0, x0.y, l0);
            l1 = fmaf(w1, x1.y, l1);
          }
          if (k < nk) {
            const float2 x0 = ml[k * GW + h];
            const float w0 = x0.x == -INFINITY ? 0.f : fast_exp2(x0.x - M);
            acc0 = fmaf(w0, mo[(k * GW + h) * kDH + r], acc0);
            l0 = fmaf(w0, x0.y, l0);
          }
          const float Lt = l0 + l1;
          const float f = Lt > 0.f ? sv / Lt : 0.f;
          const int64_t oi = (static_cast<int64_t>(b) * p.Hq + g * p.G + h) * kDH + r;
          if (guard(oi >= 0 && oi < static_cast<int64_t>(p.B) * p.Hq * kDH, p.status, 3))
            p.out[oi] = static_cast<uint16_t>(f32x2_to_bf16x2((acc0 + acc1) * f, 0.f) & 0xFFFFu);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // After an abort: wait (bounded) for the copies still in flight (the MMA
  // lane waited for its own), then free the tensor memory.
  if (*abort_flag && tid == 0) {
    for (int s = 0; s < kNst; ++s)
      if (issued[s] >= 0) mbar_wait(&full[s], static_cast<uint32_t>((issued[s] / kNst) & 1));
    if (*mcopy_s) mbar_wait(mcopy, 0u);
  }
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, Lo::kCols);
  }
}

// --------------------------------------------------------------------------
// Launch
// --------------------------------------------------------------------------

// Dynamic shared memory of a launch: the ring, the Q / P tiles, the
// barriers and the plan of B sequences over Hkv KV heads (and, in the cluster
// variant, the leader's merge area).
inline size_t smem_bytes_tc(int G, int B, int Hkv, bool clu = false) {
  if (clu) return G <= 4 ? DLay<4>::total_clu(B, Hkv) : DLay<8>::total_clu(B, Hkv);
  return G <= 4 ? DLay<4>::total(B, Hkv) : DLay<8>::total(B, Hkv);
}

template <int FMT, bool QF8, int GW, bool CLU>
static bool configure_tc(size_t maxsmem) {
  auto k = decode_tc_kernel<FMT, QF8, GW, CLU>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(maxsmem)) !=
          cudaSuccess ||
      cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return false;
  if (CLU && cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return false;
  return true;
}

// The opt-in limit of dynamic shared memory per block on the current device.
inline size_t smem_optin() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return 0;
  return static_cast<size_t>(v);
}

// Largest batch of the cluster variant: its plan arrays stay small.
constexpr int kCluMaxSeqs = 64;

template <int FMT>
static bool configure_all_tc() {
  const size_t cap = smem_optin();
  auto lim = [cap](size_t need) { return need < cap ? need : cap; };
  const size_t m4 = lim(DLay<4>::total(kMaxSeqs, kMaxKvHeads));
  const size_t m8 = lim(DLay<8>::total(kMaxSeqs, kMaxKvHeads));
  const size_t c4 = lim(DLay<4>::total_clu(kCluMaxSeqs, kMaxKvHeads));
  const size_t c8 = lim(DLay<8>::total_clu(kCluMaxSeqs, kMaxKvHeads));
  return configure_tc<FMT, false, 4, false>(m4) && configure_tc<FMT, true, 4, false>(m4) &&
         configure_tc<FMT, false, 8, false>(m8) && configure_tc<FMT, true, 8, false>(m8) &&
         configure_tc<FMT, false, 4, true>(c4) && configure_tc<FMT, true, 4, true>(c4) &&
         configure_tc<FMT, false, 8, true>(c8) && configure_tc<FMT, true, 8, true>(c8);
}

template <typename K>
static cudaError_t launch_tc_kernel(K kernel, int grid, int clu, size_t smem, cudaStream_t s,
                                    const DecodeParams& p, const CUtensorMap& tk,
                                    const CUtensorMap& tv) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreadsD);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (clu > 0) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(clu);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, p, tk, tv);
}

template <int FMT>
static bool ensure_configured() {
  static DeviceOnce once;  // once per device, again after a failure
  return once.run(current_device(), [] { return configure_all_tc<FMT>(); });
}

// Clusters of `clu` CTAs (8 <= clu <= 16, one CTA per SM) of the group-size
// variant `gw` (4 or 8) that can be resident at once, with the largest
// cluster-variant batch's shared memory; queried once per device.  (The SMs
// of a GPU are grouped unevenly: on GB300 seven clusters of 16 fit at once,
// eight of 12.)
template <int FMT>
static int max_active_clusters(int clu, int gw) {
  static DeviceOnce once;  // queried until a query succeeds
  static int n[64][2][kCluMax + 1];
  const int dev = current_device();
  if (dev < 0 || dev >= 64 || clu < 1 || clu > kCluMax) return 0;
  const bool queried = once.run(dev, [dev] {
    const bool ok = ensure_configured<FMT>();
    for (int gi = 0; gi < 2; ++gi)
      for (int c = 0; c <= kCluMax; ++c) {
        n[dev][gi][c] = 0;
        const size_t smem = smem_bytes_tc(gi ? 8 : 4, kCluMaxSeqs, kMaxKvHeads, true);
        if (!ok || c < 8 || smem > smem_optin()) continue;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c);
        cfg.blockDim = dim3(kThreadsD);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(c);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int v = 0;
        const cudaError_t e =
            gi ? cudaOccupancyMaxActiveClusters(&v, decode_tc_kernel<FMT, false, 8, true>, &cfg)
               : cudaOccupancyMaxActiveClusters(&v, decode_tc_kernel<FMT, false, 4, true>, &cfg);
        if (e != cudaSuccess) {
          cudaGetLastError();
          v = 0;
        }
        n[dev][gi][c] = v;
      }
    return ok;
  });
  return queried ? n[dev][gw > 4 ? 1 : 0][clu] : 0;
}

// The cluster size of the per-segment variant for a batch of B sequences
// over Hkv KV heads, or 0 (the split variant): the largest size from 16
// down to 8 whose clusters, one per segment, all fit on the GPU at once,
// provided each CTA gets at least two tiles of a full-length segment.
template <int FMT>
int choose_clu(int G, int B, int Hkv, int max_blocks) {
  if (B > kCluMaxSeqs || Hkv > kMaxKvHeads) return 0;
  if (smem_bytes_tc(G, B, Hkv, true) > smem_optin()) return 0;
  const int segs = B * Hkv;
  for (int clu = kCluMax; clu >= 8; --clu) {
    if (max_blocks < clu * 2 * kTilePages) continue;
    if (max_active_clusters<FMT>(clu, G) >= segs) return clu;
  }
  return 0;
}

template <int FMT>
int launch_tc(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  if (!ensure_configured<FMT>()) return KVQ_ERR_CUDA;
  const bool clu = p.clu > 0;
  const size_t smem = smem_bytes_tc(p.G, p.B, p.Hkv, clu);
  if (smem > smem_optin()) return KVQ_ERR_UNSUPPORTED;
  const int grid = clu ? p.B * p.Hkv * p.clu : p.P;
  const bool qf8 = p.qs != nullptr;
  cudaError_t e;
  if (p.G <= 4) {
    if (clu)
      e = qf8 ? launch_tc_kernel(decode_tc_kernel<FMT, true, 4, true>, grid, p.clu, smem, s, p, tk, tv)
              : launch_tc_kernel(decode_tc_kernel<FMT, false, 4, true>, grid, p.clu, smem, s, p, tk, tv);
    else
      e = qf8 ? launch_tc_kernel(decode_tc_kernel<FMT, true, 4, false>, grid, 0, smem, s, p, tk, tv)
              : launch_tc_kernel(decode_tc_kernel<FMT, false, 4, false>, grid, 0, smem, s, p, tk, tv);
  } else {
    if (clu)
      e = qf8 ? launch_tc_kernel(decode_tc_kernel<FMT, true, 8, true>, grid, p.clu, smem, s, p, tk, tv)
              : launch_tc_kernel(decode_tc_kernel<FMT, false, 8, true>, grid, p.clu, smem, s, p, tk, tv);
    else
      e = qf8 ? launch_tc_kernel(decode_tc_kernel<FMT, true, 8, false>, grid, 0, smem, s, p, tk, tv)
              : launch_tc_kernel(decode_tc_kernel<FMT, false, 8, false>, grid, 0, smem, s, p, tk, tv);
  }
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace dtc
}  // namespace kvq
