// kvq_decode_blk.cuh -- paged GQA decode attention over the FP8 caches on the
// 5th-generation tensor cores, one cache block of eight KV heads per tile.
// Head size 128, four query heads per KV head, per-tensor or per-KV-head
// scales, the bf16 query or the FP8-domain query.
//
// "10.4 KV Cache quantization: INT8, KIVI 2-bit, FP8 KV", section 10.4.2:
// P = softmax(Q K^T / sqrt(dh) + mask), O = P V^, on the efficient path that
// reads the compressed KV once and feeds QK, PV and an online softmax
// directly; section 10.4.5: K^ = cast_float(K_fp8) * sK.  sK goes into the
// logit scale and sV onto the normalised output, so the MMAs work on the
// cache's codes as they arrive.
//
// Why a whole block per tile.  In the cache layout [block][KV head][16][128]
// the 16 tokens of eight consecutive KV heads are one contiguous 16 KB run
// (128 rows of 128 bytes).  One TMA box of 128 rows moves it: copies of
// 16 KB stream at the HBM rate from every SM, where 2 KB page copies stall on
// the per-SM copy rate well below it.  The tile's MMAs are block diagonal:
//   S^T = K Q^T     M = 128 rows (head j, token t: row 16 j + t), N = the
//                   query pieces of all 32 query heads, K = 128 dims; row
//                   16 j + t only uses the columns of head j's four queries.
//   O^T += V^T P^T  M = 128 dims (V as the MN-major A operand: the page
//                   layout itself), N = the probability pieces of the 32
//                   heads, K = 128 rows; P^T is zero outside the diagonal
//                   blocks (head j's probabilities sit only in rows 16 j ..
//                   16 j + 15), so every query head sums its own KV head.
// The tensor core does 8x the useful multiply-adds; it has them to spare,
// the bytes are what bounds a decode.
//
// Roles (224 threads, one CTA per SM, persistent over the CTA's units):
//   warp 4 (producer): block ids of 32 tiles at once (one per lane, looked up
//     32 tiles ahead), one K and one V box per tile into a ring of 4 stages.
//   warp 5: allocates the tensor memory; one lane issues the QK^T MMAs.
//   warp 6: one lane issues the PV MMAs; their completion frees the stage.
//   warps 0-3 (softmax; thread 32 w + l = TMEM lane = tile row 16 j + t with
//     j = 2 w + l / 16, t = l % 16): the logits of token t for head j's four
//     queries, the masks, an online softmax in the log2 domain with one
//     running maximum per query head (the 16 lanes of a half warp hold a KV
//     head's tokens; lazily raised, only when a tile exceeds it by 2^8), the
//     probability pieces into the P^T tile; at a piece's end thread d reads
//     row d of O^T (dim d of the 32 heads).
// Precision as in the per-head tensor-core kernel: the bf16 query enters as
// three E4M3 pieces of a per-head power-of-two scaling, the probabilities
// p <= 2^8 as four E4M3 pieces p1 + p2/16 + p3/256 + p4/4096 summed in fp32.
//
// Work split: a unit is one block of one group of eight KV heads of one
// sequence (a segment is a (sequence, head group)); the CTAs take
// cost-balanced ranges of units.  A piece that covers its whole segment is
// written out directly; the pieces of a split segment publish (m, l, o) per
// query head and are merged one of two ways:
//   LAST (batches): the CTA that completes a segment merges its pieces after
//     its own last tile, the pieces' o vectors staged into its idle ring.
//   GRID (few long segments, e.g. one sequence): every CTA publishes, all
//     CTAs meet at one bounded grid barrier (the grid is one CTA per SM, so
//     all of it is resident), then each CTA merges a slice of the outputs
//     (one query head x 32 dims) over all the pieces, seven warps reading
//     the pieces in parallel.  The last CTA to leave the barrier resets its
//     two counters, so the workspace stays zeroed between calls.
// Every wait is bounded; a timeout sets KVQ_DEV_WAIT_TIMEOUT, the roles stop
// at the same named barriers, and the CTA waits (bounded) for its copies and
// MMAs in flight before it frees the tensor memory.
#pragma once

#include "kvq_decode_tc.cuh"

namespace kvq {
namespace dtb {

using namespace tc;
using dtc::dec_e4m3x2;
using dtc::p_pieces;
using dtc::pow2i;
using dtc::soft_bar;
using dtc::soft_bar_or;
using dtc::sw_off;

constexpr int kDH = 128;
constexpr int kHT = kMaxHT;              // KV heads of one tile
constexpr int kRows = kHT * kBS;         // 128 tile rows
constexpr int kHalf = kRows * kDH;       // 16 KB: K (or V) of one tile
constexpr int kStageB = 2 * kHalf;       // K and V of one tile
constexpr int kThreadsB = 256;
constexpr int kSoftThreads = 128;
#ifndef KVQ_BLK_NK
#define KVQ_BLK_NK 4
#endif
#ifndef KVQ_BLK_NV
#define KVQ_BLK_NV 6
#endif
#ifndef KVQ_BLK_NP
#define KVQ_BLK_NP 2
#endif
// Ring stages of K and of V, and P^T tiles.  A V stage is held from its copy
// until PV of its tile is done (the copy's latency plus the whole QK^T ->
// softmax -> PV pipeline), a K stage only until QK^T is done: V gets more.
constexpr int kNk = KVQ_BLK_NK;
constexpr int kNv = KVQ_BLK_NV;
constexpr int kNp = KVQ_BLK_NP;          // tile t uses P^T tile t % kNp
constexpr int kFlags = 16;               // tile-validity ring the K producer fills
constexpr int kGQ = 4;                   // query heads per KV head
constexpr int kHeads = kHT * kGQ;        // 32 query heads of a tile
constexpr int kQP = 3, kPP = 4;          // query and probability pieces
constexpr int kBlkPieceCost = 2;         // fixed cost of a piece, in tiles
constexpr int kMergeWarps = kThreadsB / 32;
constexpr int kMergeBatch = 24;          // pieces a warp loads together in the grid merge
constexpr uint32_t kOS = 256;            // TMEM column of O^T (S^T buffers at 0 and 128)

struct BMisc {
  int32_t kiss[kNk];       // last tile whose K was copied into the stage (-1: none)
  int32_t viss[kNv];       // and V
  uint32_t vmask[kNp][4];  // valid rows of the tile of P^T buffer t % kNp (bit r % 32 of word r / 32)
  uint32_t tflag[kFlags];  // tile t: (t << 1) | (its block id is in range), at t % 16
  uint32_t abort_flag;
  uint32_t tmem;
  uint32_t mcopy_s;        // merge bulk copies issued (phases of the mcopy barrier)
  int32_t ub[2];           // the CTA's unit range
  int32_t nduty;           // split segments this CTA completes and merges
  int32_t duty[2][4];      // b, head group, first CTA, pieces
  int32_t qexp[2][kHeads]; // per-head power of two of the query pieces
  float alpha[kHeads];     // rescale factors of a raised maximum
  float mh[kHeads];        // a piece's per-head maxima
  float lh[kHeads];        // and denominators
  int32_t warp_tot[8];     // plan scan scratch
  float gm[kMergeWarps];   // grid merge: per-warp maxima
  float gl[kMergeWarps];   // and denominators
  float gacc[kMergeWarps][32];
};

template <bool QF8>
struct BLay {
  static constexpr int NQ = QF8 ? kHeads : kHeads * kQP;  // S^T columns
  static constexpr int NO = kHeads * kPP;                  // O^T columns
  static constexpr uint32_t kCols = 512;
  static constexpr size_t ring = 0;
  static constexpr size_t qBytes = static_cast<size_t>(NQ) * 128;
  // ring: K stages [kNk][128][128], then V stages [kNv][128][128]
  static constexpr size_t vring = ring + static_cast<size_t>(kNk) * kHalf;
  static constexpr size_t ringBytes = static_cast<size_t>(kNk + kNv) * kHalf;
  static constexpr size_t qbuf = ring + ringBytes;  // [2][NQ][128]
  static constexpr size_t pBytes = static_cast<size_t>(NO) * 128;             // 16 KB
  static constexpr size_t pbuf = qbuf + 2 * qBytes;                           // [kNp][NO][128]
  static constexpr size_t bars = pbuf + kNp * pBytes;
  // kfull[kNk], vfull[kNv], kempty[kNk], vempty[kNv], pfull[kNp], sfull[2], sfree[2],
  // qfull[2], fin, pvfin, mcopy
  static constexpr int kBars = 2 * kNk + 2 * kNv + kNp + 9;
  static constexpr size_t misc = bars + kBars * sizeof(uint64_t);
  static constexpr size_t plan = (misc + sizeof(BMisc) + 15) & ~size_t(15);
  __host__ __device__ static size_t total(int B, int Hkv) {
    return ((plan + (3 * static_cast<size_t>(B) + 2) * 4 + 2 * static_cast<size_t>(Hkv) * 4 + 15) &
            ~size_t(15)) + 1024;
  }
};
static_assert(BLay<false>::qbuf % 1024 == 0 && BLay<false>::pbuf % 1024 == 0, "swizzled tiles");
static_assert(BLay<true>::qbuf % 1024 == 0 && BLay<true>::pbuf % 1024 == 0, "swizzled tiles");

// The CTA's tiles in order: unit u of the range is block pg (of the
// sequence's attended pages) of head group hg of sequence b.
struct BIt {
  int64_t u, u1;
  int b, hg, pages, pg;
  int p0;          // first page of the current piece
  int t, piece;
  bool valid, first, last;
  int segs;

  KVQ_DEVI void locate(const int32_t* seq_off, int B) {
    b = find_seq(seq_off, B, u);
    pages = (seq_off[b + 1] - seq_off[b]) / segs;
    const int r = static_cast<int>(u - seq_off[b]);
    hg = r / pages;
    pg = r - hg * pages;
    p0 = pg;
  }
  KVQ_DEVI void set_last() { last = pg == pages - 1 || u + 1 == u1; }
  KVQ_DEVI void start(const int32_t* seq_off, int B, int segs_, int64_t u0_, int64_t u1_) {
    segs = segs_;
    u = u0_;
    u1 = u1_;
    t = 0;
    piece = 0;
    valid = u < u1;
    first = true;
    if (valid) {
      locate(seq_off, B);
      set_last();
    }
  }
  KVQ_DEVI void next(const int32_t* seq_off, int B) {
    ++t;
    ++u;
    if (u >= u1) {
      valid = false;
      return;
    }
    if (pg + 1 < pages) {
      ++pg;
      first = false;
    } else {
      locate(seq_off, B);
      ++piece;
      first = true;
    }
    set_last();
  }
  // The piece covers its whole segment (valid at its last tile).
  KVQ_DEVI bool whole() const { return p0 == 0 && pg == pages - 1; }
};

// The query of segment (b, hg) into a Q^T tile (B operand of S^T = K Q^T):
// four rounds of 128 threads, round k for query heads 8 k .. 8 k + 7 of the
// group (16 threads per head, 8 dims each).  bf16 query: rows 3 h + k hold
// the pieces of 2^a_h q_h (a_h into qexp[h]); FP8-domain query: row h holds
// enc(q_h / sQ_h).  raw[k]: the thread's 8 bf16 values of round k.
template <int FMT, bool QF8>
KVQ_DEVI void write_q_blk(const DecodeParams& p, int hg, const uint4 (&raw)[4], uint32_t qaddr,
                          int32_t* qexp, int tid) {
  const int sub = tid & 15;
  const uint32_t chunk_off = static_cast<uint32_t>((sub & 1) * 8);
#pragma unroll
  for (int k4 = 0; k4 < 4; ++k4) {
    const int h = k4 * 8 + (tid >> 4);
    const uint32_t w[4] = {raw[k4].x, raw[k4].y, raw[k4].z, raw[k4].w};
    float x[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16lo_to_f32(w[i]);
      x[2 * i + 1] = bf16hi_to_f32(w[i]);
    }
    if (QF8) {
      const float sq = __ldg(p.qs + (p.q_per_head ? hg * kHeads + h : 0));
      uint32_t c[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t lo = f32x2_to_fp8x2<FMT>(__fdiv_rn(x[4 * j], sq), __fdiv_rn(x[4 * j + 1], sq));
        const uint32_t hi =
            f32x2_to_fp8x2<FMT>(__fdiv_rn(x[4 * j + 2], sq), __fdiv_rn(x[4 * j + 3], sq));
        c[j] = lo | (hi << 16);
      }
      sts64(qaddr + h * 128 + ((((sub >> 1) ^ (h & 7))) << 4) + chunk_off, c[0], c[1]);
      continue;
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
    if (sub == 0) qexp[h] = a;
    const float sc = pow2i(a);
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = x[i] * sc;  // exact: a power of two, no overflow
#pragma unroll
    for (int k = 0; k < kQP; ++k) {
      uint32_t c[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t lo = f32x2_to_fp8x2<KVQ_FMT_E4M3>(y[4 * j], y[4 * j + 1]);
        const uint32_t hi = f32x2_to_fp8x2<KVQ_FMT_E4M3>(y[4 * j + 2], y[4 * j + 3]);
        c[j] = lo | (hi << 16);
        if (k + 1 < kQP) {
          float d0, d1, d2, d3;
          dec_e4m3x2(lo, d0, d1);
          dec_e4m3x2(hi, d2, d3);
          y[4 * j] = (y[4 * j] - d0) * 16.f;
          y[4 * j + 1] = (y[4 * j + 1] - d1) * 16.f;
          y[4 * j + 2] = (y[4 * j + 2] - d2) * 16.f;
          y[4 * j + 3] = (y[4 * j + 3] - d3) * 16.f;
        }
      }
      const int row = kQP * h + k;
      sts64(qaddr + row * 128 + ((((sub >> 1) ^ (row & 7))) << 4) + chunk_off, c[0], c[1]);
    }
  }
}

// Raw bf16 query words of thread tid for segment (b, hg): round k covers
// query head 8 k + tid / 16 of the group, dims 8 (tid % 16) ...
KVQ_DEVI void load_q_blk(const DecodeParams& p, int b, int hg, int tid, uint4 (&raw)[4]) {
  const int sub = tid & 15;
#pragma unroll
  for (int k4 = 0; k4 < 4; ++k4) {
    const int h = k4 * 8 + (tid >> 4);
    const int64_t qrow = static_cast<int64_t>(b) * p.Hq + hg * kHeads + h;
    if (guard(b >= 0 && b < p.B && qrow < static_cast<int64_t>(p.B) * p.Hq, p.status, 12))
      raw[k4] = reinterpret_cast<const uint4*>(p.q + qrow * kDH)[sub];
    else
      raw[k4] = make_uint4(0u, 0u, 0u, 0u);
  }
}

KVQ_DEVI uint32_t ld_acquire_gpu(const uint32_t* a) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// Softmax-side work that runs once per piece or rarely, kept out of line so
// that the per-tile loop stays small in the instruction cache.

// A timeout in a wait: the first one raises the abort flag and the status.
KVQ_DEVI void raise_abort(volatile uint32_t* abort_flag, uint32_t* status) {
  if (!*abort_flag) {
    *abort_flag = 1u;
    flag_status(status, KVQ_DEV_WAIT_TIMEOUT);
  }
}

// A bounded wait by a whole warp; false (and the abort raised) on timeout.
KVQ_DEVI bool wait_warp(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag, uint32_t* status) {
  if (__all_sync(kFull, mbar_test_wait(bar, parity))) return true;  // the usual case: done already
  const bool w = __all_sync(kFull, wait_or_abort(bar, parity, abort_flag));
  if (!w && (threadIdx.x & 31) == 0) raise_abort(abort_flag, status);
  return w;
}

// The query of segment (b, hg) into the Q^T tile at qaddr.
template <int FMT, bool QF8>
__device__ __noinline__ void q_tile_blk(const DecodeParams& p, int b, int hg, uint32_t qaddr,
                                        int32_t* qexp, int tid) {
  uint4 raw[4];
  load_q_blk(p, b, hg, tid, raw);
  write_q_blk<FMT, QF8>(p, hg, raw, qaddr, qexp, tid);
}

// Per-thread softmax state of the current piece: running maxima, partial
// denominators and logit factors of the thread's four query heads.
struct SoftSt {
  float m[kGQ], l[kGQ], cq[kGQ];
};

// What the out-of-line softmax helpers need of the CTA.
struct SoftCtx {
  BMisc* mi;
  uint64_t* vempty;
  volatile uint32_t* abort_flag;
  uint32_t* status;
  uint32_t tmem_o;  // this warp's lanes of O^T
  int j, tt;        // KV head and token of the thread's tile row
};

// A tile raised some running maximum by more than 2^8: the new maxima (the
// tile's maxima over the half warp's tokens), the rescaled partial sums and,
// where O^T already holds tiles of the piece, its rescaled columns.
__device__ __noinline__ bool raise_max(SoftSt& st, float x0, float x1, float x2, float x3,
                                       const SoftCtx& cx, int t, bool ok) {
  constexpr float kThr = kRescaleThreshold;
  const float x[kGQ] = {x0, x1, x2, x3};
  bool real = false;
#pragma unroll
  for (int i = 0; i < kGQ; ++i) {
    float tm = x[i];
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) tm = fmaxf(tm, __shfl_xor_sync(kFull, tm, off));
    const float nm = tm > st.m[i] + kThr ? tm : st.m[i];
    const float a = (st.m[i] == -INFINITY) ? 0.f : fast_exp2(st.m[i] - nm);
    real |= nm != st.m[i] && st.m[i] != -INFINITY;  // O^T holds tiles of this piece
    const float al = nm != st.m[i] ? a : 1.f;  // an unchanged maximum keeps its sums
    if (cx.tt == 0) cx.mi->alpha[cx.j * kGQ + i] = al;
    st.l[i] *= al;  // m = -inf before: no token yet, l = 0
    st.m[i] = nm;
  }
  // O^T already holds earlier tiles of this piece: rescale its columns once
  // the last PV issued (tile t - 1) is done
  if (soft_bar_or(real)) {
    if (ok)
      ok = wait_warp(&cx.vempty[(t - 1) % kNv], static_cast<uint32_t>(((t - 1) / kNv) & 1),
                     cx.abort_flag, cx.status);
    if (ok) {
      tc_fence_after();
#pragma unroll 1
      for (int c0 = 0; c0 < kHeads * kPP; c0 += 32) {
        float o[32];
        tmem_ld32(cx.tmem_o + c0, o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= cx.mi->alpha[(c0 + i) / kPP];
        tmem_st32(cx.tmem_o + c0, o);
      }
      tc_fence_before();
    }
  }
  soft_bar();  // alpha read by every thread before its next write
  return ok;
}

// The piece's last tile t (stage s) is in O^T once PV(t) is done: its
// output rows (a whole segment), or its published partial state (a split
// segment; under LAST, the arrival that may make this CTA the merger).
template <bool GRID>
__device__ __noinline__ bool piece_end(const DecodeParams& p, const SoftCtx& cx, const SoftSt& st,
                                       int b, int hg, int pages, bool whole, int s, int t, bool ok,
                                       const float* sv_s, const int32_t* vseq_off,
                                       const CostSplit& cost_split, int segs) {
  const int r = threadIdx.x;
  BMisc* mi = cx.mi;
  if (ok)
    ok = wait_warp(&cx.vempty[s], static_cast<uint32_t>((t / kNv) & 1), cx.abort_flag, cx.status);
  float o[kHeads];
#pragma unroll
  for (int h = 0; h < kHeads; ++h) o[h] = 0.f;
  if (ok) {
    tc_fence_after();
#pragma unroll
    for (int c0 = 0; c0 < kHeads * kPP; c0 += 32) {
      float v[32];
      tmem_ld32(cx.tmem_o + c0, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int col = c0 + i, h = col / kPP, k = col % kPP;
        const float f = k == 0 ? 1.f : (k == 1 ? 1.f / 16.f : (k == 2 ? 1.f / 256.f : 1.f / 4096.f));
        o[h] = fmaf(v[i], f, o[h]);
      }
    }
    tc_fence_before();
  }
  // per-head maxima and denominators (sums over the half warp's tokens)
#pragma unroll
  for (int i = 0; i < kGQ; ++i) {
    float v = st.l[i];
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    if (cx.tt == 0) {
      mi->lh[cx.j * kGQ + i] = v;
      mi->mh[cx.j * kGQ + i] = st.m[i];
    }
  }
  soft_bar();
  const int sigma = b * segs + hg;
  if (whole) {
    const int64_t obase = (static_cast<int64_t>(b) * p.Hq + hg * kHeads) * kDH + r;
#pragma unroll
    for (int h = 0; h < kHeads; ++h) {
      const float Lh = mi->lh[h];
      const float f = Lh > 0.f ? sv_s[hg * kHT + h / kGQ] / Lh : 0.f;
      const int64_t oi = obase + static_cast<int64_t>(h) * kDH;
      if (guard(oi >= 0 && oi < static_cast<int64_t>(p.B) * p.Hq * kDH, p.status, 3))
        p.out[oi] = static_cast<uint16_t>(f32x2_to_bf16x2(o[h] * f, 0.f) & 0xFFFFu);
    }
    soft_bar();  // lh / mh read by every thread before their next write
    return ok;
  }
  // ---- a split segment: publish this piece
  const int64_t slot = static_cast<int64_t>(blockIdx.x) + sigma;
  const bool slot_ok = guard(slot >= 0 && (slot + 1) * kHT <= p.n_slots, p.status, 4);
  if (slot_ok) {
    float* wo = p.ws_o + slot * kHeads * kDH + r;
#pragma unroll
    for (int h = 0; h < kHeads; ++h) wo[h * kDH] = o[h];
    if (r < kHeads)
      *reinterpret_cast<float2*>(p.ws_ml + (slot * kHeads + r) * 2) = make_float2(mi->mh[r], mi->lh[r]);
  }
  soft_bar();  // every store of the piece before the arrival; lh / mh reads done
  if (!GRID && r == 0 && slot_ok && !*cx.abort_flag) {
    const int v_first = vseq_off[b] + hg * (pages + kBlkPieceCost) + kBlkPieceCost;
    const int seg_lo = cost_split.cta_of(v_first);
    const int seg_n = cost_split.cta_of(v_first + pages - 1) - seg_lo + 1;
    const uint32_t prev = atom_add_acq_rel_gpu(p.ws_cnt + sigma, 1u);
    if (prev + 1 == static_cast<uint32_t>(seg_n) && mi->nduty < 2) {
      int32_t* d = mi->duty[mi->nduty];
      d[0] = b;
      d[1] = hg;
      d[2] = seg_lo;
      d[3] = seg_n;
      mi->nduty = mi->nduty + 1;
    }
  }
  return ok;
}

template <int FMT, bool QF8, bool GRID>
__global__ void __launch_bounds__(kThreadsB, 1)
    decode_blk_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
  using Lo = BLay<QF8>;
  constexpr int NQ = Lo::NQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lo::bars);
  // K and V have rings of their own: a K stage is free once QK^T of its tile
  // is done, long before PV of the tile, so K copies run ahead of V ones.
  uint64_t* kfull = bars;              // [kNk] K of the tile landed (TMA bytes)
  uint64_t* vfull = kfull + kNk;       // [kNv] V landed
  uint64_t* kempty = vfull + kNv;      // [kNk] QK^T of the stage's tile done (commit)
  uint64_t* vempty = kempty + kNk;     // [kNv] PV of the stage's tile done (commit)
  uint64_t* pfull = vempty + kNv;      // [kNp] P^T tile t % kNp written (4 warp arrivals)
  uint64_t* sfull = pfull + kNp;       // [2] S^T buffer written (commit)
  uint64_t* sfree = sfull + 2;         // [2] S^T buffer read (4 warp arrivals)
  uint64_t* qfull = sfull + 4;         // [2] Q^T tile written (4 warp arrivals)
  uint64_t* fin = sfull + 6;           // every QK^T MMA done (commit)
  uint64_t* pvfin = sfull + 7;         // every PV MMA done (commit)
  uint64_t* mcopy = sfull + 8;         // the bulk copy of a segment's pieces for its merge
  // A parity wait for phase k is sound only while the barrier has completed
  // k or k + 1 phases: every waiter waits each barrier's phases in order, and
  // a barrier's next phase needs the waiter's own later progress.
  BMisc* mi = reinterpret_cast<BMisc*>(smem + Lo::misc);
  volatile uint32_t* abort_flag = &mi->abort_flag;
  int32_t* seq_off = reinterpret_cast<int32_t*>(smem + Lo::plan);  // [B+1]
  int32_t* len_s = seq_off + p.B + 1;                              // [B]
  int32_t* vseq_off = len_s + p.B;                                 // [B+1]
  float* sk_s = reinterpret_cast<float*>(vseq_off + p.B + 1);      // [Hkv]
  float* sv_s = sk_s + p.Hkv;                                      // [Hkv]
  const int segs = p.Hkv / kHT;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < kNk; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
      mi->kiss[i] = -1;
    }
    for (int i = 0; i < kNv; ++i) {
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], 1);
      mi->viss[i] = -1;
    }
    for (int i = 0; i < kNp; ++i) mbar_init(&pfull[i], 4);
    for (int i = 0; i < kFlags; ++i) mi->tflag[i] = 0xFFFFFFFFu;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sfree[i], 4);
      mbar_init(&qfull[i], 4);
    }
    mbar_init(fin, 1);
    mbar_init(pvfin, 1);
    mbar_init(mcopy, 1);
    mi->abort_flag = 0u;
    mi->mcopy_s = 0u;
    mi->nduty = 0;
    fence_mbar_init();
  }
  // P^T tiles are zero outside their diagonal blocks: cleared once, the
  // softmax rewrites the same bytes of every tile.
  for (int i = tid; i < static_cast<int>(kNp * Lo::pBytes / 16); i += kThreadsB)
    sts128(sbase + static_cast<uint32_t>(Lo::pbuf) + 16 * i, 0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  if (warp == 5) {
    tmem_alloc(&mi->tmem, Lo::kCols);
    tc_fence_before();
  }
  if (!p.early) {
    // The metadata read first (lengths, scales, this CTA's share of the block
    // tables and of q) into L2 while the previous kernel drains: a prefetch
    // returns no data, so what that kernel still writes is read after the
    // wait as usual.
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
      if (lane >= 8 && lane < 16)
        slice(p.block_tables, static_cast<int64_t>(p.B) * p.max_blocks * 4, lane - 8);
      if (lane >= 16 && lane < 24) slice(p.q, static_cast<int64_t>(p.B) * p.Hq * kDH * 2, lane - 16);
    }
    pdl_wait();
    pdl_allow_next();
  }
  build_plan<true, kThreadsB>(p, seq_off, len_s, vseq_off, sk_s, sv_s, mi->warp_tot, segs,
                              kBlkPieceCost);  // ends in __syncthreads
  tc_fence_after();
  const uint32_t tmem = mi->tmem;
  const int c = blockIdx.x;
  const int64_t W = seq_off[p.B];
  const int Pe = static_cast<int>(W < p.P ? W : p.P);
  const CostSplit cost_split(vseq_off[p.B], Pe);
  if ((tid == 0 || tid == 32) && c < Pe)
    mi->ub[tid >> 5] =
        pages_before(seq_off, vseq_off, p.B, segs, cost_split(c + (tid >> 5)), kBlkPieceCost);
  __syncthreads();
  const int64_t u0 = c < Pe ? mi->ub[0] : 0, u1 = c < Pe ? mi->ub[1] : 0;

  auto fail = [&]() {
    if (!*abort_flag) {
      *abort_flag = 1u;
      flag_status(p.status, KVQ_DEV_WAIT_TIMEOUT);
    }
  };
  // The CTAs holding the pieces of segment (b, hg): [lo, lo + n).
  auto seg_ctas = [&](int b, int hg, int pages, int& lo, int& n) {
    const int v_first = vseq_off[b] + hg * (pages + kBlkPieceCost) + kBlkPieceCost;
    lo = cost_split.cta_of(v_first);
    n = cost_split.cta_of(v_first + pages - 1) - lo + 1;
  };

  // The cache row of a tile's block (the first of its eight KV heads), or
  // -1 when its block id is out of range.
  auto tile_row = [&](int blk, int hg) {
    if (blk < 0 || blk >= p.num_blocks) return -1;
    const int64_t row = (static_cast<int64_t>(blk) * p.Hkv + hg * kHT) * kBS;
    return (row >= 0 && row + kRows <= p.rows && row + kRows <= INT32_MAX) ? static_cast<int>(row) : -1;
  };
  if (warp == 4 || warp == 7) {
    // ------------------------------------------------------------ producers
    // Warp 4 copies the tiles' K, warp 7 their V, each into its own ring.
    // Lane i looks up tile 32 g + i; the ids of group g + 1 are requested
    // when group g starts, so their loads hide behind 32 tiles.
    const bool isk = warp == 4;
    const int NS = isk ? kNk : kNv;  // the ring's stages
    uint64_t* fullb = isk ? kfull : vfull;
    uint64_t* emptyb = isk ? kempty : vempty;
    int32_t* iss = isk ? mi->kiss : mi->viss;
    const CUtensorMap* map = isk ? &tmk : &tmv;
    uint8_t* ring = smem + (isk ? Lo::ring : Lo::vring);
    auto look_issue = [&](int64_t t, int& blk, int& meta) {
      // meta: -2 no tile; else (hg << 1 | newest-token block)
      meta = -2;
      blk = -1;
      const int64_t u = u0 + t;
      if (u >= u1) return;
      const int b = find_seq(seq_off, p.B, u);
      const int pages = (seq_off[b + 1] - seq_off[b]) / segs;
      const int r = static_cast<int>(u - seq_off[b]);
      const int hg = r / pages, pg = r - hg * pages;
      const int col = first_page_of(p, len_s[b]) + pg;
      if (col >= 0 && col < p.max_blocks)
        blk = p.block_tables[static_cast<int64_t>(b) * p.max_blocks + col];
      else if (isk)
        guard(false, p.status, 0);
      meta = (hg << 1) | (pg == pages - 1 ? 1 : 0);
    };
    auto look_finish = [&](int blk, int meta, bool& lastp) {
      lastp = meta >= 0 && (meta & 1);
      if (meta < 0) return -2;
      const int row = tile_row(blk, meta >> 1);
      if (row < 0 && isk) flag_status(p.status, KVQ_DEV_BAD_BLOCK);
      return row;
    };
    const uint64_t pol = l2_evict_first_policy();
    bool waited = !p.early;
    const int64_t nt = u1 - u0;
    int nb_blk = -1, nb_meta = -2, cur_row = -2;
    bool cur_last = false;
    if (nt > 0) look_issue(lane, nb_blk, nb_meta);
    for (int64_t t = 0; t < nt; ++t) {
      const int i = static_cast<int>(t & 31), s = static_cast<int>(t % NS);
      if (i == 0) {
        cur_row = look_finish(nb_blk, nb_meta, cur_last);
        look_issue(t + 32 + lane, nb_blk, nb_meta);
      }
      const int row = __shfl_sync(kFull, cur_row, i);
      const bool lastp = __shfl_sync(kFull, cur_last ? 1 : 0, i) != 0;
      if (isk && lane == 0)  // tile t's validity, for the softmax (overwritten 16 tiles on)
        *reinterpret_cast<volatile uint32_t*>(&mi->tflag[t & (kFlags - 1)]) =
            (static_cast<uint32_t>(t) << 1) | (row >= 0 ? 1u : 0u);
      if (!waited && lastp) {  // the block of a sequence's newest token: wait first
        pdl_wait();
        waited = true;
      }
      bool ok = true;
      if (lane == 0) {
        ok = t < NS ||
             wait_or_abort(&emptyb[s], static_cast<uint32_t>(((t / NS) - 1) & 1), abort_flag);
        ok = ok && !*abort_flag;
        if (!ok) fail();
      }
      if (!__shfl_sync(kFull, ok ? 1 : 0, 0)) break;
      if (lane == 0) {
        iss[s] = row < 0 ? -1 : static_cast<int32_t>(t);  // the stage's copy in flight, if any
        if (row < 0) {
          mbar_arrive(&fullb[s]);  // nothing to load: complete the phase by hand
        } else {
          mbar_arrive_expect_tx(&fullb[s], kHalf);
          tma_load_2d_hint(ring + static_cast<size_t>(s) * kHalf, map, 0, row, &fullb[s], pol);
        }
      }
      __syncwarp();
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ QK^T issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_f8(kRows, NQ, tc_type(FMT), QF8 ? tc_type(FMT) : kTcE4M3,
                                      false, false);
      // a 32-byte K step adds 2 to the start address field, a stage kHalf / 16
      const uint64_t dk0 = sw128_desc(sbase + static_cast<uint32_t>(Lo::ring));
      const uint64_t dq0 = sw128_desc(sbase + static_cast<uint32_t>(Lo::qbuf));
      bool ok = true;
      BIt it;
      it.start(seq_off, p.B, segs, u0, u1);
      for (; it.valid && ok; it.next(seq_off, p.B)) {
        const int t = it.t, s = t % kNk, sb = t & 1;
        if (it.first)
          ok = wait_or_abort(&qfull[it.piece & 1], static_cast<uint32_t>((it.piece >> 1) & 1),
                             abort_flag);
        if (ok && t >= 2)
          ok = wait_or_abort(&sfree[sb], static_cast<uint32_t>(((t >> 1) - 1) & 1), abort_flag);
        if (ok) ok = wait_or_abort(&kfull[s], static_cast<uint32_t>((t / kNk) & 1), abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dk = dk0 + static_cast<uint64_t>(s) * (kHalf >> 4);
        const uint64_t dq = dq0 + static_cast<uint64_t>(it.piece & 1) * (Lo::qBytes >> 4);
#pragma unroll
        for (int k = 0; k < kDH / 32; ++k)
          mma_f8_ss(tmem + sb * 128, dk + 2 * k, dq + 2 * k, id_qk, k > 0 ? 1u : 0u);
        mma_commit(&sfull[sb]);
        mma_commit(&kempty[s]);  // the K stage is free once these MMAs are done
      }
      if (!ok) fail();
      mma_commit(fin);  // completes when every MMA issued above has
      if (!mbar_wait(fin, 0u)) fail();
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------------------ PV warp
    // Once P^T(t) is written and V(t) has landed, the warp clears the V rows
    // of masked tokens (their bytes may be anything, NaN included, and
    // p = 0 would not clear a NaN), then one lane issues the MMAs.
    const uint32_t id_pv = idesc_f8(kDH, Lo::NO, tc_type(FMT), kTcE4M3, true, false);
    // V as the MN-major A operand: a 32-row K step is 4096 bytes (256 in the
    // address field); the P^T tile K-major like Q
    const uint64_t dv0 = sw128_desc(sbase + static_cast<uint32_t>(Lo::vring), 16384, 1024);
    const uint64_t dp0 = sw128_desc(sbase + static_cast<uint32_t>(Lo::pbuf));
    bool ok = true;
    BIt it;
    it.start(seq_off, p.B, segs, u0, u1);
    for (; it.valid; it.next(seq_off, p.B)) {
      const int t = it.t, s = t % kNv, pb = t % kNp;
      if (lane == 0) {
        ok = wait_or_abort(&pfull[pb], static_cast<uint32_t>((t / kNp) & 1), abort_flag) &&
             wait_or_abort(&vfull[s], static_cast<uint32_t>((t / kNv) & 1), abort_flag);
        if (!ok) fail();
      }
      ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      __syncwarp();  // the masks lane 0 acquired, for every lane
      bool zeroed = false;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t m = mi->vmask[pb][w];
        if (m == kFull) continue;
        zeroed = true;
        if (!((m >> lane) & 1u)) {
          const uint32_t vr = sbase + static_cast<uint32_t>(Lo::vring + s * kHalf) + (32 * w + lane) * 128;
#pragma unroll
          for (int i = 0; i < 8; ++i) sts128(vr + 16 * i, 0u, 0u, 0u, 0u);
        }
      }
      if (zeroed) fence_proxy_async_smem();  // the cleared rows -> the tensor core
      __syncwarp();
      if (lane == 0) {
        tc_fence_after();
        const uint64_t dv = dv0 + static_cast<uint64_t>(s) * (kHalf >> 4);
        const uint64_t dp = dp0 + static_cast<uint64_t>(pb) * (Lo::pBytes >> 4);
#pragma unroll
        for (int k = 0; k < kRows / 32; ++k)
          mma_f8_ss(tmem + kOS, dv + 256 * k, dp + 2 * k, id_pv, (k > 0 || !it.first) ? 1u : 0u);
        mma_commit(&vempty[s]);  // the V stage and P^T tile t % kNp are free, O^T holds this tile
      }
      __syncwarp();
    }
    if (lane == 0) {
      mma_commit(pvfin);
      if (!mbar_wait(pvfin, 0u)) fail();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int r = tid;              // tile row r = TMEM lane r; dim r of O^T
    const int hi = lane >> 4;       // which of the warp's two KV heads
    const int j = 2 * warp + hi;    // KV head of the group
    const int tt = lane & 15;       // token of the block
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    if (p.early) {  // q and every write wait for the previous kernel
      pdl_wait();
      pdl_allow_next();
    }
    // Sequences with nothing to attend to get a zero output row.
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
      if (seq_off[b + 1] != seq_off[b]) continue;
      uint16_t* orow = p.out + static_cast<int64_t>(b) * p.Hq * kDH;
      for (int i = r; i < p.Hq * kDH; i += kSoftThreads) orow[i] = 0;
    }
    auto wait_w = [&](uint64_t* bar, uint32_t parity) {
      return wait_warp(bar, parity, abort_flag, p.status);
    };
    SoftCtx cx;
    cx.mi = mi;
    cx.vempty = vempty;
    cx.abort_flag = abort_flag;
    cx.status = p.status;
    cx.tmem_o = tmem + lane_base + kOS;
    cx.j = j;
    cx.tt = tt;
    // q rows of segment (b, hg) into L2 (32 heads x 256 bytes)
    auto q_prefetch = [&](int b, int hg) {
      if (r < 64) {
        const uint8_t* a = reinterpret_cast<const uint8_t*>(p.q + (static_cast<int64_t>(b) * p.Hq + hg * kHeads) * kDH);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a + 128 * r));
      }
    };
    bool ok = true;  // this warp's waits so far (the named barriers run regardless)
    BIt it;
    it.start(seq_off, p.B, segs, u0, u1);
    BIt nx = it;  // the next piece to get its Q
    if (it.valid) {
      q_tile_blk<FMT, QF8>(p, it.b, it.hg, sbase + static_cast<uint32_t>(Lo::qbuf), mi->qexp[0], r);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&qfull[0]);
      while (nx.valid && nx.piece == 0) nx.next(seq_off, p.B);
      if (nx.valid) q_prefetch(nx.b, nx.hg);
    }
    constexpr float kThr = kRescaleThreshold;
    SoftSt st;
    int L = 0, lo = 0, fp = 0;
    // Tile t's validity as the K producer published it (lane 0 polls, bounded).
    auto tile_ok = [&](int t) {
      uint32_t v = 0u;
      if (lane == 0) {
        const volatile uint32_t* f = &mi->tflag[t & (kFlags - 1)];
        bool got = false;
        for (uint32_t i = 0; i < kMaxPolls && !got; ++i) {
          v = *f;
          got = (v >> 1) == static_cast<uint32_t>(t);
          if (!got && (i & 63u) == 63u && *abort_flag) break;
        }
        if (!got) {
          raise_abort(abort_flag, p.status);
          v = 0u;
        }
      }
      return (__shfl_sync(kFull, v, 0) & 1u) != 0u;
    };
    // The logits of token tt for head j's four queries from S^T buffer sb.
    auto logits = [&](int sb, float (&sv4)[kGQ]) {
      if (QF8) {
        uint32_t a[16];
        tmem_ld16(tmem + lane_base + sb * 128 + 8 * warp, a);
#pragma unroll
        for (int i = 0; i < kGQ; ++i) sv4[i] = __uint_as_float(hi ? a[kGQ + i] : a[i]);
      } else {
        float a[32];
        tmem_ld32(tmem + lane_base + sb * 128 + 24 * warp, a);
#pragma unroll
        for (int i = 0; i < kGQ; ++i) {
          const float s0 = hi ? a[12 + 3 * i] : a[3 * i];
          const float s1 = hi ? a[13 + 3 * i] : a[3 * i + 1];
          const float s2 = hi ? a[14 + 3 * i] : a[3 * i + 2];
          sv4[i] = fmaf(s2, 1.f / 256.f, fmaf(s1, 1.f / 16.f, s0));
        }
      }
    };
    // The probability pieces of token tt into P^T tile pb.
    auto store_p = [&](int pb, const uint32_t (&pc)[2][kPP]) {
      const uint32_t pt = sbase + static_cast<uint32_t>(Lo::pbuf + pb * Lo::pBytes);
#pragma unroll
      for (int i = 0; i < kGQ; ++i)
#pragma unroll
        for (int k = 0; k < kPP; ++k)
          sts8(pt + sw_off((j * kGQ + i) * kPP + k, r), (pc[i >> 1][k] >> ((i & 1) * 8)) & 0xFFu);
    };
    // Two tiles of a piece per step (one when the piece ends at the first):
    // A = it, B = the tile after it.
    while (it.valid) {
      const bool has2 = !it.last;
      BIt itB = it;
      if (has2) itB.next(seq_off, p.B);
      const int tA = it.t, tB = tA + 1;
      if (it.first) {
        soft_bar();  // qexp of this piece is written (by the Q writers)
        L = len_s[it.b];
        lo = window_lo(p, L);
        fp = lo / kBS;
        const float lk = sk_s[it.hg * kHT + j] * p.logit_scale;
#pragma unroll
        for (int i = 0; i < kGQ; ++i) {
          const int h = j * kGQ + i;
          st.m[i] = -INFINITY;
          st.l[i] = 0.f;
          if (QF8)
            st.cq[i] = lk * __ldg(p.qs + (p.q_per_head ? it.hg * kHeads + h : 0));
          else
            st.cq[i] = lk * pow2i(-mi->qexp[it.piece & 1][h]);
        }
      }
      const bool okA = ok && tile_ok(tA);
      const bool okB = has2 && ok && tile_ok(tB);
      // ---- logits of token tt for head j's queries, tiles A and B
      if (ok) ok = wait_w(&sfull[tA & 1], static_cast<uint32_t>((tA >> 1) & 1));
      if (ok && has2) ok = wait_w(&sfull[tB & 1], static_cast<uint32_t>((tB >> 1) & 1));
      float sA[kGQ], sB[kGQ];
#pragma unroll
      for (int i = 0; i < kGQ; ++i) sA[i] = sB[i] = 0.f;
      if (ok) {
        tc_fence_after();
        __syncwarp();
        logits(tA & 1, sA);
        if (has2) logits(tB & 1, sB);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sfree[tA & 1]);
          if (has2) mbar_arrive(&sfree[tB & 1]);
        }
      }
      const int posA = (fp + it.pg) * kBS + tt, posB = posA + kBS;
      const bool vA = ok && okA && posA >= lo && posA < L;
      const bool vB = ok && okB && posB >= lo && posB < L;
      float xA[kGQ], xB[kGQ];
      bool need = false;  // a logit exceeds its running maximum by more than 2^8
#pragma unroll
      for (int i = 0; i < kGQ; ++i) {
        xA[i] = vA ? sA[i] * st.cq[i] : -INFINITY;
        xB[i] = vB ? sB[i] * st.cq[i] : -INFINITY;
        need |= fmaxf(xA[i], xB[i]) > st.m[i] + kThr;
      }
      // ---- running maxima: raised only when a tile exceeds them by 2^8
      if (soft_bar_or(need)) {
        SoftSt tmp = st;
        ok = raise_max(tmp, fmaxf(xA[0], xB[0]), fmaxf(xA[1], xB[1]), fmaxf(xA[2], xB[2]),
                       fmaxf(xA[3], xB[3]), cx, tA, ok);
        st = tmp;
      }
      // ---- probabilities and their pieces into P^T tiles tA % 4, tB % 4
      float pA[kGQ], pB[kGQ];
#pragma unroll
      for (int i = 0; i < kGQ; ++i) {
        const bool live = st.m[i] != -INFINITY;
        pA[i] = (xA[i] == -INFINITY || !live) ? 0.f : fast_exp2(xA[i] - st.m[i]);
        pB[i] = (xB[i] == -INFINITY || !live) ? 0.f : fast_exp2(xB[i] - st.m[i]);
        st.l[i] += pA[i] + pB[i];
      }
      uint32_t pcA[2][kPP], pcB[2][kPP];
      p_pieces(pA[0], pA[1], pcA[0]);
      p_pieces(pA[2], pA[3], pcA[1]);
      p_pieces(pB[0], pB[1], pcB[0]);
      p_pieces(pB[2], pB[3], pcB[1]);
      // a P^T tile was last read by PV four tiles before
      if (ok && tA >= kNp)
        ok = wait_w(&vempty[(tA - kNp) % kNv], static_cast<uint32_t>(((tA - kNp) / kNv) & 1));
      if (ok && has2 && tB >= kNp)
        ok = wait_w(&vempty[(tB - kNp) % kNv], static_cast<uint32_t>(((tB - kNp) / kNv) & 1));
      if (ok) {
        store_p(tA % kNp, pcA);
        if (has2) store_p(tB % kNp, pcB);
      }
      {  // the masked rows, for the PV warp to clear in V
        const uint32_t mA = __ballot_sync(kFull, vA), mB = __ballot_sync(kFull, vB);
        if (lane == 0) {
          mi->vmask[tA % kNp][warp] = mA;
          if (has2) mi->vmask[tB % kNp][warp] = mB;
        }
      }
      fence_proxy_async_smem();  // P^T bytes -> the tensor core
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&pfull[tA % kNp]);
        if (has2) mbar_arrive(&pfull[tB % kNp]);
      }
      // ---- the next piece's Q once this piece has started
      if (it.first && nx.valid) {
        q_tile_blk<FMT, QF8>(p, nx.b, nx.hg,
                             sbase + static_cast<uint32_t>(Lo::qbuf + (nx.piece & 1) * Lo::qBytes),
                             mi->qexp[nx.piece & 1], r);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&qfull[nx.piece & 1]);
        const int cur = nx.piece;
        while (nx.valid && nx.piece == cur) nx.next(seq_off, p.B);
        if (nx.valid) q_prefetch(nx.b, nx.hg);
      }
      if (has2) it = itB;
      if (it.last)  // ---- piece end: out of line
        ok = piece_end<GRID>(p, cx, st, it.b, it.hg, it.pages, it.whole(), it.t % kNv, it.t, ok, sv_s,
                             vseq_off, cost_split, segs);
      it.next(seq_off, p.B);
    }
    if (!ok) fail();
  }

  tc_fence_before();
  __syncthreads();
  // ---------------------------------------------------------------- merges
  // M = max m_c, w_c = 2^(m_c - M), O = sV sum w_c o_c / sum w_c l_c.
  if (!GRID) {
    // LAST: the segments this CTA completed; the ring is idle now.  (The
    // loop's condition is read right after a block barrier, so every thread
    // sees the same abort flag.)
    int ncopy = 0;
    for (int di = 0; di < mi->nduty && !*abort_flag; ++di) {
      const int b = mi->duty[di][0], hg = mi->duty[di][1];
      const int seg_lo = mi->duty[di][2], seg_n = mi->duty[di][3];
      const int sigma = b * segs + hg;
      const int64_t base = static_cast<int64_t>(seg_lo) + sigma;
      const bool mok = guard(seg_lo >= 0 && seg_n >= 1 && seg_n <= p.P &&
                                 (base + seg_n) * kHT <= p.n_slots, p.status, 5);
      float* so = reinterpret_cast<float*>(smem + Lo::ring);          // [8][32][128]
      float2* sml = reinterpret_cast<float2*>(smem + Lo::pbuf);       // [seg_n][32]
      float* sw = reinterpret_cast<float*>(smem + Lo::pbuf + 16384);  // [seg_n][32]
      float* sL = reinterpret_cast<float*>(smem + Lo::qbuf);          // [32]
      // the pieces' o vectors come in 8 at a time (128 KB, the ring); their
      // (m, l) pairs and weights must fit the two P^T tiles
      constexpr int kChunk = static_cast<int>(Lo::ringBytes / (kHeads * kDH * 4));
      const bool staged = mok && seg_n * kHeads <= 2048;
      if (staged) {
        for (int i = tid; i < seg_n * kHeads; i += kThreadsB)
          sml[i] = __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + base * kHeads + i);
        __syncthreads();
        if (tid < kHeads) {  // head tid: maximum, weights and denominator over the pieces
          const int h = tid;
          float mx = -INFINITY;
          for (int k = 0; k < seg_n; ++k) mx = fmaxf(mx, sml[k * kHeads + h].x);
          float ls = 0.f;
          for (int k = 0; k < seg_n; ++k) {
            const float2 x = sml[k * kHeads + h];
            const float w = x.x == -INFINITY ? 0.f : fast_exp2(x.x - mx);
            sw[k * kHeads + h] = w;
            ls = fmaf(w, x.y, ls);
          }
          sL[h] = ls;
        }
        float acc[kHeads];
#pragma unroll
        for (int h = 0; h < kHeads; ++h) acc[h] = 0.f;
        bool cok = true;
        for (int k0 = 0; k0 < seg_n && cok; k0 += kChunk) {
          const int nk = seg_n - k0 < kChunk ? seg_n - k0 : kChunk;
          const uint32_t obytes = static_cast<uint32_t>(nk) * kHeads * kDH * 4;
          if (tid == 0) {
            mi->mcopy_s = static_cast<uint32_t>(ncopy + 1);
            mbar_arrive_expect_tx(mcopy, obytes);
            fence_proxy_async_global();  // the pieces were acquired through the counter
            const uint8_t* src =
                reinterpret_cast<const uint8_t*>(p.ws_o + (base + k0) * kHeads * kDH);
            for (uint32_t off = 0; off < obytes; off += 16384)
              bulk_load(reinterpret_cast<uint8_t*>(so) + off, src + off,
                        obytes - off < 16384 ? obytes - off : 16384, mcopy);
          }
          __syncthreads();  // (first chunk: the weights are written)
          cok = __syncthreads_and(mbar_wait(mcopy, static_cast<uint32_t>(ncopy & 1)) ? 1 : 0) != 0;
          ++ncopy;
          if (cok && tid < kSoftThreads) {
            const int d = tid;
#pragma unroll
            for (int h = 0; h < kHeads; ++h)
              for (int k = 0; k < nk; ++k)
                acc[h] = fmaf(sw[(k0 + k) * kHeads + h], so[(k * kHeads + h) * kDH + d], acc[h]);
          }
          __syncthreads();  // the staged pieces read before the next copy
        }
        if (!cok) {
          if (tid == 0) fail();
        } else if (tid < kSoftThreads) {
          const int d = tid;
          const int64_t obase = (static_cast<int64_t>(b) * p.Hq + hg * kHeads) * kDH + d;
#pragma unroll
          for (int h = 0; h < kHeads; ++h) {
            const float f = sL[h] > 0.f ? sv_s[hg * kHT + h / kGQ] / sL[h] : 0.f;
            const int64_t oi = obase + static_cast<int64_t>(h) * kDH;
            if (guard(oi >= 0 && oi < static_cast<int64_t>(p.B) * p.Hq * kDH, p.status, 3))
              p.out[oi] = static_cast<uint16_t>(f32x2_to_bf16x2(acc[h] * f, 0.f) & 0xFFFFu);
          }
        }
      } else if (mok && tid < kSoftThreads) {  // too many pieces to stage: from global memory
        const int d = tid;
        const int64_t obase = (static_cast<int64_t>(b) * p.Hq + hg * kHeads) * kDH + d;
        for (int h = 0; h < kHeads; ++h) {
          float M = -INFINITY, acc = 0.f, Lt = 0.f;
          for (int k = 0; k < seg_n; ++k) {
            const int64_t sl = base + k;
            const float2 x = __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + sl * kHeads + h);
            const float ov = __ldcg(p.ws_o + (sl * kHeads + h) * kDH + d);
            if (x.x == -INFINITY) continue;
            if (x.x > M) {
              const float sc = M == -INFINITY ? 0.f : fast_exp2(M - x.x);
              acc *= sc;
              Lt *= sc;
              M = x.x;
            }
            const float w = fast_exp2(x.x - M);
            acc = fmaf(w, ov, acc);
            Lt = fmaf(w, x.y, Lt);
          }
          const float f = Lt > 0.f ? sv_s[hg * kHT + h / kGQ] / Lt : 0.f;
          const int64_t oi = obase + static_cast<int64_t>(h) * kDH;
          if (guard(oi >= 0 && oi < static_cast<int64_t>(p.B) * p.Hq * kDH, p.status, 3))
            p.out[oi] = static_cast<uint16_t>(f32x2_to_bf16x2(acc * f, 0.f) & 0xFFFFu);
        }
      }
      if (tid == 0) p.ws_cnt[sigma] = 0u;
      __syncthreads();
    }
  } else {
    // GRID: every CTA has published its split pieces; meet all the others.
    uint32_t* arrive = p.ws_cnt + (kMaxSegments - 2);
    uint32_t* depart = p.ws_cnt + (kMaxSegments - 1);
    if (tid == 0) {
      __threadfence();
      atomicAdd(arrive, 1u);
      bool met = false;
      for (uint32_t i = 0; i < kMaxPolls; ++i) {
        if (ld_acquire_gpu(arrive) >= gridDim.x) {
          met = true;
          break;
        }
        __nanosleep(64);
      }
      if (!met) fail();
      __threadfence();
      if (atomicAdd(depart, 1u) + 1 == gridDim.x) {  // the last to leave resets both
        atomicExch(arrive, 0u);
        atomicExch(depart, 0u);
      }
    }
    __syncthreads();
    // The outputs of the split segments, sliced (segment, head, 32 dims) over
    // the CTAs.  Warp w reads pieces w, w + 7, ...; lane = dim.
    const bool aborted = *abort_flag != 0u;  // read by all after the barrier
    const int nseg = p.B * segs;
    const int G = static_cast<int>(gridDim.x);
    int item0 = 0;  // items of the segments before sigma
    for (int sigma = 0; sigma < nseg && !aborted; ++sigma) {
      const int b = sigma / segs, hg = sigma - b * segs;
      const int pages = (seq_off[b + 1] - seq_off[b]) / segs;
      if (pages == 0) continue;
      int seg_lo, seg_n;
      seg_ctas(b, hg, pages, seg_lo, seg_n);
      if (seg_n < 2) continue;
      const int nitems = kHeads * (kDH / 32);
      const int64_t base = static_cast<int64_t>(seg_lo) + sigma;
      const bool mok = guard(seg_lo >= 0 && seg_n <= p.P && (base + seg_n) * kHT <= p.n_slots,
                             p.status, 5);
      // this CTA's items: global indices c, c + G, ... (item0 + local index)
      for (int it = ((c - item0) % G + G) % G; mok && it < nitems; it += G) {
        const int h = it >> 2, d = (it & 3) * 32 + lane;
        float M = -INFINITY, acc = 0.f, Lt = 0.f;
        for (int k0 = warp; k0 < seg_n; k0 += kMergeWarps * kMergeBatch) {
          float2 x[kMergeBatch];
          float ov[kMergeBatch];
#pragma unroll
          for (int q = 0; q < kMergeBatch; ++q) {
            const int k = k0 + q * kMergeWarps;
            const int64_t sl = base + k;
            x[q] = k < seg_n ? __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + sl * kHeads + h)
                             : make_float2(-INFINITY, 0.f);
            ov[q] = k < seg_n ? __ldcg(p.ws_o + (sl * kHeads + h) * kDH + d) : 0.f;
          }
#pragma unroll
          for (int q = 0; q < kMergeBatch; ++q) {
            if (x[q].x == -INFINITY) continue;
            if (x[q].x > M) {
              const float sc = M == -INFINITY ? 0.f : fast_exp2(M - x[q].x);
              acc *= sc;
              Lt *= sc;
              M = x[q].x;
            }
            const float w = fast_exp2(x[q].x - M);
            acc = fmaf(w, ov[q], acc);
            Lt = fmaf(w, x[q].y, Lt);
          }
        }
        if (lane == 0) {
          mi->gm[warp] = M;
          mi->gl[warp] = Lt;
        }
        mi->gacc[warp][lane] = acc;
        __syncthreads();
        if (warp == 0) {
          float Mt = -INFINITY;
#pragma unroll
          for (int w = 0; w < kMergeWarps; ++w) Mt = fmaxf(Mt, mi->gm[w]);
          float a = 0.f, lt = 0.f;
#pragma unroll
          for (int w = 0; w < kMergeWarps; ++w) {
            const float wm = mi->gm[w];
            const float sc = wm == -INFINITY ? 0.f : fast_exp2(wm - Mt);
            a = fmaf(sc, mi->gacc[w][lane], a);
            lt = fmaf(sc, mi->gl[w], lt);
          }
          const float f = lt > 0.f ? sv_s[hg * kHT + h / kGQ] / lt : 0.f;
          const int64_t oi = (static_cast<int64_t>(b) * p.Hq + hg * kHeads + h) * kDH + d;
          if (guard(oi >= 0 && oi < static_cast<int64_t>(p.B) * p.Hq * kDH, p.status, 3))
            p.out[oi] = static_cast<uint16_t>(f32x2_to_bf16x2(a * f, 0.f) & 0xFFFFu);
        }
        __syncthreads();
      }
      item0 += nitems;
    }
  }

  __syncthreads();
  // After an abort: wait (bounded) for the copies still in flight (the MMA
  // lanes waited for their own), then free the tensor memory.
  if (*abort_flag && tid == 0) {
    for (int s = 0; s < kNk; ++s)
      if (mi->kiss[s] >= 0) mbar_wait(&kfull[s], static_cast<uint32_t>((mi->kiss[s] / kNk) & 1));
    for (int s = 0; s < kNv; ++s)
      if (mi->viss[s] >= 0) mbar_wait(&vfull[s], static_cast<uint32_t>((mi->viss[s] / kNv) & 1));
    if (mi->mcopy_s) mbar_wait(mcopy, (mi->mcopy_s - 1u) & 1u);
  }
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, Lo::kCols);
  }
}

}  // namespace dtb
}  // namespace kvq
