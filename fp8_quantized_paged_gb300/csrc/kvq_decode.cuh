// kvq_decode.cuh -- paged GQA decode attention with the dequantization fused in:
// the kernel and its launch, instantiated per cache format and head size by
// kvq_decode_variant.cu; the entry points are in kvq_decode.cu.
//
// "10.4 KV Cache quantization: INT8, KIVI 2-bit, FP8 KV", section 10.4.2:
// P = softmax(Q K^T / sqrt(dh) + mask), O = P V^, computed on the efficient
// path that reads the compressed KV, restores it in registers and feeds QK,
// PV and an online softmax directly; section 10.4.5: K^ = cast_float(K_fp8)
// * sK.  The scale sK is folded into the logit scale and sV is applied once to
// the normalised output, so the inner loop works on the raw codes.
//
// Work decomposition (one GPU, persistent grid)
//   A unit of work is one KV-head page: block_size = 16 tokens of K and of V
//   for one (sequence b, KV head g).  Units are numbered sequence by
//   sequence, head by head, page by page; CTA c of P takes the contiguous
//   range [floor(c W / P), floor((c+1) W / P)) of the W units, so every CTA
//   streams the same number of bytes whatever the length mix.  A range cut
//   through a (b, g) segment leaves partial softmax states (m, l, o) in the
//   workspace; the CTA that completes a segment's last piece merges them.
//   A segment held by one CTA is written directly.
//
// Inside a CTA
//   warp 4 (producer): one lane issues TMA tile loads of the K page and the V
//   page of each unit into a ring of shared-memory stages (128-byte swizzle,
//   mbarrier completion); the block ids of the next 32 units are fetched by
//   the 32 lanes ahead of use.
//   warps 0-3 (consumers): take the pages of the current segment round-robin.
//   Per page: the K tile is an m16n8k16 A operand (16 tokens x 16 dims),
//   converted FP8 -> f16 in registers (exact), against the G <= 8 query heads
//   of the group as the B operand; the logits feed a warp online softmax; P
//   (split into f16 hi + lo parts, ~22-bit weights) and the V tile (converted
//   the same way, transposed with byte permutes) give O^T += V^T P^T.  The
//   bf16 cache mode feeds the bf16 tiles to bf16 MMAs unchanged.
//   Segment end: the four warps' states merge in shared memory.
#pragma once

#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>

#include "kvq_common.cuh"
#include "kvq_host.h"

namespace kvq {

#ifndef KVQ_CONSUMER_WARPS
#define KVQ_CONSUMER_WARPS 4
#endif
#ifndef KVQ_CTAS_PER_SM
#define KVQ_CTAS_PER_SM 2
#endif
#ifndef KVQ_RING_KB
#define KVQ_RING_KB 80
#endif
// CTAs per SM of the tensor-core decode (kvq_decode_tc.cuh)
#ifndef KVQ_DTC_CTAS_PER_SM
#define KVQ_DTC_CTAS_PER_SM 1
#endif

constexpr int kBS = 16;  // tokens per page (block_size)
constexpr int kConsumerWarps = KVQ_CONSUMER_WARPS;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kCtasPerSM = KVQ_CTAS_PER_SM;
constexpr int kRingBytes = KVQ_RING_KB * 1024;
constexpr int kMaxSeqs = 4096;
constexpr int kMaxGroup = 8;
constexpr int kMaxKvHeads = 256;
constexpr int kMaxSegments = 65536;  // num_seqs * num_kv_heads (counter table entries)
constexpr int kMaxHT = 8;  // KV heads one tile of the whole-block decode covers
constexpr float kRescaleThreshold = 8.0f;  // log2 units: lazily rescale O
#ifndef KVQ_PIECE_COST
#define KVQ_PIECE_COST 16
#endif
// Fixed cost of one piece (its setup, the warps' combine and the publication
// of its state) counted in pages when the units are split among the CTAs.
constexpr int kPieceCost = KVQ_PIECE_COST;
constexpr uint32_t kFull = 0xFFFFFFFFu;

// atomicAdd with acquire-release semantics at GPU scope (one instruction in
// place of a fence, the add and a second fence).
KVQ_DEVI uint32_t atom_add_acq_rel_gpu(uint32_t* addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}

template <int FMT, int DH>
struct Cfg {
  static constexpr int kElem = (FMT == KVQ_FMT_BF16) ? 2 : 1;
  static constexpr int kRow = DH * kElem;         // bytes of one token row
  static constexpr int kPage = kBS * kRow;        // bytes of one tensor's page
  static constexpr int kSlot = 2 * kPage;         // K page + V page
  // A multiple of the consumer-warp count: position pos of the CTA's page
  // stream goes to warp pos % 4 and slot pos % kStages, so every slot is
  // used by one warp only, in order, and a parity wait can never alias a
  // phase two behind.
  static constexpr int kStagesFit =
      kConsumerWarps * (kRingBytes / (kConsumerWarps * kSlot) > 0 ? kRingBytes / (kConsumerWarps * kSlot) : 1);
  // at most 64 (two ring slots per producer lane; a multiple of the warp count)
  static constexpr int kStages = kStagesFit < 64 ? kStagesFit : 64 - 64 % kConsumerWarps;
  static constexpr uint32_t kSwz = (kRow >= 128) ? 7u : 3u;  // 128B or 64B swizzle
  // Pages a consumer warp works on at once.  Two (independent MMA chains)
  // measured slower: each warp then holds two ring slots before it starts.
  static constexpr int kPagesPerStep = 1;
};

// Dynamic shared memory of the decode kernel (offsets from a 1024-aligned
// base): the ring and barriers at fixed offsets, then the merge scratch (the
// warps' states for the group's G heads, reused for the weights of up to P
// pieces when a split segment is merged), the plan ([B+1] unit offsets, [B]
// checked lengths, [B+1] cost offsets) and the k/v scales.
template <int FMT, int DH, bool TS = false>
struct SmemLayout {
  using C = Cfg<FMT, DH>;
  static constexpr int S = C::kStages;
  static constexpr size_t ring = 0;
  // per-(token, head) scales of each staged page (TS only): [S][K 16, V 16] fp32
  static constexpr size_t tsc = ring + static_cast<size_t>(S) * C::kSlot;
  // full[S], empty[S], and the barrier of the segment-merge bulk copy
  static constexpr size_t bars = tsc + (TS ? static_cast<size_t>(S) * 128 : 0);
  // bad[S], abort, merge decision, tot[8], last[S], merge copy issued, u0, u1
  static constexpr size_t flags = bars + (2 * S + 1) * sizeof(uint64_t);
  static constexpr size_t comb = (flags + (2 * S + 5 + 8) * sizeof(uint32_t) + 15) & ~size_t(15);
  __host__ __device__ static size_t comb_floats(int G, int P) {
    const size_t warps = static_cast<size_t>(kConsumerWarps) * G * (DH + 2);
    const size_t pieces = (static_cast<size_t>(P) + 1) * G;
    return warps > pieces ? warps : pieces;
  }
  __host__ __device__ static size_t seq(int G, int P) {
    return comb + ((comb_floats(G, P) * sizeof(float) + 15) & ~size_t(15));
  }
  __host__ __device__ static size_t scales(int G, int P, int B) {
    return seq(G, P) + (3 * static_cast<size_t>(B) + 2) * sizeof(int32_t);
  }
  __host__ __device__ static size_t total(int G, int P, int B, int Hkv) {
    return scales(G, P, B) + 2 * static_cast<size_t>(Hkv) * sizeof(float) + 1024;
  }
};

struct DecodeParams {
  const uint16_t* q;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  int max_blocks;
  int B, Hq, Hkv, G;
  int window;
  int64_t num_blocks;
  const float* ks;  // [1], [Hkv], or the scale caches [num_blocks][Hkv][16] (ts)
  const float* vs;
  int per_head;
  int ts;  // per-(token, KV head) scales
  int P;
  int early;  // KVQ_CACHE_READY: tables, lengths, scales and all but the last pages before the wait
  const float* qs;  // KVQ_Q_FP8: query scales, [1] or [Hq]
  int q_per_head;
  float logit_scale;  // log2(e) / sqrt(dh)
  uint32_t* ws_cnt;  // [B * Hkv] arrivals of the pieces of each segment (zero between calls)
  float* ws_ml;
  float* ws_o;
  uint16_t* out;
  uint32_t* status;
  int64_t rows;     // rows of the cache tensor maps (num_blocks * Hkv * 16)
  int64_t n_slots;  // partial slots in the workspace
  int clu;          // tensor-core decode: CTAs per cluster of the per-segment variant (0: split)
  int ncl;          // whole-block decode, cluster variant: clusters per segment
  int withhold;     // test builds (KVQ_TEST_HOOKS) only: CTA 0 never copies its page at this
                    // stream position, so the wait for it runs out; -1 otherwise
};

// Workspace: a table of kMaxSegments uint32 arrival counters, one per
// (sequence, KV head) segment (zero before the first call, left zero by
// every completed call), then per partial slot the (m, l) pairs
// and o vectors for the G heads of a group.  The partial slot of the piece of
// segment sigma = b * Hkv + g held by CTA c is c + sigma (unique: CTA ranges
// are ordered).
struct WsLayout {
  size_t cnt, ml, o, total;
};

inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(int B, int G, int Hkv, int DH, int P) {
  WsLayout w;
  // partial slots in units of one KV head's G query heads: a piece of the
  // whole-block decode carries 8 KV heads
  const size_t slots = static_cast<size_t>(kMaxHT) * P + static_cast<size_t>(B) * Hkv;
  w.cnt = 0;  // a fixed-size table, so every batch shape reuses the same zeroed counters
  w.ml = round256(sizeof(uint32_t) * static_cast<size_t>(kMaxSegments));
  w.o = w.ml + round256(slots * G * 2 * sizeof(float));
  w.total = w.o + round256(slots * G * DH * sizeof(float));
  return w;
}

KVQ_DEVI uint32_t swz(uint32_t logical, uint32_t mask) {
  return logical ^ (((logical >> 7) & mask) << 4);
}

// Byte b of token row r inside one staged page.  Rows of at most 128 bytes are
// stored row after row; a 256-byte bf16 row (dh = 128) is staged as two
// 16-row sub-tiles of 128-byte half rows, one TMA box each.
template <int ROW>
KVQ_DEVI uint32_t page_off(int r, int b) {
  if (ROW > 128) return static_cast<uint32_t>((b >> 7) * (16 * 128) + r * 128 + (b & 127));
  return static_cast<uint32_t>(r * ROW + b);
}

KVQ_DEVI uint4 lds128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}

KVQ_DEVI uint2 lds64(uint32_t addr) {
  uint2 r;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(addr));
  return r;
}

KVQ_DEVI void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}


KVQ_DEVI int window_lo(int window, int L) { return (window > 0 && L > window) ? L - window : 0; }
KVQ_DEVI int window_lo(const DecodeParams& p, int L) { return window_lo(p.window, L); }

// Last b with seq_off[b] <= u (seq_off non-decreasing, seq_off[B] > u).
KVQ_DEVI int find_seq(const int32_t* seq_off, int B, int64_t u) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seq_off[mid] <= u)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Exclusive scans of the per-sequence unit counts into seq_off[0..B] and of
// the costs into vseq_off[0..B], the checked length of every sequence into
// len_s[0..B), and the k/v scales of the KV heads into sk_s / sv_s
// (per-tensor scales replicated).
KVQ_DEVI int first_page_of(const DecodeParams& p, int L) { return window_lo(p, L) / kBS; }

// Pages sequence b attends to (0 for an empty or invalid length), the unit
// count of the partition being pages * Hkv.
KVQ_DEVI int seq_pages(int raw_len, int max_blocks, int window) {
  const int L = (raw_len < 0 || raw_len > max_blocks * kBS) ? 0 : raw_len;
  return L > 0 ? (L + kBS - 1) / kBS - window_lo(window, L) / kBS : 0;
}

// The split of the units among the CTAs balances cost, not units: segment
// (b, g) costs kPieceCost + pages_b, laid out as kPieceCost cost units
// followed by its pages, sequence after sequence, head after head
// (vseq_off[b] is the cost before sequence b, seq_off[b] the pages).  CTA c
// takes the cost range [floor(c V / Pe), floor((c + 1) V / Pe)) of the total
// V, i.e. the pages between the page counts at those two cost positions, so
// a CTA of many short segments gets fewer pages.
// Pages before cost position v (0 <= v <= V).
// All offsets stay below 2^31 (checked on the host), so 32-bit division does.
// pc: the fixed cost of a piece (kPieceCost unless the kernel says otherwise).
KVQ_DEVI int pages_before(const int32_t* seq_off, const int32_t* vseq_off, int B, int Hkv, int v,
                          int pc = kPieceCost) {
  if (v >= vseq_off[B]) return seq_off[B];
  const int b = find_seq(vseq_off, B, v);
  const int pages = (seq_off[b + 1] - seq_off[b]) / Hkv;
  const int r = v - vseq_off[b];
  const int g = r / (pages + pc);
  const int in = r - g * (pages + pc) - pc;  // < 0: in the fixed cost
  return seq_off[b] + g * pages + (in < 0 ? 0 : (in > pages ? pages : in));
}

// Cost position where CTA c's range starts, floor(c V / Pe), for
// 0 <= c <= Pe < 2^15 and V < 2^31, in 32-bit integers: with V = a Pe + r,
// c V / Pe = c a + c r / Pe and c r < Pe^2.
struct CostSplit {
  int V, a, r, Pe;
  KVQ_DEVI CostSplit(int V_, int Pe_)
      : V(V_), a(Pe_ > 0 ? V_ / Pe_ : 0), r(Pe_ > 0 ? V_ % Pe_ : 0), Pe(Pe_) {}
  KVQ_DEVI int operator()(int c) const { return c * a + (c * r) / Pe; }
  // The CTA whose cost range holds cost position v (0 <= v < V, Pe > 0): a
  // binary32 estimate of ceil((v + 1) Pe / V) - 1, off by at most one, then
  // corrected against the exact range starts.
  KVQ_DEVI int cta_of(int v) const {
    int cc = static_cast<int>(static_cast<float>(v + 1) * static_cast<float>(Pe) / static_cast<float>(V));
    cc = cc < 0 ? 0 : (cc > Pe - 1 ? Pe - 1 : cc);
    for (int i = 0; i < 3 && cc > 0 && (*this)(cc) > v; ++i) --cc;
    for (int i = 0; i < 3 && cc + 1 < Pe && (*this)(cc + 1) <= v; ++i) ++cc;
    return cc;
  }
};



// segs: segments per sequence (the KV heads, or groups of them that one
// unit covers together); pc: the fixed cost of a piece in units.
template <bool SCALED, int NT = kThreads>
KVQ_DEVI void build_plan(const DecodeParams& p, int32_t* seq_off, int32_t* len_s,
                         int32_t* vseq_off, float* sk_s, float* sv_s, int32_t* warp_tot,
                         int segs = -1, int pc = kPieceCost) {
  if (segs < 0) segs = p.Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int h = tid; h < p.Hkv; h += NT) {
    sk_s[h] = SCALED ? p.ks[p.per_head ? h : 0] : 1.f;
    sv_s[h] = SCALED ? p.vs[p.per_head ? h : 0] : 1.f;
  }
  const int per = (p.B + NT - 1) / NT;
  const int b0 = tid * per, b1 = min(p.B, b0 + per);
  int local = 0, vlocal = 0;
  for (int b = b0; b < b1; ++b) {
    const int raw = p.seq_lens[b];
    if ((raw < 0 || raw > p.max_blocks * kBS) && blockIdx.x == 0)
      flag_status(p.status, KVQ_DEV_BAD_SEQLEN);
    const int L = (raw < 0 || raw > p.max_blocks * kBS) ? 0 : raw;
    const int pages = seq_pages(raw, p.max_blocks, p.window);
    len_s[b] = L;
    seq_off[b] = local;
    vseq_off[b] = vlocal;
    local += pages * segs;
    vlocal += pages > 0 ? (pages + pc) * segs : 0;
  }
  auto scan = [&](int v, int& total) {  // block-wide exclusive scan
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int base = 0;
    total = 0;
    for (int w = 0; w < NT / 32; ++w) {
      base += w < warp ? warp_tot[w] : 0;
      total += warp_tot[w];
    }
    __syncthreads();
    return base + incl - v;
  };
  int total, vtotal;
  const int excl = scan(local, total);
  const int vexcl = scan(vlocal, vtotal);
  for (int b = b0; b < b1; ++b) {
    seq_off[b] += excl;
    vseq_off[b] += vexcl;
  }
  if (tid == 0) {
    seq_off[p.B] = total;
    vseq_off[p.B] = vtotal;
  }
  __syncthreads();
}

// Bounded mbarrier wait that also gives up when another warp has aborted.
KVQ_DEVI bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  for (uint32_t i = 0; i < kMaxPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u && *abort_flag) return false;
  }
  return false;
}

// --------------------------------------------------------------------------
// One page of one consumer warp
// --------------------------------------------------------------------------

struct SoftmaxState {
  float m[2];  // running max (log2 units) of heads 2t, 2t+1; warp-uniform per t
  float l[2];  // per-lane partial denominators
};

// Online softmax update of NP 16-token pages.  x[4i .. 4i+3] hold page i's
// log2-domain logits of (token g, head 2t), (token g, head 2t+1),
// (token g+8, head 2t), (token g+8, head 2t+1).  Returns the probabilities
// in pr; rescales o (lazily: only when the running max grows by more than
// kRescaleThreshold, so p <= 2^8 and the exact max is rarely reduced).
template <int NP, int MT>
KVQ_DEVI void softmax_pages(const float (&x)[4 * NP], float (&pr)[4 * NP], SoftmaxState& st,
                            float (&o)[MT][4]) {
  const float ninf = -INFINITY;
  float lm0 = ninf, lm1 = ninf;
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    lm0 = fmaxf(lm0, fmaxf(x[4 * i], x[4 * i + 2]));
    lm1 = fmaxf(lm1, fmaxf(x[4 * i + 1], x[4 * i + 3]));
  }
  const bool need = (lm0 > st.m[0] + kRescaleThreshold) || (lm1 > st.m[1] + kRescaleThreshold);
  if (__any_sync(kFull, need)) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      lm0 = fmaxf(lm0, __shfl_xor_sync(kFull, lm0, off));
      lm1 = fmaxf(lm1, __shfl_xor_sync(kFull, lm1, off));
    }
    const float n0 = fmaxf(st.m[0], lm0), n1 = fmaxf(st.m[1], lm1);
    const float a0 = (n0 == ninf) ? 1.f : fast_exp2(st.m[0] - n0);
    const float a1 = (n1 == ninf) ? 1.f : fast_exp2(st.m[1] - n1);
    st.l[0] *= a0;
    st.l[1] *= a1;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      o[mt][0] *= a0;
      o[mt][2] *= a0;
      o[mt][1] *= a1;
      o[mt][3] *= a1;
    }
    st.m[0] = n0;
    st.m[1] = n1;
  }
#pragma unroll
  for (int i = 0; i < 4 * NP; ++i) {
    const float m = (i & 1) ? st.m[1] : st.m[0];
    pr[i] = (x[i] == ninf) ? 0.f : fast_exp2(x[i] - m);
  }
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    st.l[0] += pr[4 * i] + pr[4 * i + 2];
    st.l[1] += pr[4 * i + 1] + pr[4 * i + 3];
  }
}

// P^T as the B operand of the PV MMA (k = token, n = head), split into a high
// and a low 16-bit part.  PV uses the token order k -> {2t: 2t, 2t+1: 2t+8,
// 2t+8: 2t+1, 2t+9: 2t+9} so that a lane's two k values of a register come
// from one source lane's (token g', token g'+8) pair.
template <bool BF16P>
KVQ_DEVI void p_fragments(const float* pr, int g, int t, int G, uint32_t (&bh)[2],
                          uint32_t (&bl)[2]) {
  uint32_t h0, h1, l0, l1;
  if (BF16P) {
    h0 = f32x2_to_bf16x2(pr[0], pr[2]);
    h1 = f32x2_to_bf16x2(pr[1], pr[3]);
    l0 = f32x2_to_bf16x2(pr[0] - bf16lo_to_f32(h0), pr[2] - bf16hi_to_f32(h0));
    l1 = f32x2_to_bf16x2(pr[1] - bf16lo_to_f32(h1), pr[3] - bf16hi_to_f32(h1));
  } else {
    h0 = f32x2_to_f16x2(pr[0], pr[2]);
    h1 = f32x2_to_f16x2(pr[1], pr[3]);
    l0 = f32x2_to_f16x2(pr[0] - f16lo_to_f32(h0), pr[2] - f16hi_to_f32(h0));
    l1 = f32x2_to_f16x2(pr[1] - f16lo_to_f32(h1), pr[3] - f16hi_to_f32(h1));
  }
  const int srcA = (2 * t) * 4 + (g >> 1), srcB = (2 * t + 1) * 4 + (g >> 1);
  const bool odd = g & 1;
  const uint32_t ha0 = __shfl_sync(kFull, h0, srcA), ha1 = __shfl_sync(kFull, h1, srcA);
  const uint32_t hb0 = __shfl_sync(kFull, h0, srcB), hb1 = __shfl_sync(kFull, h1, srcB);
  const uint32_t la0 = __shfl_sync(kFull, l0, srcA), la1 = __shfl_sync(kFull, l1, srcA);
  const uint32_t lb0 = __shfl_sync(kFull, l0, srcB), lb1 = __shfl_sync(kFull, l1, srcB);
  const bool live = g < G;
  bh[0] = live ? (odd ? ha1 : ha0) : 0u;
  bh[1] = live ? (odd ? hb1 : hb0) : 0u;
  bl[0] = live ? (odd ? la1 : la0) : 0u;
  bl[1] = live ? (odd ? lb1 : lb0) : 0u;
}

// Packed variant for groups of at most 4 heads: the PV MMA's 8 columns hold
// P_hi of heads 0..3 (columns 0..3) and P_lo of heads 0..3 (columns 4..7), so
// one MMA per m-tile accumulates both parts (summed once per piece).  Q is
// replicated into columns 4..7 of the QK MMA, so lane (g, t) with t >= 2 holds
// the same probabilities as lane (g, t - 2) and supplies the lo parts: each
// destination needs one source lane per token pair (2 shuffles each).
template <bool BF16P>
KVQ_DEVI void p_fragments_packed(const float* pr, int g, int t, int G, uint32_t (&b)[2]) {
  const bool lo_src = t >= 2;
  uint32_t pk0, pk1;
  if (BF16P) {
    const uint32_t h0 = f32x2_to_bf16x2(pr[0], pr[2]), h1 = f32x2_to_bf16x2(pr[1], pr[3]);
    pk0 = lo_src ? f32x2_to_bf16x2(pr[0] - bf16lo_to_f32(h0), pr[2] - bf16hi_to_f32(h0)) : h0;
    pk1 = lo_src ? f32x2_to_bf16x2(pr[1] - bf16lo_to_f32(h1), pr[3] - bf16hi_to_f32(h1)) : h1;
  } else {
    const uint32_t h0 = f32x2_to_f16x2(pr[0], pr[2]), h1 = f32x2_to_f16x2(pr[1], pr[3]);
    pk0 = lo_src ? f32x2_to_f16x2(pr[0] - f16lo_to_f32(h0), pr[2] - f16hi_to_f32(h0)) : h0;
    pk1 = lo_src ? f32x2_to_f16x2(pr[1] - f16lo_to_f32(h1), pr[3] - f16hi_to_f32(h1)) : h1;
  }
  const int hh = g & 3;                            // head of this lane's B column
  const int src = ((hh >> 1) + ((g >> 2) << 1));   // source lane's t: hi (g < 4) or lo part
  const int srcA = (2 * t) * 4 + src, srcB = (2 * t + 1) * 4 + src;
  const uint32_t a0 = __shfl_sync(kFull, pk0, srcA), a1 = __shfl_sync(kFull, pk1, srcA);
  const uint32_t b0 = __shfl_sync(kFull, pk0, srcB), b1 = __shfl_sync(kFull, pk1, srcB);
  const bool live = hh < G, odd = hh & 1;
  b[0] = live ? (odd ? a1 : a0) : 0u;
  b[1] = live ? (odd ? b1 : b0) : 0u;
}

KVQ_DEVI bool token_valid(int tok, int lo, int L, bool bad) { return !bad && tok >= lo && tok < L; }


// Register image of one staged page: the lane's K fragment words (token rows
// g and g+8) and V fragment words (tokens 2t, 2t+8, 2t+1, 2t+9).  Reading the
// page into registers first lets the ring slot go back to the producer
// before the math, so slots are held only while their data is in flight.
template <int FMT, int DH>
struct PageRegs {
  using C = Cfg<FMT, DH>;
  static constexpr int KB = C::kRow / 4;  // bytes of one K row a lane reads
  static constexpr int VB = C::kRow / 8;  // bytes of one V row a lane reads
  uint32_t k0[KB / 4], k1[KB / 4];
  uint32_t v[4][VB / 4];
};

template <int FMT, int DH>
KVQ_DEVI void load_page(uint32_t kp, uint32_t vp, int g, int t, int tok0, int lo, int L,
                        bool bad, PageRegs<FMT, DH>& r) {
  using C = Cfg<FMT, DH>;
  using R = PageRegs<FMT, DH>;
#pragma unroll
  for (int c = 0; c < R::KB / 16; ++c) {
    const int off = t * R::KB + c * 16;
    const uint4 a = lds128(kp + swz(page_off<C::kRow>(g, off), C::kSwz));
    const uint4 b = lds128(kp + swz(page_off<C::kRow>(g + 8, off), C::kSwz));
    r.k0[4 * c] = a.x; r.k0[4 * c + 1] = a.y; r.k0[4 * c + 2] = a.z; r.k0[4 * c + 3] = a.w;
    r.k1[4 * c] = b.x; r.k1[4 * c + 1] = b.y; r.k1[4 * c + 2] = b.z; r.k1[4 * c + 3] = b.w;
  }
  const int rows[4] = {2 * t, 2 * t + 8, 2 * t + 1, 2 * t + 9};
  const bool edge = bad || tok0 < lo || tok0 + kBS > L;  // warp-uniform
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (R::VB >= 16) {
#pragma unroll
      for (int c = 0; c < R::VB / 16; ++c) {
        const uint4 v = lds128(vp + swz(page_off<C::kRow>(rows[q], g * R::VB + c * 16), C::kSwz));
        r.v[q][4 * c] = v.x; r.v[q][4 * c + 1] = v.y; r.v[q][4 * c + 2] = v.z; r.v[q][4 * c + 3] = v.w;
      }
    } else {
      const uint2 v = lds64(vp + swz(page_off<C::kRow>(rows[q], g * R::VB), C::kSwz));
      r.v[q][0] = v.x;
      r.v[q][1] = v.y;
    }
    // a masked token's V row may hold anything (p = 0 would not clear a NaN)
    if (edge && !token_valid(tok0 + rows[q], lo, L, bad)) {
#pragma unroll
      for (int w = 0; w < R::VB / 4; ++w) r.v[q][w] = 0u;
    }
  }
}

// QK^T, online softmax and PV of NP pages held in registers (the pages'
// MMA chains are independent, which hides their latency).
//   QK: the K tile is the m16n8k16 A operand (16 tokens x 16 dims; FP8 codes
//   converted to f16 exactly, or bf16 as is), the group's query heads the B
//   operand; lane (g, t) covers dims t*(DH/4) + 4kk + {0..3} of step kk.
//   PV: O^T += V^T P^T with m-tile mt, row r -> dim g*(DH/8) + 2mt + r/8.
//   TS (per-(token, head) scales): sK of token rows g, g+8 multiplies the
//   logits; the probabilities that weight V carry sV_t / sigma (sigma the
//   page's largest sV, so they stay <= 2^8 in f16), the page's PV goes to a
//   fresh accumulator added to O times sigma; the denominator sums plain p.
template <int FMT, int DH, int NP, bool PK, bool QF8, bool TS>
KVQ_DEVI void compute_pages(const PageRegs<FMT, DH> (&r)[NP], const int (&tok0)[NP],
                            const bool (&bad)[NP], int g, int t, int G,
                            const uint32_t (&qb)[DH / 16][2], float (&o)[DH / 16][4],
                            SoftmaxState& st, float lscale0, float lscale1, int lo, int L,
                            const float (&tsk)[NP][2], const float (&tsv)[NP][2]) {
  using R = PageRegs<FMT, DH>;
  constexpr bool BF = FMT == KVQ_FMT_BF16;
  static_assert(!TS || NP == 1, "per-token scales take one page per step");
  // QK^T as two independent MMA chains (even and odd k-steps), summed at
  // the end: half the dependent latency per page
  float s[NP][4], s2[NP][4];
#pragma unroll
  for (int i = 0; i < NP; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) s[i][j] = s2[i][j] = 0.f;
#pragma unroll
  for (int kk = 0; kk < (QF8 ? DH / 32 : DH / 16); ++kk) {
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      uint32_t a[4];
      if (QF8) {  // the FP8 codes themselves: dims 8kk .. 8kk + 7 of the lane's run
        a[0] = r[i].k0[2 * kk]; a[1] = r[i].k1[2 * kk];
        a[2] = r[i].k0[2 * kk + 1]; a[3] = r[i].k1[2 * kk + 1];
        mma_fp8<FMT>((kk & 1) ? s2[i] : s[i], a, qb[kk][0], qb[kk][1]);
      } else if (BF) {
        a[0] = r[i].k0[2 * kk]; a[1] = r[i].k1[2 * kk];
        a[2] = r[i].k0[2 * kk + 1]; a[3] = r[i].k1[2 * kk + 1];
        mma_bf16((kk & 1) ? s2[i] : s[i], a, qb[kk][0], qb[kk][1]);
      } else {
        fp8x4_to_f16x2x2<FMT>(r[i].k0[kk], a[0], a[2]);
        fp8x4_to_f16x2x2<FMT>(r[i].k1[kk], a[1], a[3]);
        mma_f16((kk & 1) ? s2[i] : s[i], a, qb[kk][0], qb[kk][1]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NP; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) s[i][j] += s2[i][j];
  float x[4 * NP];
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const int ta = tok0[i] + g, tb = ta + 8;
    const bool va = token_valid(ta, lo, L, bad[i]), vb = token_valid(tb, lo, L, bad[i]);
    const float ka = TS ? tsk[i][0] : 1.f, kb = TS ? tsk[i][1] : 1.f;
    x[4 * i] = va ? s[i][0] * lscale0 * ka : -INFINITY;
    x[4 * i + 1] = va ? s[i][1] * lscale1 * ka : -INFINITY;
    x[4 * i + 2] = vb ? s[i][2] * lscale0 * kb : -INFINITY;
    x[4 * i + 3] = vb ? s[i][3] * lscale1 * kb : -INFINITY;
  }
  float pr[4 * NP];
  softmax_pages<NP, DH / 16>(x, pr, st, o);
  float sigma[NP];
  if (TS) {  // V weights p sV_t / sigma
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int ta = tok0[i] + g;
      const float a = token_valid(ta, lo, L, bad[i]) ? tsv[i][0] : 0.f;
      const float b = token_valid(ta + 8, lo, L, bad[i]) ? tsv[i][1] : 0.f;
      float m = fmaxf(a, b);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
      sigma[i] = m;
      const float inv = m > 0.f ? __frcp_rn(m) : 0.f;
      const float ra = a * inv, rb = b * inv;
      pr[4 * i] *= ra;
      pr[4 * i + 1] *= ra;
      pr[4 * i + 2] *= rb;
      pr[4 * i + 3] *= rb;
    }
  }
  uint32_t bh[NP][2], bl[NP][2];
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    if (PK)
      p_fragments_packed<BF>(pr + 4 * i, g, t, G, bh[i]);
    else
      p_fragments<BF>(pr + 4 * i, g, t, G, bh[i], bl[i]);
  }
  float ot[DH / 16][4];  // the page's PV (TS), added to O times sigma
  if (TS) {
#pragma unroll
    for (int mt = 0; mt < DH / 16; ++mt) ot[mt][0] = ot[mt][1] = ot[mt][2] = ot[mt][3] = 0.f;
  }
  float (&acc)[DH / 16][4] = TS ? ot : o;

#pragma unroll
  for (int w = 0; w < R::VB / 4; ++w) {
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const uint32_t* v0 = r[i].v[0];
      const uint32_t* v1 = r[i].v[1];
      const uint32_t* v2 = r[i].v[2];
      const uint32_t* v3 = r[i].v[3];
      if (BF) {  // word w = dims g*(DH/8) + 2w, +1 -> m-tile w, rows g (lo) and g+8 (hi)
        const uint32_t a[4] = {prmt(v0[w], v1[w], 0x5410u), prmt(v0[w], v1[w], 0x7632u),
                               prmt(v2[w], v3[w], 0x5410u), prmt(v2[w], v3[w], 0x7632u)};
        mma_bf16(acc[w], a, bh[i][0], bh[i][1]);
        if (!PK) mma_bf16(acc[w], a, bl[i][0], bl[i][1]);
      } else {  // word w = dims g*(DH/8) + 4w .. +3 -> m-tiles 2w, 2w+1
        const uint32_t x0 = prmt(v0[w], v1[w], 0x5140u), y0 = prmt(v0[w], v1[w], 0x7362u);
        const uint32_t z0 = prmt(v2[w], v3[w], 0x5140u), u0 = prmt(v2[w], v3[w], 0x7362u);
        uint32_t a[4], c[4];
        fp8x4_to_f16x2x2<FMT>(x0, a[0], a[1]);
        fp8x4_to_f16x2x2<FMT>(z0, a[2], a[3]);
        fp8x4_to_f16x2x2<FMT>(y0, c[0], c[1]);
        fp8x4_to_f16x2x2<FMT>(u0, c[2], c[3]);
        mma_f16(acc[2 * w], a, bh[i][0], bh[i][1]);
        mma_f16(acc[2 * w + 1], c, bh[i][0], bh[i][1]);
        if (!PK) {
          mma_f16(acc[2 * w], a, bl[i][0], bl[i][1]);
          mma_f16(acc[2 * w + 1], c, bl[i][0], bl[i][1]);
        }
      }
    }
  }
  if (TS) {
#pragma unroll
    for (int mt = 0; mt < DH / 16; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j) o[mt][j] = fmaf(sigma[0], ot[mt][j], o[mt][j]);
  }
}

// Q of head g (lane row) of the group, dims t*(DH/4) + 4kk + {0..3}: the
// raw bf16 words (issued a piece ahead), then the B operand of the QK MMA:
// f16 for the FP8 caches (exact for |q| in the f16 normal range), the bf16
// bits for the bf16 cache.  Rows past the group (g >= G) are zero.
template <int DH>
KVQ_DEVI void load_q_raw(const DecodeParams& p, int b, int gkv, int hq, int t,
                         uint32_t (&w)[DH / 8]) {
  const int64_t qrow = static_cast<int64_t>(b) * p.Hq + gkv * p.G + hq;
  const bool ok = hq < p.G && guard(b >= 0 && b < p.B && qrow < static_cast<int64_t>(p.B) * p.Hq,
                                    p.status, 2);
  const uint4* src = reinterpret_cast<const uint4*>(p.q + (ok ? qrow : 0) * DH + t * (DH / 4));
#pragma unroll
  for (int i = 0; i < DH / 32; ++i) {
    const uint4 v = ok ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
    w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
  }
}

// For the FP8 caches the f16 operand is the query times a per-head power of
// two 2^a (a returned; the four lanes of a head agree) that puts the head's
// largest |q| in [2^14, 2^15): exact, and every bf16 query fits f16's range
// (elements below 2^-38 of the head's largest lose bits as f16 subnormals).
// The caller folds 2^-a into the head's logit scale.
template <int FMT, int DH>
KVQ_DEVI int q_fragments(const uint32_t (&w)[DH / 8], uint32_t (&qb)[DH / 16][2]) {
  if (FMT == KVQ_FMT_BF16) {
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk) {
      qb[kk][0] = w[2 * kk];
      qb[kk][1] = w[2 * kk + 1];
    }
    return 0;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < DH / 8; ++i)
    amax = fmaxf(amax, fmaxf(fabsf(bf16lo_to_f32(w[i])), fabsf(bf16hi_to_f32(w[i]))));
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));  // the head's 4 lanes (t = 0..3)
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
  int a = 0;
  if (amax > 0.f) {  // finite bf16: exponent field 0 .. 254
    a = 14 - (static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127);
    a = a > 126 ? 126 : (a < -126 ? -126 : a);
  }
  const float sc = __int_as_float((a + 127) << 23);
#pragma unroll
  for (int kk = 0; kk < DH / 16; ++kk) {
    qb[kk][0] = f32x2_to_f16x2(bf16lo_to_f32(w[2 * kk]) * sc, bf16hi_to_f32(w[2 * kk]) * sc);
    qb[kk][1] = f32x2_to_f16x2(bf16lo_to_f32(w[2 * kk + 1]) * sc, bf16hi_to_f32(w[2 * kk + 1]) * sc);
  }
  return a;
}

// Q of the FP8-domain mode: the lane's DH/4 query values divided by the
// head's scale (binary32, round to nearest even) and encoded to the cache's
// FP8 format (RNE, satfinite), four codes a word in dim order; MMA step kk
// takes words 2kk and 2kk + 1 (dims 8kk .. 8kk + 7 of the run, as the K
// words).
template <int FMT, int DH>
KVQ_DEVI void q_fragments_fp8(const uint32_t (&w)[DH / 8], float sq, uint32_t (&qb)[DH / 16][2]) {
#pragma unroll
  for (int j = 0; j < DH / 16; ++j) {  // output word j: bf16 words 2j, 2j + 1
    const uint32_t lo = f32x2_to_fp8x2<FMT>(__fdiv_rn(bf16lo_to_f32(w[2 * j]), sq),
                                            __fdiv_rn(bf16hi_to_f32(w[2 * j]), sq));
    const uint32_t hi = f32x2_to_fp8x2<FMT>(__fdiv_rn(bf16lo_to_f32(w[2 * j + 1]), sq),
                                            __fdiv_rn(bf16hi_to_f32(w[2 * j + 1]), sq));
    qb[j >> 1][j & 1] = lo | (hi << 16);
  }
}

// Merge of the partial states of a segment split across CTAs, run by the
// consumer threads of the CTA that completed the segment's last piece.
//   M = max_c m_c,  l = sum_c l_c 2^(m_c - M),  O = sV sum_c o_c 2^(m_c - M) / l
// Warp w forms M, the weights 2^(m_c - M) (into wgt, [n][G]) and l of heads
// w, w + 4, ...; then every thread sums a float4 of O over the pieces.  The
// pieces' o vectors come either from so, a shared-memory copy the caller has
// started (bulk copy completing on sbar, phase 0), or straight from global
// memory (independent loads, 16 in flight).
template <int DH>
KVQ_DEVI void merge_segment(const DecodeParams& p, int b, int gkv, int64_t sigma, int64_t c_lo,
                            int n, float sv, float* wgt, const float* so, uint64_t* sbar,
                            volatile uint32_t* abort_flag, int ctid) {
  const int G = p.G;
  constexpr int NT = kConsumerWarps * 32;
  constexpr int KR = 10;  // pieces per lane kept in registers (n <= 320 in one pass)
  const int lane = ctid & 31, warp = ctid >> 5;
  uint16_t* out = p.out + (static_cast<int64_t>(b) * p.Hq + gkv * G) * DH;
  const bool ok = guard(c_lo >= 0 && c_lo + n - 1 + sigma < p.n_slots && n <= p.P, p.status, 5);
  float* Lh = wgt + static_cast<size_t>(n) * G;  // [G]
  const float2* ml = reinterpret_cast<const float2*>(p.ws_ml) + (c_lo + sigma) * G;
  for (int h = warp; ok && h < G; h += kConsumerWarps) {
    float2 v[KR];
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < KR; ++k) {
      const int c = lane + 32 * k;
      v[k] = c < n ? __ldcg(ml + c * G + h) : make_float2(-INFINITY, 0.f);
      M = fmaxf(M, v[k].x);
    }
    for (int c = lane + 32 * KR; c < n; c += 32) M = fmaxf(M, __ldcg(ml + c * G + h).x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
    float L = 0.f;
#pragma unroll
    for (int k = 0; k < KR; ++k) {
      const int c = lane + 32 * k;
      if (c < n) {
        const float w = (v[k].x == -INFINITY) ? 0.f : fast_exp2(v[k].x - M);
        wgt[c * G + h] = w;
        L += v[k].y * w;
      }
    }
    for (int c = lane + 32 * KR; c < n; c += 32) {
      const float2 x = __ldcg(ml + c * G + h);
      const float w = (x.x == -INFINITY) ? 0.f : fast_exp2(x.x - M);
      wgt[c * G + h] = w;
      L += x.y * w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
    if (lane == 0) Lh[h] = L;
  }
  consumer_bar();
  bool staged = so != nullptr;
  if (staged && !mbar_wait(sbar, 0u)) {
    staged = false;
    if (ctid == 0) {
      *abort_flag = 1u;
      flag_status(p.status, KVQ_DEV_WAIT_TIMEOUT);
    }
  }
  const int n4 = G * DH / 4;
  if (ok && (so == nullptr || staged)) {
    const float4* ob = staged ? reinterpret_cast<const float4*>(so)
                              : reinterpret_cast<const float4*>(p.ws_o + (c_lo + sigma) * G * DH);
    for (int q4 = ctid; q4 < n4; q4 += NT) {
      const int h = (4 * q4) / DH;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (staged) {
#pragma unroll 8
        for (int c = 0; c < n; ++c) {
          const float w = wgt[c * G + h];
          const float4 v = ob[static_cast<int64_t>(c) * n4 + q4];
          acc.x += w * v.x;
          acc.y += w * v.y;
          acc.z += w * v.z;
          acc.w += w * v.w;
        }
      } else {
#pragma unroll 16
        for (int c = 0; c < n; ++c) {
          const float w = wgt[c * G + h];
          const float4 v = __ldcg(ob + static_cast<int64_t>(c) * n4 + q4);
          acc.x += w * v.x;
          acc.y += w * v.y;
          acc.z += w * v.z;
          acc.w += w * v.w;
        }
      }
      const float ls = Lh[h];
      const float f = ls > 0.f ? sv / ls : 0.f;
      uint2 packed;
      packed.x = f32x2_to_bf16x2(acc.x * f, acc.y * f);
      packed.y = f32x2_to_bf16x2(acc.z * f, acc.w * f);
      *reinterpret_cast<uint2*>(out + 4 * q4) = packed;
    }
  }
  consumer_bar();
}

// --------------------------------------------------------------------------
// Decode kernel
// --------------------------------------------------------------------------

template <int FMT, int DH, bool PK, bool QF8, bool TS>
__global__ void __launch_bounds__(kThreads, kCtasPerSM)
    decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv) {
  using C = Cfg<FMT, DH>;
  constexpr int S = C::kStages;
  constexpr int MT = DH / 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  using SL = SmemLayout<FMT, DH, TS>;
  uint8_t* ring = smem + SL::ring;
  float* tsc_s = reinterpret_cast<float*>(smem + SL::tsc);  // [S][32] (TS)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SL::bars);
  uint64_t* empty = full + S;
  uint32_t* bad_s = reinterpret_cast<uint32_t*>(smem + SL::flags);
  volatile uint32_t* abort_flag = bad_s + S;
  volatile uint32_t* merge_s = bad_s + S + 1;
  int32_t* warp_tot = reinterpret_cast<int32_t*>(bad_s + S + 2);  // [8]
  int32_t* last_s = warp_tot + 8;  // [S] last position issued into each slot
  volatile uint32_t* mcopy_s = reinterpret_cast<volatile uint32_t*>(last_s + S);  // merge copy issued
  uint64_t* mbar = empty + S;  // completion of the segment-merge bulk copy
  int32_t* ub = reinterpret_cast<int32_t*>(const_cast<uint32_t*>(mcopy_s + 1));  // [2] u0, u1
  float* cm = reinterpret_cast<float*>(smem + SL::comb);   // [warps][G] running max
  float* cl = cm + kConsumerWarps * p.G;                   // [warps][G] denominators
  float* co = cl + kConsumerWarps * p.G;                   // [warps][G][DH] unnormalised O
  int32_t* seq_off = reinterpret_cast<int32_t*>(smem + SL::seq(p.G, p.P));  // [B+1]
  int32_t* len_s = seq_off + p.B + 1;                                  // [B]
  int32_t* vseq_off = len_s + p.B;                                     // [B+1]
  float* sk_s = reinterpret_cast<float*>(smem + SL::scales(p.G, p.P, p.B)); // [Hkv]
  float* sv_s = sk_s + p.Hkv;                                          // [Hkv]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  static_assert(S < kThreads, "one thread per ring slot initialises its barriers");
  if (tid < S) {
    mbar_init(&full[tid], 1);
    mbar_init(&empty[tid], 1);
    last_s[tid] = -1;
    fence_mbar_init();
  } else if (tid == S) {
    mbar_init(mbar, 1);
    *mcopy_s = 0u;
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  // Inputs may come from the kernel before this one on the stream: wait for
  // it here, or -- under KVQ_CACHE_READY -- only before reading q or a
  // sequence's last page and before the first write.
  if (!p.early) {
    pdl_wait();
    pdl_allow_next();
  }
  build_plan<FMT != KVQ_FMT_BF16 && !TS>(p, seq_off, len_s, vseq_off, sk_s, sv_s, warp_tot);

  const int64_t W = seq_off[p.B];
  // Sequences with nothing to attend to get a zero output row (CTAs share them).
  auto zero_empty_rows = [&](int first, int step) {
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
      if (seq_off[b + 1] != seq_off[b]) continue;
      uint16_t* row = p.out + static_cast<int64_t>(b) * p.Hq * DH;
      for (int i = first; i < p.Hq * DH; i += step) row[i] = 0;
    }
  };
  if (!p.early) zero_empty_rows(tid, kThreads);
  // Partition size: never more CTAs than units (the others idle).  CTA c
  // takes units [u0, u1), a cost-balanced range; a CTA whose cost
  // range lies in one segment's fixed cost may get none.
  const int Pe = static_cast<int>(W < p.P ? W : p.P);
  const int c = blockIdx.x;
  const CostSplit cost_split(vseq_off[p.B], Pe);
  if ((tid == 0 || tid == 32) && c < Pe)  // this CTA's bounds, two warps in parallel
    ub[tid >> 5] = pages_before(seq_off, vseq_off, p.B, p.Hkv, cost_split(c + (tid >> 5)));
  __syncthreads();
  const int64_t u0 = c < Pe ? ub[0] : 0;
  const int64_t u1 = c < Pe ? ub[1] : 0;
  const int64_t total = u1 - u0;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // Lane j owns ring slots j and j + 32 and issues their positions
    // slot, slot + S, slot + 2S, ... of the CTA's page stream.  Each lane
    // polls its own empty barriers without blocking, so up to S pages are
    // requested at once, and looks up the block id of a slot's next position
    // right after an issue, one ring turn ahead.
    constexpr int SPL = (S + 31) / 32;  // slots per lane
    static_assert(SPL <= 2, "at most 64 ring slots");
    // blk_out: the page's block id (-1 if out of range); last_out: the page
    // holds the sequence's last token (read only after the wait).
    auto lookup = [&](int64_t i, int& blk_out, int& g_out, bool& last_out) {
      const int64_t u = u0 + i;
      const int b = find_seq(seq_off, p.B, u);
      const int pages = (seq_off[b + 1] - seq_off[b]) / p.Hkv;
      const int r = static_cast<int>(u - seq_off[b]);
      g_out = r / pages;
      const int pg = r - g_out * pages;
      const int col = first_page_of(p, len_s[b]) + pg;
      last_out = pg == pages - 1;
      if (guard(b >= 0 && b < p.B && col >= 0 && col < p.max_blocks && g_out >= 0 &&
                    g_out < p.Hkv,
                p.status, 0))
        blk_out = __ldg(p.block_tables + static_cast<int64_t>(b) * p.max_blocks + col);
      else
        blk_out = -1;
    };
    int64_t q[SPL];
    int blk[SPL], gg[SPL];
    uint32_t par[SPL];
    bool done[SPL], lastp[SPL];
    bool waited = !p.early;
#pragma unroll
    for (int k = 0; k < SPL; ++k) {
      q[k] = lane + 32 * k;
      par[k] = 1u;  // the first wait on a fresh empty barrier passes
      done[k] = lane + 32 * k >= S || q[k] >= total;
      blk[k] = gg[k] = 0;
      lastp[k] = false;
      if (!done[k]) lookup(q[k], blk[k], gg[k], lastp[k]);
    }
    // The cache pages are read once per call: first out of L2, so the
    // stream does not push out the tables, partial states or code.
    const uint64_t pol = l2_evict_first_policy();
    uint32_t idle = 0;
    while (true) {
      bool live = false, progressed = false, blocked = false;
#pragma unroll
      for (int k = 0; k < SPL; ++k) {
        if (done[k]) continue;
        live = true;
        if (!waited && lastp[k]) {
          blocked = true;
          continue;
        }
        const int slot = lane + 32 * k;
        if (!mbar_test_wait(&empty[slot], par[k])) continue;
#ifdef KVQ_TEST_HOOKS
        if (blockIdx.x == 0 && q[k] == p.withhold) {
          // Test builds only: this position's copy is never issued and its
          // full barrier never completes, so the consumer's bounded wait on
          // it runs out.  The slot is left for the aborting consumers.
          done[k] = true;
          progressed = true;
          continue;
        }
#endif
        const bool bad = blk[k] < 0 || blk[k] >= p.num_blocks;
        if (bad) flag_status(p.status, KVQ_DEV_BAD_BLOCK);
        int32_t row = ((bad ? 0 : blk[k]) * p.Hkv + gg[k]) * kBS;
        bool skip = bad;
        if (!guard(row >= 0 && row + kBS <= p.rows, p.status, 1)) {
          row = 0;
          skip = true;
        }
        bad_s[slot] = skip ? 1u : 0u;
        uint8_t* dstK = ring + slot * C::kSlot;
        mbar_arrive_expect_tx(&full[slot], C::kSlot + (TS ? 128 : 0));
        if (C::kRow > 128) {  // two 128-byte column boxes per page
          tma_load_2d_hint(dstK, &tmk, 0, row, &full[slot], pol);
          tma_load_2d_hint(dstK + C::kPage / 2, &tmk, 64, row, &full[slot], pol);
          tma_load_2d_hint(dstK + C::kPage, &tmv, 0, row, &full[slot], pol);
          tma_load_2d_hint(dstK + C::kPage + C::kPage / 2, &tmv, 64, row, &full[slot], pol);
        } else {
          tma_load_2d_hint(dstK, &tmk, 0, row, &full[slot], pol);
          tma_load_2d_hint(dstK + C::kPage, &tmv, 0, row, &full[slot], pol);
        }
        if (TS) {  // the page's 16 K and 16 V scales (row is a multiple of 16)
          bulk_load(tsc_s + slot * 32, p.ks + row, 64, &full[slot]);
          bulk_load(tsc_s + slot * 32 + 16, p.vs + row, 64, &full[slot]);
        }
        last_s[slot] = static_cast<int32_t>(q[k]);
        q[k] += S;
        par[k] ^= 1u;
        if (q[k] < total)
          lookup(q[k], blk[k], gg[k], lastp[k]);
        else
          done[k] = true;
        progressed = true;
      }
      if (!__any_sync(kFull, live)) break;
      if (!waited && __any_sync(kFull, blocked)) {  // a last page is next: wait for the previous kernel
        pdl_wait();
        waited = true;
        continue;
      }
      if (__any_sync(kFull, progressed)) {
        idle = 0;
      } else {
        if (*abort_flag) break;
        if (++idle > kMaxPolls) {
          if (lane == 0) {
            *abort_flag = 1u;
            flag_status(p.status, KVQ_DEV_WAIT_TIMEOUT);
          }
          break;
        }
        __nanosleep(20);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3;
    const int ctid = tid;  // 0 .. 127
    const int qhead = PK ? (g & 3) : g;  // query head of this lane's QK column
    uint32_t qb[MT][2];
    uint32_t qraw[DH / 8];  // raw Q words of the current piece, loaded a piece ahead
    float o[MT][4];
    int pos_base = 0;
    bool aborted = false;
    // piece = the part of one (sequence, KV head) segment inside [u0, u1)
    if (p.early) {  // q and every write wait for the previous kernel
      pdl_wait();
      pdl_allow_next();
      zero_empty_rows(ctid, kConsumerWarps * 32);
    }
    auto piece_at = [&](int64_t u, int& b, int& gkv, int& pages, int& p0) {
      b = find_seq(seq_off, p.B, u);
      pages = (seq_off[b + 1] - seq_off[b]) / p.Hkv;
      const int r = static_cast<int>(u - seq_off[b]);
      gkv = pages > 0 ? r / pages : 0;
      p0 = r - gkv * pages;
    };
    if (u0 < u1) {
      int b, gkv, pages, p0;
      piece_at(u0, b, gkv, pages, p0);
      load_q_raw<DH>(p, b, gkv, qhead, t, qraw);
    }

    for (int64_t u = u0; u < u1;) {
      int b, gkv, pages, p0;
      piece_at(u, b, gkv, pages, p0);
      if (!guard(pages > 0 && u >= seq_off[b] && u < seq_off[b + 1], p.status, 10)) break;
      const int n = static_cast<int>((u1 - u) < (pages - p0) ? (u1 - u) : (pages - p0));
      const int L = len_s[b];
      const int lo = window_lo(p, L);
      const int fp = lo / kBS;
      const float sv = sv_s[gkv];
      const float lscale = sk_s[gkv] * p.logit_scale;
      // FP8-domain query: this lane's query head scale, and the two MMA
      // columns' (heads 2t, 2t + 1 of the group, or their P_lo copies) logit
      // scales carry their heads' sQ
      float lscale0 = lscale, lscale1 = lscale, sq = 1.f;
      if (QF8) {
        auto q_scale_of = [&](int hh) {
          return hh < p.G ? __ldg(p.qs + (p.q_per_head ? gkv * p.G + hh : 0)) : 1.f;
        };
        sq = q_scale_of(qhead);
        lscale0 = lscale * q_scale_of(PK ? ((2 * t) & 3) : 2 * t);
        lscale1 = lscale * q_scale_of(PK ? ((2 * t + 1) & 3) : 2 * t + 1);
      }
      const bool single = (p0 == 0 && n == pages);
      // A split segment's pieces are those of CTAs seg_lo .. seg_lo + seg_n - 1:
      // the CTAs holding the cost positions of its first and last pages.
      int seg_lo = c, seg_n = 1;
      if (!single) {
        const int v_first = vseq_off[b] + gkv * (pages + kPieceCost) + kPieceCost;
        seg_lo = cost_split.cta_of(v_first);
        seg_n = cost_split.cta_of(v_first + pages - 1) - seg_lo + 1;
      }
      if (QF8) {
        q_fragments_fp8<FMT, DH>(qraw, sq, qb);
      } else {
        const int qa = q_fragments<FMT, DH>(qraw, qb);
        if (FMT != KVQ_FMT_BF16) {  // 2^-a of each column's head (held by its lane t = 0)
          const int a0 = __shfl_sync(kFull, qa, 4 * (PK ? ((2 * t) & 3) : 2 * t));
          const int a1 = __shfl_sync(kFull, qa, 4 * (PK ? ((2 * t + 1) & 3) : 2 * t + 1));
          lscale0 *= __int_as_float((127 - a0) << 23);
          lscale1 *= __int_as_float((127 - a1) << 23);
        }
      }
      if (u + n < u1) {  // next piece's Q, in flight while this piece runs
        int nb, ng, npg, np0;
        piece_at(u + n, nb, ng, npg, np0);
        load_q_raw<DH>(p, nb, ng, qhead, t, qraw);
      }
      SoftmaxState st;
      st.m[0] = st.m[1] = -INFINITY;
      st.l[0] = st.l[1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

      static_assert(S % kConsumerWarps == 0, "slots must split evenly among the consumer warps");
      // This warp's positions in the piece are j0, j0 + 4, j0 + 8, ...; it
      // takes them NP at a time (positions j, j + 4, ..., j + 4 (NP - 1)).
      constexpr int NP = C::kPagesPerStep;
      const int j0 = (warp - pos_base % kConsumerWarps + kConsumerWarps) % kConsumerWarps;
      int cur_slot = (pos_base + j0) % S;  // stage and phase parity of position pos_base + j0
      uint32_t cur_par = static_cast<uint32_t>(((pos_base + j0) / S) & 1);
      for (int j = j0; j < n; j += NP * kConsumerWarps) {
        int slot[NP];
        uint32_t spar[NP];
        bool have[NP];
        bool ok = true;
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          have[i] = j + i * kConsumerWarps < n;  // warp-uniform
          slot[i] = cur_slot;
          spar[i] = cur_par;
          if (have[i] && ok && !aborted) ok = wait_or_abort(&full[cur_slot], cur_par, abort_flag);
          cur_slot += kConsumerWarps;
          if (cur_slot >= S) {
            cur_slot -= S;
            cur_par ^= 1u;
          }
        }
        if (!__all_sync(kFull, ok) && !aborted) {
          aborted = true;
          if (lane == 0) {
            *abort_flag = 1u;
            flag_status(p.status, KVQ_DEV_WAIT_TIMEOUT);
          }
        }
        if (!aborted) {
          PageRegs<FMT, DH> pr[NP];
          int tok0[NP];
          bool bad[NP];
          float tsk[NP][2], tsv[NP][2];
#pragma unroll
          for (int i = 0; i < NP; ++i) {
            tok0[i] = (fp + p0 + j + i * kConsumerWarps) * kBS;
            tsk[i][0] = tsk[i][1] = tsv[i][0] = tsv[i][1] = 0.f;
            if (have[i]) {
              const uint32_t kp = smem_u32(ring + slot[i] * C::kSlot);
              bad[i] = bad_s[slot[i]] != 0u;
              load_page<FMT, DH>(kp, kp + C::kPage, g, t, tok0[i], lo, L, bad[i], pr[i]);
              if (TS) {  // scales of token rows g and g + 8
                const float* sc = tsc_s + slot[i] * 32;
                tsk[i][0] = sc[g];
                tsk[i][1] = sc[g + 8];
                tsv[i][0] = sc[16 + g];
                tsv[i][1] = sc[24 + g];
              }
            } else {  // past the piece's last page: an empty, masked page
              bad[i] = true;
              pr[i] = PageRegs<FMT, DH>{};
            }
          }
          __syncwarp();
          if (lane == 0) {  // slots free: their data is in registers
#pragma unroll
            for (int i = 0; i < NP; ++i)
              if (have[i]) mbar_arrive(&empty[slot[i]]);
          }
          compute_pages<FMT, DH, NP, PK, QF8, TS>(pr, tok0, bad, g, t, p.G, qb, o, st, lscale0,
                                                  lscale1, lo, L, tsk, tsv);
        } else {
          // Aborted: a slot goes back only once its copy has landed, so the
          // producer never re-arms a slot whose copy is still in flight (it
          // then idles, sees the abort and stops).
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int i = 0; i < NP; ++i)
              if (have[i] && mbar_test_wait(&full[slot[i]], spar[i])) mbar_arrive(&empty[slot[i]]);
          }
        }
      }

      // ---- merge the four warps' states of this segment piece
      if (PK) {  // columns 4..7 hold the P_lo contributions of heads 0..3
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) o[mt][i] += __shfl_xor_sync(kFull, o[mt][i], 2);
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        st.l[0] += __shfl_xor_sync(kFull, st.l[0], off);
        st.l[1] += __shfl_xor_sync(kFull, st.l[1], off);
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int h = 2 * t + c;
        if (h < p.G) {
          if (g == 0) {
            cm[warp * p.G + h] = st.m[c];
            cl[warp * p.G + h] = st.l[c];
          }
          float* dst = co + (warp * p.G + h) * DH + g * (DH / 8);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
            *reinterpret_cast<float2*>(dst + 2 * mt) = make_float2(o[mt][c], o[mt][2 + c]);
        }
      }
      consumer_bar();
      const int64_t slot_idx = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(b) * p.Hkv + gkv;
      // Each thread combines four consecutive dims of one head: the four
      // warps' weights 2^(m_w - M) once, then float4 rows of O.
      for (int q4 = ctid; q4 < p.G * (DH / 4); q4 += kConsumerWarps * 32) {
        const int h = q4 / (DH / 4), d = 4 * q4 - h * DH;
        float mw[kConsumerWarps], M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          mw[w] = cm[w * p.G + h];
          M = fmaxf(M, mw[w]);
        }
        float ls = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float sc = (mw[w] == -INFINITY) ? 0.f : fast_exp2(mw[w] - M);
          const float4 v = *reinterpret_cast<const float4*>(co + (w * p.G + h) * DH + d);
          ls += cl[w * p.G + h] * sc;
          acc.x += v.x * sc;
          acc.y += v.y * sc;
          acc.z += v.z * sc;
          acc.w += v.w * sc;
        }
        if (single) {
          const float f = ls > 0.f ? sv / ls : 0.f;
          const int64_t oi = (static_cast<int64_t>(b) * p.Hq + gkv * p.G + h) * DH + d;
          if (guard(oi >= 0 && oi + 4 <= static_cast<int64_t>(p.B) * p.Hq * DH, p.status, 3)) {
            uint2 packed;
            packed.x = f32x2_to_bf16x2(acc.x * f, acc.y * f);
            packed.y = f32x2_to_bf16x2(acc.z * f, acc.w * f);
            *reinterpret_cast<uint2*>(p.out + oi) = packed;
          }
        } else if (guard(slot_idx >= 0 && slot_idx < p.n_slots, p.status, 4)) {
          *reinterpret_cast<float4*>(p.ws_o + (slot_idx * p.G + h) * DH + d) = acc;
          if (d == 0)
            *reinterpret_cast<float2*>(p.ws_ml + (slot_idx * p.G + h) * 2) = make_float2(M, ls);
        }
      }
      consumer_bar();
      if (!single) {
        // Publish this piece; the CTA whose piece completes the segment merges
        // all of its pieces and resets the segment's counter.
        const int64_t sigma = static_cast<int64_t>(b) * p.Hkv + gkv;
        // The barrier above orders every thread's partial stores before
        // thread 0's arrival, an acquire-release atomic at GPU scope: its
        // release publishes them, and for the arrival that completes the
        // count its acquire (then the barrier below) makes every piece's
        // stores visible to the merging threads.
        const int64_t c_lo = seg_lo;  // CTA holding the segment's first unit
        const int npieces = seg_n;
        if (ctid == 0) {
          const uint32_t prev = atom_add_acq_rel_gpu(p.ws_cnt + sigma, 1u);
          const bool last = prev + 1 == static_cast<uint32_t>(npieces);
          merge_s[0] = last ? 1u : 0u;
        }
        consumer_bar();
        if (merge_s[0]) {
          // After the CTA's last piece the ring is idle (every issued page
          // has been consumed): the pieces' o vectors are bulk-copied into it
          // while the weights are formed.
          const uint32_t pbytes = static_cast<uint32_t>(p.G * DH * sizeof(float));
          const bool stage = (u + n == u1) && !*abort_flag && c_lo >= 0 && npieces <= p.P &&
                             c_lo + sigma + npieces <= p.n_slots &&
                             static_cast<size_t>(npieces) * pbytes <= static_cast<size_t>(S) * C::kSlot;
          if (stage && warp == 0) {
            if (lane == 0) {
              *mcopy_s = 1u;
              mbar_arrive_expect_tx(mbar, npieces * pbytes);
            }
            __syncwarp();
            fence_proxy_async_global();  // the partials were acquired through the counter
            fence_proxy_async_smem();    // the ring was last read by generic loads
            const float* src = p.ws_o + (c_lo + sigma) * p.G * DH;
            for (int c = lane; c < npieces; c += 32)
              bulk_load(ring + static_cast<size_t>(c) * pbytes, src + static_cast<size_t>(c) * p.G * DH,
                        pbytes, mbar);
          }
          merge_segment<DH>(p, b, gkv, sigma, c_lo, npieces, sv, cm,
                            stage ? reinterpret_cast<const float*>(ring) : nullptr, mbar, abort_flag,
                            ctid);
          if (ctid == 0) p.ws_cnt[sigma] = 0u;
        }
      }
      pos_base += n;
      u += n;
    }
  }
  __syncthreads();
  // After an abort, wait (bounded) for copies still in flight before exit.
  if (*abort_flag && tid == 0) {
    for (int s = 0; s < S; ++s)
      if (last_s[s] >= 0) mbar_wait(&full[s], static_cast<uint32_t>((last_s[s] / S) & 1));
    if (*mcopy_s) mbar_wait(mbar, 0u);
  }
}

// --------------------------------------------------------------------------
// Launch
// --------------------------------------------------------------------------

template <int FMT, int DH, bool TS>
static size_t smem_bytes(int G, int P, int B, int Hkv) {
  return SmemLayout<FMT, DH, TS>::total(G, P, B, Hkv);
}

template <int FMT, int DH, bool TS>
static int launch_ts(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                     cudaStream_t s) {
  constexpr bool FP8 = FMT != KVQ_FMT_BF16;
  const size_t smem = smem_bytes<FMT, DH, TS>(p.G, p.P, p.B, p.Hkv);
  // The kernels' attributes, set once per device (again after a failure).
  static DeviceOnce once;
  const bool configured = once.run(current_device(), [] {
    const int maxsmem = static_cast<int>(
        smem_bytes<FMT, DH, TS>(kMaxGroup, kCtasPerSM * device_sm_count(), kMaxSeqs, kMaxKvHeads));
    // The largest shared-memory carveout, so that two CTAs fit on every SM.
    auto configure = [&](auto kernel) {
      return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, maxsmem) ==
                 cudaSuccess &&
             cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared) == cudaSuccess;
    };
    bool ok = configure(decode_kernel<FMT, DH, true, false, TS>) &&
              configure(decode_kernel<FMT, DH, false, false, TS>);
    if constexpr (FP8)
      ok = ok && configure(decode_kernel<FMT, DH, true, FP8, TS>) &&
           configure(decode_kernel<FMT, DH, false, FP8, TS>);
    return ok;
  });
  if (!configured) return KVQ_ERR_CUDA;
  const dim3 grid(p.P), block(kThreads);
  cudaError_t e;
  // the FP8-domain query variants exist for FP8 caches only (QF8 = FP8)
  if (FP8 && p.qs)
    e = p.G <= 4 ? launch_pdl(decode_kernel<FMT, DH, true, FP8, TS>, grid, block, smem, s, p, tk, tv)
                 : launch_pdl(decode_kernel<FMT, DH, false, FP8, TS>, grid, block, smem, s, p, tk, tv);
  else
    e = p.G <= 4 ? launch_pdl(decode_kernel<FMT, DH, true, false, TS>, grid, block, smem, s, p, tk, tv)
                 : launch_pdl(decode_kernel<FMT, DH, false, false, TS>, grid, block, smem, s, p, tk, tv);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// Decode launch for one cache format and head size (per-token scales only
// for the FP8 formats).
template <int FMT, int DH>
int launch(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  if constexpr (FMT != KVQ_FMT_BF16) {
    if (p.ts) return launch_ts<FMT, DH, true>(p, tk, tv, s);
  }
  return launch_ts<FMT, DH, false>(p, tk, tv, s);
}

}  // namespace kvq
