// kvq_prefill_tc.cuh -- the prefill kernel of the FP8 caches on the 5th-
// generation tensor cores (tcgen05, accumulators in tensor memory).
//
// One CTA per (sequence, KV head, one or two adjacent tiles of 128 query
// rows); a row is a (query token, query head of the group) pair, so a tile
// holds 128 / G tokens.  The keys stream in blocks of 64 tokens (4 pages),
// each converted once for both tiles:
//   warp 12 (producer): block ids 32 pages at a time (one per lane), TMA loads
//     of each block's 4 K and 4 V FP8 pages into a 3-stage ring (the
//     decode's 128-byte-swizzled page boxes).
//   warps 8-11 (converters): each block's pages to f16 in shared memory, K as
//     the B operand of QK^T and V as the MN-major B operand of PV, both
//     token-major in the same layout, in 3 buffers.
//   warps 13 and 14 (MMA of tiles 0 and 1; warp 13 allocates the 512 TMEM
//     columns: per tile a 64-column S, two 32-column P buffers and the
//     dh-column O accumulator): one elected lane each issues, per block of
//     its tile, S = Q K^T (M = 128, N = 64, K = dh in steps of 16) once the
//     softmax has read the previous S, and O += P V (A = P from tensor
//     memory, N = dh, K = 64 tokens) once the block's P is in, each
//     completion signalled to an mbarrier by tcgen05.commit.  A tile skips
//     the blocks none of its rows sees.
//   warps 0-3 and 4-7 (softmax of tiles 0 and 1; thread r of a tile = row r
//     = TMEM lane r): Q row r to f16, then per block the S row from TMEM
//     (released at once), causal / window mask (skipped for blocks the whole
//     row sees), online max with a lazy rescale of the O row in TMEM, and
//     P = 2^(x-m) as f16 into P buffer i % 2 once the PV of block i - 2 has
//     read it.
// Every shared-memory operand is in the K-major 128-byte-swizzle layout:
// 8-row groups of 1024 bytes, 128-byte rows of 64 f16, 16-byte chunk c of
// row r at chunk c ^ (r % 8); wider K in further 64-column blocks of the
// tile.  All waits are bounded; a timeout sets KVQ_DEV_WAIT_TIMEOUT, the
// roles stop, and the CTA waits (bounded) for its copies and MMAs in flight
// before it frees the tensor memory.
#pragma once

#include "kvq_tc.cuh"

namespace kvq {
namespace tc {

constexpr int kRows = 128;      // query rows per tile (MMA M)
constexpr int kTiles = 2;       // query tiles per CTA
constexpr int kKeys = 64;       // tokens per key block (QK^T N, PV K)
// warps 0-7 softmax (4 per tile), 8-11 convert, 12 producer, 13-14 MMA (one per tile)
constexpr int kThreadsTc = 480;
constexpr int kConvWarp = 8, kProdWarp = 12, kMmaWarp = 13;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTileCols = 256;  // per tile: S at +0, P buffers at +64, +96, O at +128

// Shared memory: the two Q tiles, kB f16 K / V buffers (the converters run
// kB - 1 blocks ahead of the PVs) and kS FP8 page stages.
template <int DH, bool TS>
struct Layout {
  static constexpr int kS = 3;
  static constexpr int kB = 3;
  static constexpr int kPage8 = kBS * DH;                  // bytes of one FP8 page
  static constexpr int kStage = 8 * kPage8;                // 4 K pages + 4 V pages
  static constexpr size_t q = 0;                           // Q   kTiles x [128][DH] f16
  static constexpr size_t qBytes = static_cast<size_t>(kRows) * DH * 2;
  static constexpr size_t k = q + kTiles * qBytes;         // K   kB x [64][DH] f16
  static constexpr size_t kBytes = static_cast<size_t>(kKeys) * DH * 2;
  static constexpr size_t vt = k + kB * kBytes;            // V   kB x [64][DH] f16
  static constexpr size_t vtBytes = static_cast<size_t>(DH) * kKeys * 2;
  static constexpr size_t stage = vt + kB * vtBytes;       // FP8 pages, kS stages
  // per-(token, head) scales: each stage's [4 pages][K 16, V 16] fp32, then
  // each f16 buffer's block [K 64, V 64] fp32 (zero where masked)
  static constexpr size_t ssc = stage + static_cast<size_t>(kS) * kStage;
  static constexpr size_t bsc = ssc + (TS ? static_cast<size_t>(kS) * 4 * 32 * 4 : 0);
  static constexpr size_t bars = bsc + (TS ? static_cast<size_t>(kB) * 128 * 4 : 0);
  // barriers: full[S], empty[S], conv[kB], kvdone[kB], sfull[kTiles], sfree[kTiles],
  // pfull[kTiles][2], pdone[kTiles][2], fin, qready
  static constexpr int kBars = 2 * kS + 2 * kB + 6 * kTiles + 2;
  static constexpr size_t misc = bars + kBars * sizeof(uint64_t);
  // misc: tmem address, abort flag, page flags [S stages][4 pages], issued[S],
  // masked pages of the blocks in the f16 buffers [kB]
  static constexpr size_t total = misc + 256 + 1024;
};

// Byte offset of f16 element (row, col) in a K-major 128-byte-swizzled tile
// of `rows` rows (col = K index).
KVQ_DEVI uint32_t sw128_off(int row, int col, int rows) {
  const int blk = col >> 6, c16 = (col & 63) >> 3;
  return static_cast<uint32_t>(blk * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
                               ((c16 ^ (row & 7)) << 4) + ((col & 7) << 1));
}

// Descriptor of V as the MN-major B operand of PV (N = head dims along each
// 128-byte row, K = tokens down the rows; the K tile's layout): the leading
// byte offset steps to the next 64 dims (64 token rows on, 8192 bytes), the
// stride byte offset to the next 8 tokens (1024 bytes).  (The other
// assignment of the two strides gave wrong sums; this one reproduced the
// transposed-V kernel's output bit for bit.)
KVQ_DEVI uint64_t sw128_desc_mn(uint32_t saddr) {
  constexpr uint64_t lbo = kKeys * 128, sbo = 1024;
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | ((lbo >> 4) << 16) | ((sbo >> 4) << 32) |
         (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
}

// TS: per-(token, head) scales (p.ts), a separate instance so that the other
// scale modes keep their loop free of the per-key scaling.
template <int FMT, int DH, bool TS>
__global__ void __launch_bounds__(kThreadsTc, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillParams p,
                      const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
  using Lo = Layout<DH, TS>;
  using C = Cfg<FMT, DH>;
  constexpr int S = Lo::kS;
  constexpr int kBufs = Lo::kB;
  constexpr int KSTEPS = DH / 16;  // QK^T MMAs per block
  static_assert(C::kRow == DH && C::kPage == Lo::kPage8, "FP8 pages");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lo::bars);
  uint64_t* full = bars;               // [S] FP8 stage landed
  uint64_t* empty = bars + S;          // [S] FP8 stage converted (128 arrivals)
  uint64_t* conv = bars + 2 * S;            // [kBufs] f16 K / V buffer b ready (128 arrivals)
  uint64_t* kvdone = conv + kBufs;          // [kBufs] buffer b's block released by both issuers
  uint64_t* sfull = kvdone + kBufs;         // [kTiles] a tile's S written (commit)
  uint64_t* sfree = sfull + kTiles;         // [kTiles] a tile's S read (128 arrivals)
  uint64_t* pfull = sfree + kTiles;         // [kTiles][2] P buffer of a tile written (128 arrivals)
  uint64_t* pdone = pfull + 2 * kTiles;     // [kTiles][2] PV from a tile's P buffer done (commit)
  uint64_t* fin = pdone + 2 * kTiles;       // every MMA done (a commit of each issuer)
  uint64_t* qready = fin + 1;               // both Q tiles written (256 arrivals)
  // A parity wait for phase p of a barrier is sound only while the barrier
  // has completed p or p + 1 phases.  Every waiter therefore waits each of
  // its barriers' phases in order, never skipping one (so p - 1 is known
  // complete), and a barrier's phase after p needs the waiter's own later
  // progress; P buffers and their barriers come in pairs (even and odd
  // blocks), so that no waiter can fall two phases behind, and a tile's
  // single S buffer is rewritten only after its softmax has read it.  A tile's
  // softmax, which may start after block 0, waits for a
  // block's conversion only once the block's S is in (the MMA lane issued
  // QK^T after that conversion): the phase is then complete, and the next
  // one needs this tile's PV of the block.  Completion order is not assumed
  // between MMAs that write different accumulators: QK^T of a block may
  // finish before the PV issued ahead of it, so "S is ready" says nothing
  // about earlier PVs.
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + Lo::misc);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  uint32_t* pg_bad = const_cast<uint32_t*>(tmem_slot + 2);    // [S][4] page masked out
  int32_t* issued = reinterpret_cast<int32_t*>(pg_bad + S * 4);  // [S] last block issued
  volatile uint32_t* bufmask = reinterpret_cast<volatile uint32_t*>(issued + S);  // [kBufs]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.z, gkv = blockIdx.y;
  // p.tpc tiles a CTA (1 or kTiles; with 1, tile 1's warps have no rows)
  const int groups = (p.tiles + p.tpc - 1) / p.tpc;
  const int pair = groups - 1 - static_cast<int>(blockIdx.x);  // longest first
  const int TQ = kRows / p.G;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 128);
      issued[i] = -1;
    }
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(&conv[i], 128);
      mbar_init(&kvdone[i], kTiles);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&sfull[t], 1);
      mbar_init(&sfree[t], 128);
      mbar_init(&pfull[2 * t], 128);
      mbar_init(&pfull[2 * t + 1], 128);
      mbar_init(&pdone[2 * t], 1);
      mbar_init(&pdone[2 * t + 1], 1);
    }
    mbar_init(fin, kTiles);
    mbar_init(qready, kTiles * 128);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kProdWarp && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  pdl_wait();
  pdl_allow_next();

  const int q0 = __ldg(p.cu_q + b);
  const int n = __ldg(p.cu_q + b + 1) - q0;
  const int j0 = pair * p.tpc * TQ;  // first query token of tile 0
  // a chunk longer than the grid covers (max_q_len): its later rows stay unwritten
  if (blockIdx.x == 0 && gkv == 0 && tid == 0 && n > p.tiles * TQ)
    flag_status(p.status, KVQ_DEV_BAD_QLEN);
  if (n <= 0 || j0 >= n) return;  // the whole CTA, before any tensor memory is taken
  const int j1 = min(n, j0 + p.tpc * TQ);  // past the CTA's last query token
  const int L = __ldg(p.seq_lens + b);
  if (!(L >= n && L <= p.max_blocks * kBS)) {
    if (pair == 0 && gkv == 0 && tid == 0) flag_status(p.status, KVQ_DEV_BAD_SEQLEN);
    for (int i = tid; i < (j1 - j0) * p.G * DH; i += kThreadsTc) {
      const int r = i / DH, d = i - r * DH;
      const int64_t orow = static_cast<int64_t>(q0 + j0 + r / p.G) * p.Hq + gkv * p.G + r % p.G;
      if (guard(orow >= 0 && orow < p.total_q * p.Hq, p.status, 20)) p.out[orow * DH + d] = 0;
    }
    return;
  }
  const int base = L - n;  // position of query token 0
  const int pos_first = base + j0, pos_last = base + j1 - 1;
  const int p_begin = window_lo(p.window, pos_first + 1) / kBS;  // first page
  const int p_end = pos_last / kBS;                              // last page
  const int nblk = (p_end - p_begin) / 4 + 1;                    // key blocks of 4 pages
  // Tile t's blocks [jb[t], je[t]): from its first row's window start to its
  // last row (empty for a tile past the chunk).  Adjacent tiles leave no
  // block between them uncovered.
  int jb[kTiles], je[kTiles];
#pragma unroll
  for (int t = 0; t < kTiles; ++t) {
    const int a = j0 + t * TQ, e = min(n, a + TQ);
    if (t >= p.tpc || a >= n) {
      jb[t] = je[t] = 0;
    } else {
      jb[t] = (window_lo(p.window, base + a + 1) / kBS - p_begin) / 4;
      je[t] = ((base + e - 1) / kBS - p_begin) / 4 + 1;
    }
  }

  if (warp == kMmaWarp) {  // tensor memory: per tile S (2 x 64 columns) and O (DH columns)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(const_cast<uint32_t*>(tmem_slot))), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&](void) {
    if (!*abort_flag) {
      *abort_flag = 1u;
      flag_status(p.status, KVQ_DEV_WAIT_TIMEOUT);
    }
  };

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    // The 32 lanes look up the block ids of 8 blocks (32 pages) at once, a
    // group ahead; lane 0 takes each block's four by shuffle and issues its
    // TMA loads.  (One lane looking them up in turn made the page stream wait
    // four L2 round trips per block.)
    int my_row = -1;  // cache row of page p_begin + 4 (j - j % 8) + lane, -1 if masked out
    for (int j = 0; j < nblk; ++j) {
      const int s = j % S;
      if ((j & 7) == 0) {
        const int col = p_begin + 4 * j + lane;
        const bool in = col <= p_end;
        int blk = -1;
        if (in && guard(col >= 0 && col < p.max_blocks, p.status, 21))
          blk = __ldg(p.block_tables + static_cast<int64_t>(b) * p.max_blocks + col);
        bool bad = blk < 0 || blk >= p.num_blocks;
        if (bad && in) flag_status(p.status, KVQ_DEV_BAD_BLOCK);
        const int32_t row = ((bad ? 0 : blk) * p.Hkv + gkv) * kBS;
        if (!bad && !guard(row >= 0 && row + kBS <= p.rows, p.status, 22)) bad = true;
        my_row = bad ? -1 : row;
      }
      int rows[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) rows[i] = __shfl_sync(kFull, my_row, 4 * (j & 7) + i);
      const bool ok = j < S || __all_sync(kFull, wait_or_abort(&empty[s], static_cast<uint32_t>(((j / S) - 1) & 1), abort_flag));
      if (__any_sync(kFull, !ok || *abort_flag)) {  // the same decision on every lane
        if (lane == 0) fail();
        break;
      }
      if (lane == 0) {
        uint32_t bytes = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          pg_bad[s * 4 + i] = rows[i] < 0 ? 1u : 0u;
          if (rows[i] >= 0) bytes += 2 * Lo::kPage8 + (TS ? 2 * 64 : 0);
        }
        issued[s] = j;
        if (bytes == 0) {  // nothing to load: complete the phase by hand
          mbar_arrive(&full[s]);
        } else {
          mbar_arrive_expect_tx(&full[s], bytes);
          uint8_t* dst = smem + Lo::stage + static_cast<size_t>(s) * Lo::kStage;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (rows[i] < 0) continue;
            tma_load_2d(dst + i * Lo::kPage8, &tmk, 0, rows[i], &full[s]);
            tma_load_2d(dst + (4 + i) * Lo::kPage8, &tmv, 0, rows[i], &full[s]);
            if (TS) {  // the page's 16 K and 16 V scales (the row is a multiple of 16)
              float* sc = reinterpret_cast<float*>(smem + Lo::ssc) + (s * 4 + i) * 32;
              bulk_load(sc, p.ks + rows[i], 64, &full[s]);
              bulk_load(sc + 16, p.vs + rows[i], 64, &full[s]);
            }
          }
        }
      }
      __syncwarp();
    }
  } else if (warp >= kMmaWarp) {
    // ------------------------------------------------------------ MMA issuers
    // One elected lane per tile (warp kMmaWarp + t), in the tile's order
    // QK(0), QK(1), PV(0), QK(2), PV(1), ...: QK^T of tile block i once the
    // softmax has read the tile's S of block i - 1 (one S buffer), PV of
    // block i - 1 once its P is in (two P buffers, which the softmax reuses
    // only after the PV two blocks back).  A block's K / V buffer goes back
    // to the converters once both issuers have released it (kvdone counts
    // one commit of each, in block order).
    const int t = warp - kMmaWarp;
    if (lane == 0) {
      const uint32_t id_qk = idesc_f16(kRows, kKeys), id_pv = idesc_f16(kRows, DH);
      const uint32_t tm_t = tmem + t * kTileCols;  // S at +0, P buffers at +64 and +96, O at +128
      const int nI = je[t] - jb[t];
      bool ok = wait_or_abort(qready, 0u, abort_flag);
      int pv = 0;  // PVs issued (tile blocks)
      auto issue_pv = [&]() -> bool {
        const int i = pv, jp = jb[t] + i;
        if (!wait_or_abort(&pfull[2 * t + (i & 1)], static_cast<uint32_t>((i >> 1) & 1), abort_flag))
          return false;
        tc_fence_after();
        const uint32_t b_v = sbase + Lo::vt + (jp % kBufs) * Lo::vtBytes;
        const uint32_t a_pt = tm_t + kKeys + (i & 1) * (kKeys / 2);  // P: 8 columns per 16 tokens
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          // 16 tokens = two 8-row groups of V; B is MN-major (bit 16)
          mma_f16_ts(tm_t + 128, a_pt + kk * 8, sw128_desc_mn(b_v + kk * 2048),
                     id_pv | (1u << 16), (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&pdone[2 * t + (i & 1)]);  // the P buffer read, O updated
        mma_commit(&kvdone[jp % kBufs]);      // this tile is done with the K / V buffer
        ++pv;
        return true;
      };
      for (int j = 0; j < nblk && ok; ++j) {
        const int i = j - jb[t];
        if (j >= je[t]) {  // past the tile's blocks: its last PVs, in order, then release
          while (ok && pv < nI) ok = issue_pv();
          if (!ok) break;
        }
        // every conversion phase in order, used or not (kvdone needs this issuer's
        // release of each block; the next phase of a buffer needs it)
        ok = wait_or_abort(&conv[j % kBufs], static_cast<uint32_t>((j / kBufs) & 1), abort_flag);
        if (!ok) break;
        if (i < 0 || i >= nI) {
          mma_commit(&kvdone[j % kBufs]);  // a block the tile does not see: released at once
          continue;
        }
        if (i >= 1) {  // the softmax has read S of block i - 1
          ok = wait_or_abort(&sfree[t], static_cast<uint32_t>((i - 1) & 1), abort_flag);
          if (!ok) break;
        }
        tc_fence_after();
        const uint32_t b_k = sbase + Lo::k + (j % kBufs) * Lo::kBytes;
        const uint32_t a_q = sbase + Lo::q + t * Lo::qBytes;
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
          const uint32_t off_a = (ks >> 2) * (kRows * 128) + (ks & 3) * 32;
          const uint32_t off_b = (ks >> 2) * (kKeys * 128) + (ks & 3) * 32;
          mma_f16_ss(tm_t, sw128_desc(a_q + off_a), sw128_desc(b_k + off_b), id_qk, ks > 0 ? 1u : 0u);
        }
        mma_commit(&sfull[t]);
        if (i >= 1) ok = issue_pv();  // PV of block i - 1
      }
      while (ok && pv < nI) ok = issue_pv();
      if (!ok) fail();
      mma_commit(fin);  // completes when every MMA issued above (by both issuers) has
      if (!mbar_wait(fin, 0u)) fail();
    }
  } else if (warp >= kConvWarp) {
    // ------------------------------------------------------------ converters
    const int ct = tid - kConvWarp * 32;  // 0 .. 127
    auto wait_w = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(kFull, wait_or_abort(bar, parity, abort_flag));
    };
    // Block j's FP8 pages -> f16 K and V (token rows), buffer j % kBufs.
    auto convert = [&](int j) -> bool {
      const int s = j % S;
      if (!wait_w(&full[s], static_cast<uint32_t>((j / S) & 1))) return false;
      if (j >= kBufs && !wait_w(&kvdone[j % kBufs], static_cast<uint32_t>((j / kBufs - 1) & 1)))
        return false;  // the PVs of block j - kBufs (the buffer's last readers) are done
      // the stage's page flags, kept for the softmax of block j (the
      // producer rewrites the stage's flags once the stage is released)
      const uint32_t bmask = (pg_bad[s * 4] ? 1u : 0u) | (pg_bad[s * 4 + 1] ? 2u : 0u) |
                       (pg_bad[s * 4 + 2] ? 4u : 0u) | (pg_bad[s * 4 + 3] ? 8u : 0u);
      // for the softmax of block j (read after it waits for conv[j % kBufs])
      if (ct == 0) bufmask[j % kBufs] = bmask;
      const uint32_t stg = sbase + Lo::stage + s * Lo::kStage;
      const uint32_t kb = sbase + Lo::k + (j % kBufs) * Lo::kBytes;
      const uint32_t vb = sbase + Lo::vt + (j % kBufs) * Lo::vtBytes;
      const int tok_base = (p_begin + 4 * j) * kBS;
      // K: 16-byte chunk (token t, dims 16c .. 16c + 15) -> 32 bytes of f16
      constexpr int KCH = DH / 16;  // chunks per token row
      static_assert((kKeys * KCH) % 128 == 0 && ((kKeys / 8) * (DH / 4)) % 128 == 0, "whole passes");
#pragma unroll
      for (int it = 0; it < kKeys * KCH / 128; ++it) {  // fixed count: the loads go out together
        const int e = ct + 128 * it;
        const int t = e / KCH, c = e - t * KCH;
        const int pg = t >> 4, tr = t & 15;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (!(bmask >> pg & 1u))
          w = lds128(stg + pg * Lo::kPage8 + swz(page_off<C::kRow>(tr, 16 * c), C::kSwz));
        uint32_t h[8];
        fp8x4_to_f16x2x2<FMT>(w.x, h[0], h[1]);
        fp8x4_to_f16x2x2<FMT>(w.y, h[2], h[3]);
        fp8x4_to_f16x2x2<FMT>(w.z, h[4], h[5]);
        fp8x4_to_f16x2x2<FMT>(w.w, h[6], h[7]);
        sts128(kb + sw128_off(t, 16 * c, kKeys), h[0], h[1], h[2], h[3]);
        sts128(kb + sw128_off(t, 16 * c + 8, kKeys), h[4], h[5], h[6], h[7]);
      }
      // V token-major like K (the MN-major B operand of PV); tokens past the
      // sequence or in masked pages are zero (p = 0 would not clear a NaN)
#pragma unroll
      for (int it = 0; it < kKeys * KCH / 128; ++it) {
        const int e = ct + 128 * it;
        const int t = e / KCH, c = e - t * KCH;
        const int pg = t >> 4, tr = t & 15;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (!(bmask >> pg & 1u) && tok_base + t < L)
          w = lds128(stg + (4 + pg) * Lo::kPage8 + swz(page_off<C::kRow>(tr, 16 * c), C::kSwz));
        uint32_t h[8];
        fp8x4_to_f16x2x2<FMT>(w.x, h[0], h[1]);
        fp8x4_to_f16x2x2<FMT>(w.y, h[2], h[3]);
        fp8x4_to_f16x2x2<FMT>(w.z, h[4], h[5]);
        fp8x4_to_f16x2x2<FMT>(w.w, h[6], h[7]);
        sts128(vb + sw128_off(t, 16 * c, kKeys), h[0], h[1], h[2], h[3]);
        sts128(vb + sw128_off(t, 16 * c + 8, kKeys), h[4], h[5], h[6], h[7]);
      }
      if (TS) {  // the block's scales, for the softmax: 0 for masked pages and tokens past L
        const int t = ct & 63, kv = ct >> 6, pg = t >> 4;
        const float* sc = reinterpret_cast<const float*>(smem + Lo::ssc) + (s * 4 + pg) * 32;
        const bool in = !(bmask >> pg & 1u) && tok_base + t < L;
        reinterpret_cast<float*>(smem + Lo::bsc)[(j % kBufs) * 128 + ct] = in ? sc[kv * 16 + (t & 15)] : 0.f;
      }
      fence_proxy_async_smem();  // generic writes -> the tensor core's reads
      mbar_arrive(&conv[j % kBufs]);
      mbar_arrive(&empty[s]);
      return true;
    };

    for (int j = 0; j < nblk; ++j)
      if (!convert(j)) {
        fail();
        break;
      }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;   // this warp group's tile
    const int r = tid & 127;   // row = TMEM lane
    const int jr = j0 + t * TQ + r / p.G;
    const bool live = t < p.tpc && jr < n;
    const int pos = live ? base + jr : -1;
    const int lo = live ? window_lo(p.window, pos + 1) : 0;
    const int64_t qrow = live ? static_cast<int64_t>(q0 + jr) * p.Hq + gkv * p.G + r % p.G : -1;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tm_s = tmem + lane_base + t * kTileCols;  // S of this tile (P buffers at +64, +96)
    const uint32_t tm_o = tm_s + 128;                          // O of this tile

    // FP8-domain query: the row's head scale sQ; the row's codes enc(q / sQ)
    const float sq = p.qs ? __ldg(p.qs + (p.q_per_head ? gkv * p.G + r % p.G : 0)) : 1.f;
    // Q row r -> f16 into the tile's A tile (under KVQ_Q_FP8 the decoded codes, exact)
    {
      const bool ok = live && guard(qrow < p.total_q * p.Hq, p.status, 23);
      const uint4* src = reinterpret_cast<const uint4*>(p.q + (ok ? qrow : 0) * DH);
#pragma unroll
      for (int c = 0; c < DH / 8; ++c) {
        const uint4 v = ok ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (p.qs)
            h[i] = fp8x2_to_f16x2<FMT>(f32x2_to_fp8x2<FMT>(__fdiv_rn(bf16lo_to_f32(w[i]), sq),
                                                           __fdiv_rn(bf16hi_to_f32(w[i]), sq)));
          else
            h[i] = f32x2_to_f16x2(bf16lo_to_f32(w[i]), bf16hi_to_f32(w[i]));
        }
        sts128(sbase + Lo::q + t * Lo::qBytes + sw128_off(r, 8 * c, kRows), h[0], h[1], h[2], h[3]);
      }
    }
    // per-(token, head) scales multiply each key's logit and each value's
    // probability inside the loop; the fixed factors here
    const float sk = TS ? 1.f : __ldg(p.ks + (p.per_head ? gkv : 0));
    const float sv = TS ? 1.f : __ldg(p.vs + (p.per_head ? gkv : 0));
    const float lscale = sk * sq * p.logit_scale;
    // Per-(token, head) V scales: P's columns carry 2^7 sV_t / sigma, sigma a
    // power of two at least the largest sV_t so far, so P stays <= 2^15 in
    // f16 while the keys with small sV_t / sigma keep their precision (out of
    // f16's subnormal range down to 2^-21); the epilogue takes the 2^7 off.
    // When a block raises sigma, O is rescaled with the running maximum.
    float sigma = 0.f;

    // Waits of this role are warp-uniform (the TMEM accesses after them are
    // warp-collective).
    auto wait_w = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(kFull, wait_or_abort(bar, parity, abort_flag));
    };
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    fence_proxy_async_smem();  // the Q tile -> the tensor core
    mbar_arrive(qready);
    const int nI = je[t] - jb[t];  // this tile's blocks
    for (int i = 0; i < nI && ok; ++i) {
      const int j = jb[t] + i;
      if (!wait_w(&sfull[t], static_cast<uint32_t>(i & 1))) {
        ok = false;
        break;
      }
      // the block's masked pages (the converters wrote them before conv[j % kBufs])
      if (!wait_w(&conv[j % kBufs], static_cast<uint32_t>((j / kBufs) & 1))) {
        ok = false;
        break;
      }
      const uint32_t bm = bufmask[j % kBufs];
      tc_fence_after();
      float x[kKeys];
      {
        float t0[32], t1[32];
        tmem_ld32(tm_s, t0);
        tmem_ld32(tm_s + 32, t1);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          x[e] = t0[e];
          x[32 + e] = t1[e];
        }
      }
      tc_fence_before();
      mbar_arrive(&sfree[t]);  // S read: the next QK^T may overwrite it
      const int kb0 = (p_begin + 4 * j) * kBS;
      const float* bsc = reinterpret_cast<const float*>(smem + Lo::bsc) + (j % kBufs) * 128;
      float sig_new = sigma;
      if (TS) {  // sK of each key (0 where masked); sigma over the block's sV
        float vm = 0.f;
#pragma unroll
        for (int e = 0; e < kKeys; e += 4) {
          const float4 k4 = *reinterpret_cast<const float4*>(bsc + e);
          const float4 v4 = *reinterpret_cast<const float4*>(bsc + kKeys + e);
          x[e] *= k4.x;
          x[e + 1] *= k4.y;
          x[e + 2] *= k4.z;
          x[e + 3] *= k4.w;
          vm = fmaxf(vm, fmaxf(fmaxf(v4.x, v4.y), fmaxf(v4.z, v4.w)));
        }
        if (vm > sigma) {  // the smallest power of two >= vm (vm itself when infinite)
          const uint32_t e = __float_as_uint(vm) & 0x7F800000u;
          sig_new = (__uint_as_float(e) == vm || e == 0x7F800000u) ? vm : __uint_as_float(e + 0x00800000u);
        }
      }
      // eight partial maxima: independent chains (max is exact in any order)
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
      if (live && bm == 0u && kb0 >= lo && kb0 + kKeys - 1 <= pos) {  // the row sees the block
#pragma unroll
        for (int e = 0; e < kKeys; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], x[e]);
      } else {
#pragma unroll
        for (int e = 0; e < kKeys; ++e) {
          const int kp = kb0 + e;
          const bool valid = live && kp >= lo && kp <= pos && !(bm >> (e >> 4) & 1u);
          x[e] = valid ? x[e] : -INFINITY;
          mx8[e & 7] = fmaxf(mx8[e & 7], x[e]);
        }
      }
      float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      // the logits are x * lscale (log2 units): the scale goes into the max
      // and into the exponent's fused multiply-add
      mx *= lscale;
      const bool grow = mx > m + kRescaleThreshold;
      // sigma is the same on every row (sV depends on the token and KV head)
      const bool rescale = __any_sync(kFull, grow) || sig_new != sigma;
      // Rescaling O waits for its last writer, the tile's PV of block i - 1.
      // (This role waits for every PV, two blocks back, before it rewrites
      // that PV's P buffer below; this extra wait comes after the one for
      // block i - 3 on the same barrier, so its parity wait is sound.)
      if (rescale && i >= 1 &&
          !wait_w(&pdone[2 * t + ((i - 1) & 1)], static_cast<uint32_t>(((i - 1) >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (rescale) {  // rescale O rows (warp-collective TMEM access)
        const float nm = grow ? mx : m;
        const float a = (m == -INFINITY) ? 0.f : fast_exp2(m - nm);
        // O holds sum p sV / sigma V: a larger sigma scales it by sigma / sigma_new
        const float ao = (sigma > 0.f && sig_new != sigma) ? a * (sigma / sig_new) : a;
        if (i >= 1) {  // 16 columns at a time (x is live here)
#pragma unroll 1
          for (int c = 0; c < DH; c += 16) {
            uint32_t o[16];
            tmem_ld16(tm_o + c, o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * ao);
            tmem_st16(tm_o + c, o);
          }
        }
        l *= a;
        m = nm;
        sigma = sig_new;
      }
      // P row -> f16 into P buffer i % 2 (the A operand of PV), 8 keys at a
      // time, once the PV of block i - 2 has read that buffer
      if (i >= 2 && !wait_w(&pdone[2 * t + (i & 1)], static_cast<uint32_t>(((i - 2) >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tm_p = tm_s + kKeys + (i & 1) * (kKeys / 2);
      float l4[4] = {0.f, 0.f, 0.f, 0.f};  // four partial sums of the block
      // 2^7 sV_t / sigma of each value (power-of-two factors: exact)
      const float isig = sigma > 0.f ? 128.f / sigma : 0.f;
#pragma unroll
      for (int c = 0; c < kKeys / 8; ++c) {
        uint32_t ph[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const int e = 8 * c + 2 * e2;
          // m = -inf only while every key so far is masked (this block's too)
          const float p0 = (m == -INFINITY) ? 0.f : fast_exp2(fmaf(x[e], lscale, -m));
          const float p1 = (m == -INFINITY) ? 0.f : fast_exp2(fmaf(x[e + 1], lscale, -m));
          l4[e2] += p0 + p1;
          if (TS)
            ph[e2] = f32x2_to_f16x2(p0 * (bsc[kKeys + e] * isig), p1 * (bsc[kKeys + e + 1] * isig));
          else
            ph[e2] = f32x2_to_f16x2(p0, p1);
        }
        tmem_st4(tm_p + 4 * c, ph[0], ph[1], ph[2], ph[3]);
      }
      l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&pfull[2 * t + (i & 1)]);
    }
    if (!ok) fail();
    // ---- epilogue: O row / l * sV -> bf16, after the tile's last PV
    bool eok = ok && nI > 0;
    if (eok) eok = wait_w(&pdone[2 * t + ((nI - 1) & 1)], static_cast<uint32_t>(((nI - 1) >> 1) & 1));
    if (eok) {
      tc_fence_after();
      const float f = l > 0.f ? (TS ? sigma * 0.0078125f : sv) / l : 0.f;
      const bool store = live && guard(qrow < p.total_q * p.Hq, p.status, 24);
#pragma unroll
      for (int c = 0; c < DH; c += 32) {
        float o[32];
        tmem_ld32(tm_o + c, o);
        if (store) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + qrow * DH + c);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(f32x2_to_bf16x2(o[8 * v] * f, o[8 * v + 1] * f),
                                f32x2_to_bf16x2(o[8 * v + 2] * f, o[8 * v + 3] * f),
                                f32x2_to_bf16x2(o[8 * v + 4] * f, o[8 * v + 5] * f),
                                f32x2_to_bf16x2(o[8 * v + 6] * f, o[8 * v + 7] * f));
        }
      }
    } else if (ok && nI > 0) {
      fail();
    }
  }

  tc_fence_before();
  __syncthreads();
  // After an abort: wait (bounded) for the page copies still in flight and
  // for the MMAs (the MMA lane waited for its own), then free the TMEM.
  if (*abort_flag && tid == 0) {
    for (int s = 0; s < S; ++s)
      if (issued[s] >= 0) mbar_wait(&full[s], static_cast<uint32_t>((issued[s] / S) & 1));
  }
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace tc
}  // namespace kvq
