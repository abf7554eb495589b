// Sequence-sharded MLA decode: per-shard partial attention on tcgen05, bf16
// caches (fp8 caches: partial_fp8.cu).
//
// Computes, for every (request b, shard s, group of 64 query rows), the
// attention of the absorbed queries over the shard's slice of the paged
// latent cache and emits the normalised partial output o_s and its
// log-sum-exp lse_s ("Decode Context Parallelism", sections 4.1 and 5.3:
// each rank attends over its local latent slice; partial outputs and LSEs are
// merged afterwards).
//
// Data flow per persistent CTA (one per SM, 256 threads):
//   warp 0      producer: block-table lookups; TMA loads of the query group
//               (64 rows x 576, once per piece) and of 64-token KV tiles
//               (one box per page and chunk group, 128-byte swizzle) into
//               two stages; each chunk group of a stage is refilled as soon
//               as the P.V blocks that read it are done.
//               The next tile of the piece is prefetched into L2 (TMA
//               prefetch, no shared memory) when a tile's load is issued:
//               the two stages alone keep too few bytes in flight to cover
//               the DRAM latency.
//
// Stage layout: the nine 64-wide chunks of a row form three chunk groups
// (chunks 3c..3c+2 in group c, 24576 bytes each); inside a chunk group,
// token slot a lies in 8-slot group a/8 at byte (a/8)*3072 + (c%3)*1024 +
// (a%8)*128 for chunk c, so each 8-row x 128-byte swizzle atom is whole.  The
// MMAs only need a uniform stride between 8-row groups (3072 bytes), and a
// page's slots of one interleaved shard are whole groups, so one TMA box
// brings a chunk group of a page's slots: 3N boxes per tile for N
// interleaved shards.  Each chunk group of a stage has its own barrier, and
// QK^T starts on the first chunk group while the others are in flight, which
// shortens the time a stage is held after its last byte lands.
//   warps 1, 6  QK^T issuers: each issues half of S = Q K^T (M=64 rows, N=64
//               tokens; two of the four K16 steps of every 64-wide chunk of
//               K=576, into two TMEM accumulators that the softmax adds), a
//               chunk group at a time as each lands.  One thread issues a
//               tcgen05.mma about every 40 cycles, so these small MMAs need
//               several issuing warps.
//   warp 7      P.V issuer: latent blocks 0..3 of O^T += V^T P^T in order
//               (M=128 latent dims, N=rows, K=64 tokens) the moment the
//               tile's probabilities are ready, into a TMEM accumulator of
//               4 x 64 columns; chunk group c of the stage is free once
//               block c + 1 is done.
//   warps 2..5  softmax: two threads per query row (32 logits each) read S
//               from TMEM, mask, keep the running max / sum and write bf16
//               probabilities into the tile's own rope-chunk slot (free once
//               QK^T has read it), so P is double-buffered with the stages;
//               O^T is rescaled in TMEM only when a running max grows by more
//               than 2^8; the epilogue writes o = O / l and lse = m + ln l.
//
// Work is a flat list of tiles over all units (stream-K): CTA c takes work
// positions [c*per, (c+1)*per).  A unit that lies wholly inside one CTA's range is
// written straight to out_partial; pieces of a split unit go to workspace
// slots and are merged by mla_merge_kernel.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "common.cuh"
#include "host_util.h"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kThreads = 256;
constexpr int kIssuers = 2;                // QK^T-issuing warps (1 and 6)
constexpr int kPvIssuers = 1;              // P.V-issuing warp (7): the four latent blocks in order
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kBarSoftmax = 1;        // named barrier id for the softmax warps
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kSoftmaxWarps = 4;
constexpr int kPrefetch = 1;               // tiles of a piece prefetched into L2 ahead of the stage loads

struct Misc {
  uint64_t kv_full[2 * 3], kv_empty[2 * 3];   // per stage, one per chunk group
  uint64_t s_full[2], s_empty[2];
  // per-stage barriers: the softmax may run up to two tiles ahead of P.V, so a
  // single barrier could complete two phases between tests and alias parities
  uint64_t p_full[2], pv_done[2];
  uint64_t q_full, q_empty, o_free;
  uint64_t drain;                         // teardown after a failure: MMAs in flight
  uint32_t tmem_base;
  int abort;
  float alpha[2][kRows];  // by tile parity: a warp may be one tile ahead of another
  alignas(16) float inv_l[kRows];
  uint32_t orow[kRows];   // epilogue: destination row of each of the group's rows
};

constexpr int kSmemQ = 0;
constexpr int kSmemKV = kTileBytes;
// A stage holds three chunk groups of three 64-wide chunks each
// (chunks 3c..3c+2 in group c); inside a chunk group, 8-slot group a/8 of
// the tile lies at (a/8)*3072, chunk at +1024*(chunk%3), slot at +128*(a%8).
constexpr int kCg = kChunks / kCgChunks;             // chunk groups per tile
constexpr int kGroupBytes = kCgChunks * 1024;        // 3072: one 8-slot group of a chunk group
constexpr int kCgBytes = 8 * kGroupBytes;            // 24576: one chunk group of a tile
static_assert(kTileBytes == kCg * kCgBytes, "tile = 3 chunk groups");
// byte offset of 64-wide chunk c (of 8-slot group 0) inside a stage
__host__ __device__ constexpr int chunk_off(int c) { return (c / kCgChunks) * kCgBytes + (c % kCgChunks) * 1024; }
constexpr int kGroupRope = chunk_off(kChunks - 1);   // rope chunk (P after QK^T)
constexpr int kSmemMisc = 3 * kTileBytes;
constexpr int kSmemBytes = kSmemMisc + 2048 + 1024;  // + misc + alignment slack
static_assert(sizeof(Misc) <= 2048, "misc block");
static_assert(offsetof(Misc, inv_l) % 16 == 0, "inv_l is read as float4");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// TMEM columns: per stage two partial S accumulators (M=64 layout, 64
// columns each: stage st, issuer i at 128*st + 64*i), then four O^T blocks.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColO = 256;

__device__ __forceinline__ void set_error(PartialParams& p, Misc* misc, unsigned bits) {
  atomicOr(&p.hdr->err, bits);
  if (bits & kErrTimeout) *(volatile int*)&misc->abort = 1;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace

template <int kLocal, bool kRankIo, bool kJoin12>
__global__ void __launch_bounds__(kThreads, 1)
    mla_partial_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_kv,
                       const __grid_constant__ CUtensorMap tm_kv_pf, PartialParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, formed by pointer arithmetic on the shared array
  // (not through an integer) so that the compiler keeps every access through
  // it in the shared state space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Misc* misc = reinterpret_cast<Misc*>(smem + kSmemMisc);
  const ProblemDesc& pd = p.pd;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();                // the planning kernel's work list
  griddep_launch_dependents();

  const int W = p.hdr->total_cost, per = p.hdr->per_cta;
  const int lo = blockIdx.x * per;
  if (lo >= W) return;
  const int hi = min(lo + per, W);
  const int U = p.hdr->num_units;

  const uint32_t sQ = smem_u32(smem + kSmemQ);
  const uint32_t sKV = smem_u32(smem + kSmemKV);
  // barrier addresses: the two stages' barriers are 8 bytes apart
  const uint32_t b_kv_full = smem_u32(&misc->kv_full[0]);
  const uint32_t b_kv_empty = smem_u32(&misc->kv_empty[0]);
  const uint32_t b_s_full = smem_u32(&misc->s_full[0]);
  const uint32_t b_s_empty = smem_u32(&misc->s_empty[0]);
  const uint32_t b_q_full = smem_u32(&misc->q_full), b_q_empty = smem_u32(&misc->q_empty);
  const uint32_t b_p_full = smem_u32(&misc->p_full[0]), b_pv_done = smem_u32(&misc->pv_done[0]);
  const uint32_t b_o_free = smem_u32(&misc->o_free);
  volatile int* abort_flag = &misc->abort;

  if (threadIdx.x == 0) {
    for (int st = 0; st < 2; ++st) {
      for (int cg = 0; cg < kCg; ++cg) {
        mbar_init(b_kv_full + 8 * (kCg * st + cg), 1);
        mbar_init(b_kv_empty + 8 * (kCg * st + cg), 1);
      }
      mbar_init(b_s_full + 8 * st, kIssuers);
      mbar_init(b_s_empty + 8 * st, kSoftmaxWarps);
      mbar_init(b_p_full + 8 * st, kSoftmaxWarps);
      mbar_init(b_pv_done + 8 * st, kPvIssuers);
    }
    mbar_init(b_q_full, 1);
    mbar_init(b_q_empty, kIssuers);
    mbar_init(b_o_free, kSoftmaxWarps);
    mbar_init(smem_u32(&misc->drain), kIssuers + kPvIssuers);
    misc->abort = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < kRows) misc->alpha[0][threadIdx.x] = misc->alpha[1][threadIdx.x] = 1.0f;
  if (warp == 1) {
    tmem_alloc(smem_u32(&misc->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kv);
    tma_prefetch_desc(&tm_kv_pf);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  const uint64_t tmo = p.timeout_ns;

  PieceIter it;
  it.init(p.prefix, U, lo, hi, p.hdr->unit_cost);
  // producer: last armed phase per chunk-group barrier of each stage
  int armed_kv[2][kCg] = {{-1, -1, -1}, {-1, -1, -1}}, armed_q = -1;
  int unit, t0, t1, slot;
  bool whole;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lane k < nv issues the boxes of page k of the tile; lane 0 arms each
    // group barrier with the group's whole byte count first.
    // page boxes per tile: the shard's rows of ppt pages for interleaved
    // shards of a global cache (ppt = N when N divides 64), otherwise one
    // whole page
    const int nv = (pd.layout == kInterleaved && kLocal != 1) ? pd.ppt : 1;
    const int box_bytes = kCgBytes / nv;     // one chunk group of one page's slots
    int gt = 0, pc = 0;
    bool ok = true;
    while (ok && it.next(unit, t0, t1, whole, slot)) {
      Unit x = make_unit<kLocal>(pd, unit);
      const int npages_b = kLocal == 1 ? x.tiles : ceil_div(x.L, kPage);   // block-table entries
      const int32_t* bt = pd.block_table + (size_t)x.b * pd.max_pages;
      const int res = nv > 1 ? x.s : 0;
      int win_base = -1, win_val = -1;
      int pwin_base = -1, pwin_val = -1;   // block-table window of the L2 prefetches
      for (int j = t0; j < t1 && ok; ++j, ++gt) {
        const int st = gt & 1;
        // L2 prefetch of the piece's tiles up to kPrefetch ahead: with two
        // stages, an SM's own loads keep too few bytes in flight to cover
        // the DRAM latency; a stage load then reads L2
        for (int jp = (j == t0 ? j + 1 : j + kPrefetch); jp <= j + kPrefetch && jp < t1; ++jp) {
          const int fs = nv > 1 ? jp * nv : (kLocal == 1 || pd.layout == kInterleaved ? jp : x.p0 + jp);
          const int pwb = fs & ~31;
          if (pwb != pwin_base && fs < npages_b) {
            pwin_base = pwb;
            const int e = pwb + lane;
            pwin_val = (e < npages_b && e < pd.max_pages) ? __ldg(bt + e) : -1;
          }
          const int pidx = fs + lane;
          const int pg = __shfl_sync(0xffffffffu, pwin_val, pidx & 31);
          // one box per page: the prefetch needs no chunk-group barriers,
          // and every TMA box costs issue throughput
          if (lane < nv && pidx < npages_b && pg >= 0 && pg < pd.num_pages && kLocal != 2)
            tma_prefetch_l2_5d(&tm_kv_pf, 0, 0, 0, 0, pg * kPage + res);
        }
        // page slot of this lane's box; nv divides 32, so a tile never
        // straddles two 32-entry windows of the block table
        const int first_slot = nv > 1 ? j * nv : (kLocal == 1 || pd.layout == kInterleaved ? j : x.p0 + j);
        const int wb = first_slot & ~31;
        if (wb != win_base && first_slot < npages_b) {
          win_base = wb;
          const int e = wb + lane;
          win_val = (e < npages_b && e < pd.max_pages) ? __ldg(bt + e) : -1;
        }
        const int idx = first_slot + lane;
        int page = __shfl_sync(0xffffffffu, win_val, idx & 31);
        if (lane < nv && idx < npages_b && (page < 0 || page >= pd.num_pages)) {
          set_error(p, misc, kErrBadPage);
          page = pd.num_pages;
        }
        if (idx >= npages_b) page = pd.num_pages;  // past the context: TMA fills zeros
        // The chunk groups go out in order, each once the P.V that read its
        // previous contents is done and each on its own full barrier, so the
        // first chunk groups of a tile land while the last P.V blocks of the
        // tile two back still run, and QK^T starts on them early.
        const uint32_t full = b_kv_full + 8 * kCg * st;
        const uint32_t empty = b_kv_empty + 8 * kCg * st;
        // N does not divide 64: lane k*gpp + g (gpp = 8-slot groups per page)
        // loads group g of page k of the tile, rows r_k + 8 N g + N i (i < 8)
        // of the (64 dims, row in page, chunk, page) view with traversal
        // stride N along the rows, so rows past the page's end are out of
        // the view and fill zeros.  One box is one 8-slot group of a chunk
        // group (3072 bytes).
        int r0 = 0, pgk = 0;
        if (kLocal == 2) {
          const int gpp_log2 = pd.spp_log2 - 3;
          const int k = lane >> gpp_log2, g = lane & ((1 << gpp_log2) - 1);
          pgk = __shfl_sync(0xffffffffu, page, k & 31);
          r0 = shard_row0(x.s, first_slot + k, pd.num_shards) + 8 * pd.num_shards * g;
        }
        auto issue_cg = [&](int cg) {
          if (kLocal == 2) {
            if (lane < 8)
              tma_load_4d(sKV + st * kTileBytes + cg * kCgBytes + lane * kGroupBytes, &tm_kv,
                          full + 8 * cg, 0, r0, kCgChunks * cg, pgk);
          } else if (lane < nv) {
            // cache row page*64 + res of the (row-in-group, chunk, group,
            // row) view; a page of num_pages is out of range and fills zeros
            tma_load_5d(sKV + st * kTileBytes + cg * kCgBytes + lane * box_bytes, &tm_kv,
                        full + 8 * cg, 0, 0, kCgChunks * cg, 0, page * kPage + res);
          }
        };
        auto wait_free = [&](int cg) {
          return gt < 2 || __all_sync(0xffffffffu, mbar_wait(empty + 8 * cg, ((gt >> 1) - 1) & 1,
                                                             tmo, abort_flag));
        };
        if (kJoin12) {
          // Every wait costs the producer a wake-up before its boxes go out;
          // with four or more boxes per chunk group, chunk groups 1 and 2 go
          // out together after one wait.  Chunk group 0's release implies
          // that tile gt - 2 landed whole (its QK^T is done), so all three
          // full barriers are armed at once.
          ok = wait_free(0);
          if (!ok) break;
          if (lane == 0) {
#pragma unroll
            for (int cg = 0; cg < kCg; ++cg) mbar_arrive_expect_tx(full + 8 * cg, kCgBytes);
          }
          __syncwarp();
          issue_cg(0);
          if (lane == 0) armed_kv[st][0] = gt;   // the teardown drains issued copies only
          // chunk group 2's release implies chunk group 1's: one thread
          // issues the P.V blocks and their commits in order
          ok = wait_free(2);
          if (ok) {
            issue_cg(1);
            issue_cg(2);
            if (lane == 0) armed_kv[st][1] = armed_kv[st][2] = gt;
          }
          __syncwarp();
        } else {
#pragma unroll 1
          for (int cg = 0; cg < kCg; ++cg) {
            ok = wait_free(cg);
            if (!ok) break;
            if (lane == 0) {
              mbar_arrive_expect_tx(full + 8 * cg, kCgBytes);
              armed_kv[st][cg] = gt;
            }
            __syncwarp();
            issue_cg(cg);
            __syncwarp();
          }
        }
        if (!ok) break;
        if (ok && j == t0) {
          // query rows of this unit: reuse of the buffer waits for the last
          // QK^T of the previous piece
          if (pc >= 1) {
            ok = __all_sync(0xffffffffu, mbar_wait(b_q_empty, (pc - 1) & 1, tmo, abort_flag));
            if (!ok) break;
          }
          const bool load_q = !(p.withhold_query && pc == 0);
          if (lane == 0 && load_q) {
            mbar_arrive_expect_tx(b_q_full, kTileBytes);
            armed_q = pc;
          }
          __syncwarp();
          if (kRankIo && load_q) {
            // rank-major gathered query: lane k loads run k (one rank's heads
            // of one query position), chunk by chunk
            const int run = q_run_rows(pd);
            if (lane < kRows / run) {
              const int src = q_src_row(pd, x, lane * run);
#pragma unroll
              for (int c = 0; c < kChunks; ++c)
                tma_load_2d(sQ + c * kChunkBytes + lane * run * 128, &tm_q, b_q_full, c * 64, src);
            }
          } else if (lane == 0 && load_q) {
            const int row0 = x.b * pd.R + x.g * kRows;
            if (p.q_one_box) {
              tma_load_3d(sQ, &tm_q, b_q_full, 0, row0, 0);
            } else {
#pragma unroll
              for (int c = 0; c < kChunks; ++c)
                tma_load_2d(sQ + c * kChunkBytes, &tm_q, b_q_full, c * 64, row0);
            }
          }
          __syncwarp();
        }
      }
      ++pc;
    }
    if (!ok && lane == 0) set_error(p, misc, kErrTimeout);
  } else if (warp == 1 || warp == 6) {
    // ------------------------------------------------------------ QK^T issue
    const int mi = warp == 6 ? 1 : 0;
    const uint32_t id_qk = idesc_bf16_f32(64, 64, false, false);
    const uint64_t dq0 = sw128_desc(sQ, 16, 1024);
    const uint64_t dkv0 = sw128_desc(sKV, 16, kGroupBytes);
    int gbase = 0, pc = 0;
    bool ok = true;
    while (ok && it.next(unit, t0, t1, whole, slot)) {
      ok = __all_sync(0xffffffffu, mbar_wait(b_q_full, pc & 1, tmo, abort_flag));
      for (int j = t0; ok && j < t1; ++j) {
        const int g = gbase + (j - t0);
        const int st = g & 1;
        if (g >= 2) {
          ok = __all_sync(0xffffffffu, mbar_wait(b_s_empty + 8 * st, ((g >> 1) - 1) & 1, tmo,
                                                 abort_flag));
          if (!ok) break;
        }
        const uint32_t st_off = (uint32_t)(st * kTileBytes) >> 4;
        const uint32_t d = tmem + kColS0 + 128 * st + 64 * mi;
        // issuer mi takes K16 steps 2mi, 2mi+1 of every chunk, chunk group by
        // chunk group as each lands
#pragma unroll
        for (int cg = 0; cg < kCg; ++cg) {
          ok = __all_sync(0xffffffffu, mbar_wait(b_kv_full + 8 * (kCg * st + cg), (g >> 1) & 1,
                                                 tmo, abort_flag));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int c = kCgChunks * cg; c < kCgChunks * (cg + 1); ++c) {
#pragma unroll
              for (int k = 2 * mi; k < 2 * mi + 2; ++k) {
                const uint32_t offq = (uint32_t)((c * kChunkBytes + 32 * k) >> 4);
                const uint32_t offk = (uint32_t)((chunk_off(c) + 32 * k) >> 4);
                mma_bf16_ss(d, dq0 + offq, dkv0 + st_off + offk, id_qk,
                            (c != 0 || k != 2 * mi) ? 1u : 0u);
              }
            }
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) {
          mma_commit(b_s_full + 8 * st);
          if (j == t1 - 1) mma_commit(b_q_empty);
        }
        __syncwarp();
      }
      gbase += t1 - t0;
      ++pc;
    }
    if (!ok && lane == 0) set_error(p, misc, kErrTimeout);
  } else if (warp == 7) {
    // ------------------------------------------------------------ P.V issue
    // One thread issues the four latent blocks of O^T += V^T P^T in order and
    // frees each chunk group of the stage as soon as the blocks reading it
    // are done: chunks 0-2 after block 1, chunks 3-5 after block 2, chunks
    // 6-8 (the probabilities in the rope slot included) after block 3.
    // V^T of latent block b: chunks 2b and 2b + 1, the two 64-dim swizzle
    // atoms of M, lie chunk_off(2b + 1) - chunk_off(2b) apart.
    const uint64_t dp0 = sw128_desc(sKV + kGroupRope, 16, kGroupBytes);
    int gbase = 0, pc = 0;
    bool ok = true;
    while (ok && it.next(unit, t0, t1, whole, slot)) {
      Unit x = make_unit<kLocal>(pd, unit);
      const uint32_t id_pv = idesc_bf16_f32(128, x.rows, true, false);
      for (int j = t0; ok && j < t1; ++j) {
        const int g = gbase + (j - t0);
        bool w = mbar_wait(b_p_full + 8 * (g & 1), (g >> 1) & 1, tmo, abort_flag);
        if (j == t0 && pc >= 1) w = w && mbar_wait(b_o_free, (pc - 1) & 1, tmo, abort_flag);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const int st = g & 1;
          const uint32_t st_off = (uint32_t)(st * kTileBytes) >> 4;
#pragma unroll
          for (int blk = 0; blk < 4; ++blk) {
            const uint64_t dv0 = sw128_desc(sKV + chunk_off(2 * blk),
                                            chunk_off(2 * blk + 1) - chunk_off(2 * blk), kGroupBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = dv0 + st_off + (uint32_t)((kk * 2 * kGroupBytes) >> 4);
              const uint64_t bd = dp0 + st_off + (uint32_t)((32 * kk) >> 4);
              mma_bf16_ss(tmem + kColO + 64 * blk, a, bd, id_pv, (j == t0 && kk == 0) ? 0u : 1u);
            }
            if (blk >= 1) mma_commit(b_kv_empty + 8 * (kCg * st + blk - 1));
          }
          mma_commit(b_pv_done + 8 * st);
        }
        __syncwarp();
      }
      gbase += t1 - t0;
      ++pc;
    }
    if (!ok && lane == 0) set_error(p, misc, kErrTimeout);
  } else {
    // ------------------------------------------------------------ softmax
    // Thread (quadrant, lane) owns query row r = 16*quad + lane%16 and the
    // 32 logits of half h = lane/16 of each tile (16x32bx2 TMEM loads).
    const int quad = warp & 3;           // TMEM lane quadrant this warp may access
    const int tid = threadIdx.x - 64;    // 0..127
    const int half = lane >> 4;
    const int r = 16 * quad + (lane & 15);
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
    int gt = 0, pc = 0;
    bool ok = true;
    while (ok && it.next(unit, t0, t1, whole, slot)) {
      Unit x = make_unit<kLocal>(pd, unit);
      const bool owner = r < x.rows;
      const int i_row = (x.g * kRows + r) / pd.H;           // query position of row r
      const int vis_limit = x.L - x.qn + i_row;              // causal: t <= vis_limit
      float m_run = -CUDART_INF_F, l_run = 0.0f;             // l_run: this half's sum
      for (int j = t0; j < t1; ++j, ++gt) {
        const int sb = gt & 1;
        const bool ok_s = __all_sync(
            0xffffffffu, ok && mbar_wait(b_s_full + 8 * sb, (gt >> 1) & 1, tmo, abort_flag));
        bool resc = false;
        uint32_t pk[16];
        const bool full = tile_full<kLocal>(pd, x, j);
        if (ok_s) {
          tc_fence_after();
          uint32_t sr[32], sr2[32];
          tmem_ld16x2_32(tmem + lane_off + kColS0 + 128 * sb, sr);
          tmem_ld16x2_32(tmem + lane_off + kColS0 + 128 * sb + 64, sr2);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_s_empty + 8 * sb);
          float s[32];
#pragma unroll
          for (int a = 0; a < 32; ++a) s[a] = __uint_as_float(sr[a]) + __uint_as_float(sr2[a]);
          if (!full) {
#pragma unroll
            for (int a = 0; a < 32; ++a) {
              int t = slot_token<kLocal>(pd, x, j, 32 * half + a);
              bool vis = slot_valid(pd, x, t) && (!pd.causal || t <= vis_limit);
              if (!vis) s[a] = -CUDART_INF_F;
            }
          }
          // tree reduction: independent partial maxima keep the chain short
          float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
          for (int a = 4; a < 32; a += 4) {
            m4[0] = fmaxf(m4[0], s[a]);
            m4[1] = fmaxf(m4[1], s[a + 1]);
            m4[2] = fmaxf(m4[2], s[a + 2]);
            m4[3] = fmaxf(m4[3], s[a + 3]);
          }
          float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float m_new = fmaxf(m_run, mx * pd.scale_log2);
          float alpha = 1.0f;
          if (m_new > m_run + kRescaleThreshold || (j == t0 && m_new > -CUDART_INF_F)) {
            alpha = (m_run == -CUDART_INF_F) ? 0.0f : ex2_approx(m_run - m_new);
            l_run *= alpha;
            m_run = m_new;
            resc = owner && (j != t0);
          }
          if (owner && half == 0) misc->alpha[gt & 1][r] = alpha;
          const float m_use = (m_run == -CUDART_INF_F) ? 0.0f : m_run;
          float ls4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int a = 0; a < 16; ++a) {
            const float p0 = ex2_approx(fmaf(s[2 * a], pd.scale_log2, -m_use));
            const float p1 = ex2_approx(fmaf(s[2 * a + 1], pd.scale_log2, -m_use));
            pk[a] = pack_bf16x2(p0, p1);
            ls4[a & 3] += p0 + p1;
          }
          l_run += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
        }
        // every softmax thread reaches the reduction, so a failed wait
        // anywhere in the group is seen by all of them at the same point;
        // the common case (no failure, no rescale) costs one barrier
        if (named_bar_or(kBarSoftmax, kSoftmaxThreads, resc || !ok_s)) {
          if (named_bar_or(kBarSoftmax, kSoftmaxThreads, !ok_s)) { ok = false; break; }
          // some row's running max grew: rescale O^T, which needs the
          // previous P.V to have landed
          const bool ok_pv = __all_sync(
              0xffffffffu, (gt == 0) || mbar_wait(b_pv_done + 8 * ((gt - 1) & 1),
                                                  ((gt - 1) >> 1) & 1, tmo, abort_flag));
          ok = ok_pv;
          if (!ok_pv) continue;  // caught by the next reduction (or the epilogue's)
          tc_fence_after();
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
#pragma unroll 1
            for (int h2 = 0; h2 < 2; ++h2) {
              uint32_t v[32];
              const uint32_t ta = tmem + lane_off + kColO + 64 * blk + 32 * h2;
              tmem_ld32(ta, v);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c)
                v[c] = __float_as_uint(__uint_as_float(v[c]) * misc->alpha[gt & 1][32 * h2 + c]);
              tmem_st32(ta, v);
            }
          }
          tmem_wait_st();
        }
        if (owner) {
          uint8_t* prow = smem + kSmemKV + (gt & 1) * kTileBytes + (r >> 3) * kGroupBytes +
                          kGroupRope + (r & 7) * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int ch = 4 * half + c;   // 16-byte chunk of the 128-byte row
            uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            *reinterpret_cast<uint4*>(prow + ((ch ^ (r & 7)) << 4)) = v;
          }
        }
        if (!full) {
          // zero V rows of slots that hold no valid token of this shard so
          // that garbage (even NaN) past the context end cannot reach O
          uint8_t* st = smem + kSmemKV + (gt & 1) * kTileBytes;
          for (int e = tid; e < kTile * 8 * 8; e += kSoftmaxThreads) {
            int a = e >> 6, plane = (e >> 3) & 7, ch = e & 7;
            int t = slot_token<kLocal>(pd, x, j, a);
            if (!slot_valid(pd, x, t))
              *reinterpret_cast<uint4*>(st + chunk_off(plane) + (a >> 3) * kGroupBytes +
                                        (a & 7) * 128 + ch * 16) =
                  make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_p_full + 8 * (gt & 1));
      }
      // ---------------------------------------------------------- epilogue
      const bool ok_e = __all_sync(
          0xffffffffu, ok && mbar_wait(b_pv_done + 8 * ((gt - 1) & 1), ((gt - 1) >> 1) & 1, tmo,
                                       abort_flag));
      if (named_bar_or(kBarSoftmax, kSoftmaxThreads, !ok_e)) { ok = false; break; }
      tc_fence_after();
      // destination rows: a whole unit's rows of out_partial (out_row:
      // row-major, or the DCP head slices), or this CTA's workspace slot for a
      // piece of a split unit; the store loop reads them from a table
      float* const obase = whole ? p.out_partial : p.ws_o;
      float* const lbase = whole ? p.lse_partial : p.ws_lse;
      const size_t sl = 2 * (size_t)blockIdx.x + slot;
      // whole units: row-major rows (out_row), or in the DCP head slices
      // scattered rows (kRankIo), whose destinations the store loop reads
      // from a table
      const size_t row0 = whole ? ((size_t)x.so * pd.B + x.b) * pd.R + (size_t)x.g * kRows
                                : sl * kRows;
      auto dst_row = [&](int row) -> size_t {
        return (kRankIo && whole) ? out_row(pd, x, row) : row0 + row;
      };
      if (kRankIo && tid < kRows) misc->orow[tid] = (uint32_t)dst_row(tid);
      const float l_tot = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
      if (owner && half == 0) {
        float lse = (l_tot > 0.0f) ? (m_run + __log2f(l_tot)) * 0.69314718055994530942f
                                   : -CUDART_INF_F;
        misc->inv_l[r] = (l_tot > 0.0f) ? 1.0f / l_tot : 0.0f;
        lbase[dst_row(r)] = lse;
      }
      if (whole) {
        // padding rows of a request with fewer query tokens: o = 0, lse = -inf
        // (pieces of a split unit leave them to the merge kernel)
        for (int e = tid; e < (x.rows_out - x.rows) * (kDv / 4); e += kSoftmaxThreads)
          reinterpret_cast<float4*>(obase + dst_row(x.rows + e / (kDv / 4)) * kDv)[e % (kDv / 4)] =
              make_float4(0.f, 0.f, 0.f, 0.f);
        for (int rr = x.rows + tid; rr < x.rows_out; rr += kSoftmaxThreads)
          lbase[dst_row(rr)] = -CUDART_INF_F;
      }
      named_bar_sync(kBarSoftmax, kSoftmaxThreads);
      // O^T block k/2, rows 32*(k%2).. of this thread's latent dim, two TMEM
      // loads in flight: the stores of one overlap the load of the next
      {
        const uint32_t o_base = tmem + lane_off + kColO;
        auto store32 = [&](int k, const uint32_t (&v)[32]) {
          const int dim = 128 * (k >> 1) + 32 * quad + lane;
          float il[32];
          const float4* il4 = reinterpret_cast<const float4*>(misc->inv_l + 32 * (k & 1));
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 t = il4[c4];
            il[4 * c4] = t.x;
            il[4 * c4 + 1] = t.y;
            il[4 * c4 + 2] = t.z;
            il[4 * c4 + 3] = t.w;
          }
          // DCP I/O: each aligned group of 8 rows has 8 consecutive
          // destination rows (a rank's heads are a multiple of 8), so the 32
          // rows take 4 base addresses from the table and every store an
          // immediate offset from one of them: a lookup per store sits on
          // the softmax warps' critical path (one warp per scheduler)
          float* b8[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            b8[q4] = kRankIo ? obase + (size_t)misc->orow[32 * (k & 1) + 8 * q4] * kDv + dim
                             : obase + (row0 + 32 * (k & 1) + 8 * q4) * kDv + dim;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int row = 32 * (k & 1) + c;
            if (row < x.rows) b8[c >> 3][(c & 7) * kDv] = __uint_as_float(v[c]) * il[c];
          }
        };
        uint32_t va[32], vb[32];
        tmem_ld32(o_base, va);
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
          tmem_ld32(o_base + 32 * (k + 1), vb);
          tmem_wait_ld();
          store32(k, va);
          if (k + 2 < 8) tmem_ld32(o_base + 32 * (k + 2), va);
          store32(k + 1, vb);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_o_free);
      named_bar_sync(kBarSoftmax, kSoftmaxThreads);  // inv_l reused by the next piece
      ++pc;
    }
    if (!ok && tid == 0) set_error(p, misc, kErrTimeout);
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // After a failure, let this CTA's own MMAs and TMA copies complete before
    // TMEM is freed and the CTA exits.  A commit tracks every earlier MMA of
    // its thread, so one commit per issuing thread drains them all.
    int never = 0;
    if (lane == 0 && (warp == 1 || warp == 6 || warp == 7)) {
      mma_commit(smem_u32(&misc->drain));
      mbar_wait(smem_u32(&misc->drain), 0, kDrainNs, &never);
    }
    if (warp == 0 && lane == 0) {
      for (int st = 0; st < 2; ++st)
        for (int cg = 0; cg < kCg; ++cg)
          if (armed_kv[st][cg] >= 0)
            mbar_wait(b_kv_full + 8 * (kCg * st + cg), (armed_kv[st][cg] >> 1) & 1, kDrainNs, &never);
      if (armed_q >= 0) mbar_wait(b_q_full, armed_q & 1, kDrainNs, &never);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int partial_smem_bytes() { return kSmemBytes; }

template <int kLocal, bool kRankIo, bool kJoin12>
static cudaError_t launch_partial(const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                                  const CUtensorMap& tm_kv_pf, const PartialParams& p, int grid,
                                  cudaStream_t stream) {
  const cudaError_t e =
      host::ensure_dynamic_smem(
          reinterpret_cast<const void*>(&mla_partial_kernel<kLocal, kRankIo, kJoin12>), kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr = pdl_attribute();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_partial_kernel<kLocal, kRankIo, kJoin12>, tm_q, tm_kv, tm_kv_pf,
                            p);
}

// The cache kind (whole requests, a local slice, or whole requests with
// interleaved shards whose count does not divide the page) is a template
// parameter: branching on it at run time cost about 2% on the bimodal batch.
// So is the producer's wait policy, set by the TMA boxes per chunk group: a
// whole-cache tile of N interleaved shards (N | 64) has N boxes per chunk
// group, one N ∤ 64 has eight, a contiguous or local tile one.
cudaError_t launch_partial_bf16(const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                                const CUtensorMap& tm_kv_pf, const PartialParams& p, int grid,
                                cudaStream_t stream) {
  // the DCP rank-major I/O (local caches only) is an instantiation of its own
  if (p.pd.rank_heads != 0)
    return launch_partial<1, true, false>(tm_q, tm_kv, tm_kv_pf, p, grid, stream);
  if (p.pd.local) return launch_partial<1, false, false>(tm_q, tm_kv, tm_kv_pf, p, grid, stream);
  if (p.pd.pad) return launch_partial<2, false, true>(tm_q, tm_kv, tm_kv_pf, p, grid, stream);
  const int boxes = p.pd.layout == kInterleaved ? p.pd.ppt : 1;
  return boxes >= 4 ? launch_partial<0, false, true>(tm_q, tm_kv, tm_kv_pf, p, grid, stream)
                    : launch_partial<0, false, false>(tm_q, tm_kv, tm_kv_pf, p, grid, stream);
}

}  // namespace mla
