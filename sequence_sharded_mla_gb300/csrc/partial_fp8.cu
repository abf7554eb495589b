// Sequence-sharded MLA decode over an fp8 latent cache: per-shard partial
// attention on the e4m3 tensor cores (tcgen05 kind::f8f6f4), straight from
// the cache's codes.
//
// Same computation as the bf16 kernel ("Decode Context Parallelism",
// sections 4.1 and 5.3: each rank attends over its local latent slice and
// emits the partial output and its log-sum-exp), with the cache held as OCP
// e4m3 codes plus one fp32 scale per token (K and V of token t are
// code * scale_t).  The MMAs read the codes as they came from memory: nothing
// is expanded, so a 64-token stage is 36 KB and four of them are in flight.
//
// Exactness.  Both other operands are carried as two-term e4m3 sums:
//   - the query: per row a power-of-two scale s_r puts max|q| in [128, 256);
//     q*s_r = hi + lo with hi = e4m3(q*s_r), lo = e4m3(q*s_r - hi).  That is
//     exact for every component with |q*s_r| >= 2^-2 and within 2^-10 (in
//     scaled units) below.  Q_hi and Q_lo are the 128 rows of one M=128 MMA
//     (row 2k: Q_hi of query row k, row 2k+1: its Q_lo), so S_hi and S_lo of
//     a query row land in adjacent TMEM lanes and the two threads reading
//     them exchange halves by shuffle; an M=64 MMA would cost the tensor core
//     as much as an M=128 one.
//   - the probabilities: with sigma_t = mant_t * 2^E_t (mant in [0.5, 1)),
//     the softmax keeps its running max over b_t = a_t + E_t, where a_t is
//     the log2-domain logit, so that P'_t = 2^(a_t - m) * sigma_t =
//     2^(b_t - m) * mant_t is at most 2^8; P'_t carries the value scale, and
//     the normaliser sums u_t = 2^(a_t - m).  P' = hi + lo as above
//     (relative error about 2^-8, like a bf16 P), and O^T += V^T P'^T is two
//     accumulating MMAs per 32-token step.
// The tensor cores accumulate in fp32.
//
// Shared memory (1024-byte aligned base):
//   Q            72 KB      the MMA's 128 rows (Q_hi, Q_lo of query rows 4G..4G+3
//                           interleaved) in 16 groups of 8, 4608 bytes each:
//                           [chunk c][8 rows][64 codes] with 64-byte swizzle; the
//                           piece's bf16 rows land here by TMA first (9216 bytes
//                           per 8 query rows, the same bytes as their two groups)
//                           and are split in place
//   stages       4 x 36 KB  group-major: slot a's 64-code chunk c at
//                           (a/8)*4608 + c*512 + (a%8)*64 (swizzled), one TMA box per page
//   P_lo         4 KB       [8-row group][8 rows][64 tokens]; P_hi goes into the
//                           stage's rope atoms once QK^T has read them
//   misc         barriers, token scales and their exponents, the softmax groups' exchange
//
// Warps: 0 producer (block table, TMA of the codes, cp.async of the scales,
// L2 prefetch of the next tiles); 1 issues QK^T (per pair of adjacent stages
// as one N=128 chain, else per tile) and then splits the unit's token scales
// into mantissa and exponent; 6 and 7 issue P.V, two latent blocks each
// (P_lo terms first, so the one P_lo buffer is freed early); 2..5 and 8..11
// are two softmax groups, two warps per SM sub-partition: group k takes
// tokens [32 k, 32 k + 32) of every tile (two threads per query row, 16
// tokens each), the groups exchange each row's tile maximum through shared
// memory,
// and group 1 also loads each piece's query by TMA and splits it into
// Q_hi / Q_lo in place.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "common.cuh"
#include "host_util.h"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kThreads = 384;
constexpr int kPvIssuers = 2;              // P.V-issuing warps (6, 7), two latent blocks each
constexpr int kStages = 4;
constexpr int kStageBytes = kTile * kDqk;        // 36864: codes of one 64-token tile
constexpr int kAtom = 512;                       // 8 rows x 64 bytes
constexpr int kGroupBytes = kChunks * kAtom;     // 4608: one 8-slot group, nine chunks
constexpr int kRopeAtom = 8 * kAtom;             // rope chunk of a group (P_hi after QK^T)
constexpr int kQGroupBytes = 2 * kChunks * kAtom;  // 9216: bf16 of 8 query rows (= 2 MMA row groups)
constexpr int kQAGroupBytes = kChunks * kAtom;     // 4608: one 8-row group of the MMA's 128 rows
constexpr int kQBytes = 8 * kQGroupBytes;          // 73728
constexpr int kSmemQ = 0;
constexpr int kSmemKV = kQBytes;                                 // 73728
constexpr int kSmemPlo = kSmemKV + kStages * kStageBytes;        // 221184
constexpr int kSmemMisc = kSmemPlo + 8 * kAtom;                  // 225280
constexpr int kMiscBytes = 6144;
constexpr int kSmemBytes = kSmemMisc + kMiscBytes + 1024;        // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr int kSoftmaxThreads = 256;        // both groups
constexpr int kSoftmaxWarps = 8;
constexpr int kConvThreads = 128;           // softmax group 1 splits the query
constexpr uint32_t kBarSoftmax = 1;         // all softmax threads
constexpr uint32_t kBarGroup0 = 2;          // group k: kBarGroup0 + k
constexpr uint32_t kBarConv = 4;            // the query split (group 1)
constexpr float kRescaleThreshold = 8.0f;  // log2 units: 2^(b_t - m) <= 2^8 keeps P' inside e4m3
constexpr int kPrefetch = 2;               // tiles of a piece prefetched into L2 ahead of the loads

struct Misc {
  uint64_t kv_full[kStages], kv_empty[kStages], prep[kStages];
  uint64_t s_full[2], s_empty[2], p_full[2], pv_done[2];
  uint64_t plo_free[2];  // the P_lo terms of a tile's P.V have completed (P_lo may be rewritten)
  uint64_t q_full, q_conv, q_empty, o_free;
  uint64_t drain;       // teardown after a failure: MMAs in flight
  uint32_t tmem_base;
  int abort;
  float alpha[2][kRows];        // per softmax group: the rescale factor of each row
  alignas(16) float inv_l[kRows];
  uint32_t orow[kRows];         // epilogue: destination row of each of the group's rows
  float qinv[kRows];            // 1 / the row's power-of-two query scale (split by group 1)
  float qsc[kRows];             // the row's power-of-two query scale s_r (0: padding row)
  float xmax[2][2][kRows];      // by tile parity and group: the row's max over the group's tokens
  float xl[2][kRows];           // per group: the row's sum over the group's tokens (epilogue)
  // per stage and token slot: the scale (cp.async target, then sanitised in
  // place) and the exponent E of its mantissa-exponent split, as a float
  alignas(16) float sigma[kStages][kTile];
  alignas(16) float lge[kStages][kTile];
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc block");

// TMEM: two S buffers of 128 columns (M=128, lane 2k = S_hi of query row k,
// lane 2k + 1 = its S_lo: a QK^T unit of one or two tiles, tile g at columns
// 64 (g & 1)), then the four 128-dim blocks of O^T (M=128, 64 columns each).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColO = 256;

__device__ __forceinline__ void set_error(PartialParams& p, Misc* misc, unsigned bits) {
  atomicOr(&p.hdr->err, bits);
  if (bits & kErrTimeout) *(volatile int*)&misc->abort = 1;
}

// Biased exponent that fixes a row's power-of-two query scale: s_r =
// 2^(134 - e) puts max|q| (exponent e) in [128, 256); clamped so that s_r and
// 1/s_r are normal floats.
__device__ __forceinline__ uint32_t row_scale_exp(uint32_t max_bits) {
  return min(max(max_bits >> 7, 8u), 254u);
}

}  // namespace

template <int kLocal, bool kRankIo>
__global__ void __launch_bounds__(kThreads, 1)
    mla_partial_fp8_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_kv, PartialParams p) {
  extern __shared__ uint8_t smem_raw[];
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
  const uint32_t sPlo = smem_u32(smem + kSmemPlo);
  const uint32_t b_kv_full = smem_u32(&misc->kv_full[0]);
  const uint32_t b_kv_empty = smem_u32(&misc->kv_empty[0]);
  const uint32_t b_prep = smem_u32(&misc->prep[0]);
  const uint32_t b_s_full = smem_u32(&misc->s_full[0]);
  const uint32_t b_s_empty = smem_u32(&misc->s_empty[0]);
  const uint32_t b_p_full = smem_u32(&misc->p_full[0]);
  const uint32_t b_pv_done = smem_u32(&misc->pv_done[0]);
  const uint32_t b_q_conv = smem_u32(&misc->q_conv), b_q_empty = smem_u32(&misc->q_empty);
  const uint32_t b_q_full = smem_u32(&misc->q_full);
  const uint32_t b_o_free = smem_u32(&misc->o_free);
  volatile int* abort_flag = &misc->abort;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(b_kv_full + 8 * st, 1 + 32);   // expect_tx arrival + one cp.async arrival per lane
      mbar_init(b_kv_empty + 8 * st, kPvIssuers);
      mbar_init(b_prep + 8 * st, 1);
    }
    for (int sb = 0; sb < 2; ++sb) {
      mbar_init(b_s_full + 8 * sb, 1);
      mbar_init(b_s_empty + 8 * sb, kSoftmaxWarps);
      mbar_init(b_p_full + 8 * sb, kSoftmaxWarps);
      mbar_init(b_pv_done + 8 * sb, kPvIssuers);
      mbar_init(smem_u32(&misc->plo_free[sb]), kPvIssuers);
    }
    mbar_init(b_q_full, 1);
    mbar_init(b_q_conv, kConvThreads / 32);
    mbar_init(b_q_empty, 1);
    mbar_init(b_o_free, kSoftmaxWarps);
    mbar_init(smem_u32(&misc->drain), 1 + kPvIssuers);   // the MMA-issuing threads
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  const uint64_t tmo = p.timeout_ns;

  PieceIter it;
  it.init(p.prefix, U, lo, hi, p.hdr->unit_cost);
  int armed_kv[kStages] = {-1, -1, -1, -1}, armed_q = -1;
  int unit, t0, t1, slot;
  bool whole;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // nv page boxes per tile: the shard's rows of ppt pages for interleaved
    // shards of a global cache (ppt = N when N divides 64), otherwise one
    // whole page.  Lane k < nv issues box k; every lane copies the scales of
    // token slots lane and lane + 32.
    const bool shard_rows = pd.layout == kInterleaved && kLocal != 1;
    const int nv = shard_rows ? pd.ppt : 1;
    const int lg_rows = shard_rows ? pd.spp_log2 : 6;   // log2(slots per page)
    const int rstride = shard_rows ? pd.num_shards : 1;  // cache rows between slots
    const int box_bytes = kStageBytes / nv;
    int gt = 0;
    bool ok = true;
    while (ok && it.next(unit, t0, t1, whole, slot)) {
      Unit x = make_unit<kLocal>(pd, unit);
      const int npages_b = kLocal == 1 ? x.tiles : ceil_div(x.L, kPage);
      const int32_t* bt = pd.block_table + (size_t)x.b * pd.max_pages;
      const int res = nv > 1 ? x.s : 0;
      int win_base = -1, win_val = -1;
      int pwin_base = -1, pwin_val = -1;   // block-table window of the L2 prefetches
      for (int j = t0; j < t1 && ok; ++j, ++gt) {
        const int st = gt & (kStages - 1);
        // L2 prefetch of the piece's tiles up to kPrefetch ahead (this shard's
        // rows of each page, and the lines of the page's token scales), so
        // that a stage load mostly reads L2
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
          if (lane < nv && pidx < npages_b && pg >= 0 && pg < pd.num_pages && kLocal != 2) {
            tma_prefetch_l2_5d(&tm_kv, 0, 0, 0, 0, pg * kPage + res);
            prefetch_l2(p.kv_scale + (size_t)pg * kPage);
            prefetch_l2(p.kv_scale + (size_t)pg * kPage + 32);
          }
        }
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
        const float* scale_src[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int a = lane + 32 * h;
          const int k = a >> lg_rows;
          const int pg = __shfl_sync(0xffffffffu, page, k);
          const int row = (kLocal == 2 ? shard_row0(x.s, first_slot + k, pd.num_shards) : res) +
                          (a & ((1 << lg_rows) - 1)) * rstride;
          // a slot past its page's rows holds no token: any valid address
          const bool okpg = first_slot + k < npages_b && pg >= 0 && pg < pd.num_pages &&
                            row < kPage;
          scale_src[h] = p.kv_scale + (okpg ? (size_t)pg * kPage + row : 0);
        }
        if (gt >= kStages) {
          ok = __all_sync(0xffffffffu, mbar_wait(b_kv_empty + 8 * st, ((gt >> 2) - 1) & 1, tmo,
                                                 abort_flag));
          if (!ok) break;
        }
        const uint32_t full = b_kv_full + 8 * st;
        if (lane == 0) {
          mbar_arrive_expect_tx(full, kStageBytes);
          armed_kv[st] = gt;
        }
        __syncwarp();
        if (kLocal == 2) {
          // N does not divide 64: lane k*gpp + g loads 8-slot group g of
          // page k, rows r_k + 8 N g + N i of the (64 codes, row in page,
          // chunk, page) view with traversal stride N along the rows: rows
          // past the page's end are out of the view and fill zeros
          const int gpp_log2 = pd.spp_log2 - 3;
          const int k = lane >> gpp_log2, g = lane & ((1 << gpp_log2) - 1);
          const int pgk = __shfl_sync(0xffffffffu, page, k & 31);
          if (lane < 8)
            tma_load_4d(sKV + st * kStageBytes + lane * kGroupBytes, &tm_kv, full, 0,
                        shard_row0(x.s, first_slot + k, pd.num_shards) + 8 * pd.num_shards * g,
                        0, pgk);
        } else if (lane < nv) {
          tma_load_5d(sKV + st * kStageBytes + lane * box_bytes, &tm_kv, full, 0, 0, 0, 0,
                      page * kPage + res);
        }
        cp_async_4(smem_u32(&misc->sigma[st][lane]), scale_src[0]);
        cp_async_4(smem_u32(&misc->sigma[st][lane + 32]), scale_src[1]);
        cp_async_mbar_arrive_noinc(full);
        __syncwarp();
      }
    }
    if (!ok && lane == 0) set_error(p, misc, kErrTimeout);
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK^T issue
    // One QK^T unit per pair of tiles (g even, both in the piece: the two
    // stages are adjacent, so the pair's 16 slot groups are 4608 bytes apart
    // and one N=128 MMA chain covers them), else per single tile (N=64).
    // Unit u accumulates into S buffer u & 1 (128 columns); tile g's logits
    // are its columns 64 (g & 1) ..
    const uint32_t id_qk1 = idesc_e4m3_f32(128, 64, false, false);
    const uint32_t id_qk2 = idesc_e4m3_f32(128, 128, false, false);
    // Q (A, K-major, 128 rows: Q_hi and Q_lo interleaved): 8-row groups 4608
    // bytes apart, chunks 512; K (B, K-major): 8-slot groups 4608 apart
    const uint64_t dq0 = sw64_desc(sQ, 16, kQAGroupBytes);
    const uint64_t dk0 = sw64_desc(sKV, 16, kGroupBytes);
    int gbase = 0, pc = 0, qu = 0;
    bool ok = true;
    while (ok && it.next(unit, t0, t1, whole, slot)) {
      ok = __all_sync(0xffffffffu, mbar_wait(b_q_conv, pc & 1, tmo, abort_flag));
      for (int j = t0; ok && j < t1;) {
        const int g = gbase + (j - t0);
        const bool pair = (g & 1) == 0 && j + 1 < t1;
        const int st = g & (kStages - 1), sb = qu & 1;
        bool w = mbar_wait(b_kv_full + 8 * st, (g >> 2) & 1, tmo, abort_flag);
        if (pair) w = w && mbar_wait(b_kv_full + 8 * (st + 1), ((g + 1) >> 2) & 1, tmo, abort_flag);
        if (qu >= 2) w = w && mbar_wait(b_s_empty + 8 * sb, ((qu >> 1) - 1) & 1, tmo, abort_flag);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t st_off = (uint32_t)(st * kStageBytes) >> 4;
          const uint32_t d = tmem + kColS0 + 128 * sb + (pair ? 0 : 64 * (g & 1));
          const uint32_t id = pair ? id_qk2 : id_qk1;
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const uint64_t aq = dq0 + (uint32_t)((c * kAtom + 32 * k) >> 4);
              const uint64_t bk = dk0 + st_off + (uint32_t)((c * kAtom + 32 * k) >> 4);
              mma_e4m3_ss(d, aq, bk, id, (c != 0 || k != 0) ? 1u : 0u);
            }
          }
          mma_commit(b_s_full + 8 * sb);
          if (j + (pair ? 2 : 1) >= t1) mma_commit(b_q_empty);
        }
        // while the MMAs run: the unit's token scales, which have landed with
        // its stages -- sanitised in place, and the exponent E of
        // sigma = mant * 2^E (mant in [0.5, 1)) as a float
        for (int tt = 0; tt < (pair ? 2 : 1); ++tt) {
          const int sst = (g + tt) & (kStages - 1);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int a = lane + 32 * h;
            float sg = misc->sigma[sst][a];
            uint32_t bits = __float_as_uint(sg);
            uint32_t eb = (bits >> 23) & 0xFFu;
            if (eb < 27u) {
              // zero, subnormal or below 2^-100: as 2^-60 (its values are
              // negligible next to any normal token's, its logit ~0)
              sg = copysignf(8.6736174e-19f, sg);
              bits = __float_as_uint(sg);
              eb = (bits >> 23) & 0xFFu;
            }
            // inf, NaN or >= 2^126: exponent 0 and the value itself as the
            // scale, which propagates as the dequantised values would
            misc->sigma[sst][a] = sg;
            misc->lge[sst][a] = eb >= 253u ? 0.0f : (float)((int)eb - 126);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(b_prep + 8 * sst);
        }
        __syncwarp();
        ++qu;
        j += pair ? 2 : 1;
      }
      gbase += t1 - t0;
      ++pc;
    }
    if (!ok && lane == 0) set_error(p, misc, kErrTimeout);
  } else if (warp == 6 || warp == 7) {
    // ------------------------------------------------------------ P.V issue
    // O^T (4 blocks of 128 dims) += V^T P'^T per tile: V^T (A, MN-major)
    // 64-dim blocks 512 bytes apart, 8-token groups 4608; P_hi in the
    // groups' rope atoms, P_lo in its buffer (B, K-major).  Warp 6 issues
    // latent blocks 0, 1 and warp 7 blocks 2, 3; each issues its P_lo terms
    // first and commits them to plo_free, so the softmax may write the next
    // tile's P_lo (one buffer) while the P_hi terms still run.
    const int blk0 = warp == 6 ? 0 : 2;
    const uint64_t dv0 = sw64_desc(sKV, kAtom, kGroupBytes);
    const uint64_t dph0 = sw64_desc(sKV + kRopeAtom, 16, kGroupBytes);
    const uint64_t dpl = sw64_desc(sPlo, 16, kAtom);
    int gbase = 0, pc = 0;
    bool ok = true;
    while (ok && it.next(unit, t0, t1, whole, slot)) {
      Unit x = make_unit<kLocal>(pd, unit);
      const uint32_t id_pv = idesc_e4m3_f32(128, x.rows, true, false);
      for (int j = t0; ok && j < t1; ++j) {
        const int g = gbase + (j - t0);
        bool w = mbar_wait(b_p_full + 8 * (g & 1), (g >> 1) & 1, tmo, abort_flag);
        // the first P.V of a piece overwrites O^T: the previous epilogue must have read it
        if (j == t0 && pc >= 1) w = w && mbar_wait(b_o_free, (pc - 1) & 1, tmo, abort_flag);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const int st = g & (kStages - 1);
          const uint32_t st_off = (uint32_t)(st * kStageBytes) >> 4;
#pragma unroll
          for (int term = 1; term >= 0; --term) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              const int blk = blk0 + b;
#pragma unroll
              for (int kk = 0; kk < 2; ++kk) {
                const uint64_t a =
                    dv0 + st_off + (uint32_t)((2 * blk * kAtom + kk * 4 * kGroupBytes) >> 4);
                const uint32_t d = tmem + kColO + 64 * blk;
                const uint64_t pb = term ? dpl + (uint32_t)((32 * kk) >> 4)
                                         : dph0 + st_off + (uint32_t)((32 * kk) >> 4);
                // the piece's first tile starts the accumulator with its P_lo term
                mma_e4m3_ss(d, a, pb, id_pv, (j == t0 && term == 1 && kk == 0) ? 0u : 1u);
              }
            }
            if (term == 1) mma_commit(smem_u32(&misc->plo_free[g & 1]));
          }
          mma_commit(b_kv_empty + 8 * st);
          mma_commit(b_pv_done + 8 * (g & 1));
        }
        __syncwarp();
      }
      gbase += t1 - t0;
      ++pc;
    }
    if (!ok && lane == 0) set_error(p, misc, kErrTimeout);
  } else {
    // ------------------------------------------------------------ softmax
    // Group grp (warps 2..5: 0, warps 8..11: 1) takes tokens
    // [32 grp, 32 grp + 32) of every tile.  Thread (quadrant, lane) reads
    // TMEM lane 32 quadrant + lane, i.e. S_hi (even lane) or S_lo (odd lane)
    // of query row r = 16 quadrant + lane / 2, for the group's 32 tokens; the
    // two threads of a row swap halves, so each ends with S = S_hi + S_lo of
    // 16 tokens: the even one tokens 32 grp .. + 15, the odd one the rest.
    const int grp = warp >= 8 ? 1 : 0;
    const int quad = warp & 3;           // TMEM lane quadrant this warp may access
    const int gtid = threadIdx.x - (grp ? 256 : 64);   // 0..127 in the group
    const int tid = gtid + 128 * grp;    // 0..255 over both groups
    const int half = lane & 1;           // the term this thread's TMEM lane holds
    const int r = 16 * quad + (lane >> 1);
    const int tok0 = 32 * grp + 16 * half;   // this thread's first token of a tile
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
    uint8_t* plo_row = smem + kSmemPlo + (r >> 3) * kAtom + (r & 7) * 64;   // P_lo row r
    const int sw = (r & 7) >> 1;                                             // 64-byte swizzle
    int gt = 0, pc = 0, qu = 0;
    bool ok = true;
    while (ok && it.next(unit, t0, t1, whole, slot)) {
      Unit x = make_unit<kLocal>(pd, unit);
      if (grp == 1) {
        // ---------------------------------------------------- query split
        // Thread ct = 0 loads the piece's 64 bf16 query rows by TMA (8 rows
        // x 9 chunks per row group, 128-byte swizzle); thread (qr, hh) =
        // (ct / 2, ct % 2) takes row qr's largest |q| over half of its
        // 16-byte units; then, two row groups at a time, every thread reads
        // 9 units into registers and, after a barrier, writes their Q_hi /
        // Q_lo codes over the same row groups.  Decisions that end the split
        // early are taken by barrier reductions, so all 128 threads take the
        // same path; a failure leaves ok false and the first reduction of the
        // tile loop ends the piece for both groups.
        const int ct = gtid;
        const int qr = ct >> 1, hh = ct & 1;
        if (pc >= 1 && ok)
          ok = __all_sync(0xffffffffu, mbar_wait(b_q_empty, (pc - 1) & 1, tmo, abort_flag));
        if (named_bar_or(kBarConv, kConvThreads, !ok)) {
          ok = false;
          if (ct == 0) set_error(p, misc, kErrTimeout);
        }
        if (ok) {
          const bool load_q = !(p.withhold_query && pc == 0);
          if (ct == 0 && load_q) {
            mbar_arrive_expect_tx(b_q_full, kQBytes);
            armed_q = pc;
          }
          if (load_q && ct < 32) {
            __syncwarp();
            if (kRankIo) {
              // rank-major gathered query: lane k loads run k (one rank's
              // heads of one query position), run / 8 row groups per box
              const int run = q_run_rows(pd);
              if (ct < kRows / run)
                tma_load_4d(sQ + (ct * run / 8) * kQGroupBytes, &tm_q, b_q_full, 0, 0, 0,
                            q_src_row(pd, x, ct * run) >> 3);
            } else if (ct == 0) {
              tma_load_4d(sQ, &tm_q, b_q_full, 0, 0, 0, (x.b * pd.R + x.g * kRows) >> 3);
            }
          }
          ok = __all_sync(0xffffffffu, mbar_wait(b_q_full, pc & 1, tmo, abort_flag));
          if (named_bar_or(kBarConv, kConvThreads, !ok)) {
            ok = false;
            if (ct == 0) set_error(p, misc, kErrTimeout);
          }
        }
        if (ok) {
          uint8_t* q8 = smem + kSmemQ;
          {
            const int rg = qr >> 3, rr = qr & 7;
            const uint8_t* row = q8 + rg * kQGroupBytes + rr * 128;
            uint32_t mx = 0;
#pragma unroll 12
            for (int v = 0; v < 36; ++v) {
              const int w = 36 * hh + v;   // 16-byte unit of the row: chunk w / 8, unit w % 8
              const uint4 t = *reinterpret_cast<const uint4*>(row + (w >> 3) * 1024 + (w & 7) * 16);
              const uint32_t ww[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mx = max(mx, max(ww[k] & 0x7FFFu, (ww[k] >> 16) & 0x7FFFu));
            }
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            const bool live = qr < x.rows;
            if (live && (mx >> 7) == 255u) atomicOr(&p.hdr->err, kErrQRange);   // inf or NaN
            if (hh == 0) {
              // s_r = 2^(134 - e) puts max|q| in [128, 256); the softmax
              // divides it out again with 1 / s_r = 2^(e - 134)
              const uint32_t e = row_scale_exp(mx);
              misc->qinv[qr] = __uint_as_float((e - 7u) << 23);
              misc->qsc[qr] = live ? __uint_as_float((261u - e) << 23) : 0.0f;
            }
          }
          named_bar_sync(kBarConv, kConvThreads);
#pragma unroll 1
          for (int pr = 0; pr < 4; ++pr) {
            uint4 in[9];
#pragma unroll
            for (int k = 0; k < 9; ++k) {
              const int i = ct + kConvThreads * k;   // 16-byte unit of row groups 2 pr, 2 pr + 1
              in[k] = *reinterpret_cast<const uint4*>(q8 + 2 * pr * kQGroupBytes + i * 16);
            }
            named_bar_sync(kBarConv, kConvThreads);   // the pair's bf16 has been read
#pragma unroll
            for (int k = 0; k < 9; ++k) {
              const int i = ct + kConvThreads * k;
              const int rg = 2 * pr + i / 576, rem = i % 576;
              const int c = rem >> 6, rr = (rem >> 3) & 7, u = (rem & 7) ^ rr;   // u: dims 8u.. of chunk c
              const float sc = misc->qsc[rg * 8 + rr];   // s_r, 0 for a padding row
              uint32_t whi = 0, wlo = 0, whi2 = 0, wlo2 = 0;
              if (sc != 0.0f) {
                const uint32_t w[4] = {in[k].x, in[k].y, in[k].z, in[k].w};
                uint32_t sp[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  sp[e] = split_e4m3x2(__uint_as_float(w[e] << 16) * sc,
                                       __uint_as_float(w[e] & 0xFFFF0000u) * sc);
                whi = (sp[0] & 0xFFFFu) | (sp[1] << 16);
                wlo = (sp[0] >> 16) | (sp[1] & 0xFFFF0000u);
                whi2 = (sp[2] & 0xFFFFu) | (sp[3] << 16);
                wlo2 = (sp[2] >> 16) | (sp[3] & 0xFFFF0000u);
              }
              // query row 8 rg + rr is MMA row i = 2 (rr % 4) (+1 for Q_lo)
              // of group 2 rg + rr / 4; the swizzle term (i / 2) % 4 is rr % 4
              // for both terms
              uint8_t* dst = q8 + rg * kQGroupBytes + (rr >> 2) * kQAGroupBytes + c * kAtom +
                             (rr & 3) * 128 + (((u >> 1) ^ (rr & 3)) << 4) + (u & 1) * 8;
              *reinterpret_cast<uint2*>(dst) = make_uint2(whi, whi2);
              *reinterpret_cast<uint2*>(dst + 64) = make_uint2(wlo, wlo2);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_q_conv);
        }
      } else {
        ok = __all_sync(0xffffffffu, ok && mbar_wait(b_q_conv, pc & 1, tmo, abort_flag));
      }
      const bool owner = r < x.rows;
      const int i_row = (x.g * kRows + r) / pd.H;
      const int vis_limit = x.L - x.qn + i_row;
      // the row's query scale and the softmax scale, in log2 units
      const float qs = misc->qinv[r] * pd.scale_log2;
      int unit_left = 0;   // tiles of the current QK^T unit still to read
      float m_run = -CUDART_INF_F, l_run = 0.0f;   // l_run: sum of u_t over this thread's tokens
      for (int j = t0; j < t1; ++j, ++gt) {
        const int sb = qu & 1, st = gt & (kStages - 1);
        bool ok_s = ok;
        if (unit_left == 0) {
          // a new QK^T unit: a pair (gt even, next tile in the piece) or one tile
          unit_left = ((gt & 1) == 0 && j + 1 < t1) ? 2 : 1;
          ok_s = __all_sync(0xffffffffu,
                            ok_s && mbar_wait(b_s_full + 8 * sb, (qu >> 1) & 1, tmo, abort_flag));
        }
        ok_s = __all_sync(0xffffffffu,
                          ok_s && mbar_wait(b_prep + 8 * st, (gt >> 2) & 1, tmo, abort_flag));
        const bool full = tile_full<kLocal>(pd, x, j);
        float a[16], sg[16];
        uint32_t vis_mask = 0xFFFFu;
        float mx = -CUDART_INF_F;
        if (ok_s) {
          tc_fence_after();
          uint32_t sr[32];
          tmem_ld32(tmem + lane_off + kColS0 + 128 * sb + 64 * (gt & 1) + 32 * grp, sr);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (--unit_left == 0) {
            if (lane == 0) mbar_arrive(b_s_empty + 8 * sb);
            ++qu;
          }
          // keep 16 tokens, send the partner the other term of its 16
          float sv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float give = __uint_as_float(half ? sr[i] : sr[16 + i]);
            const float got = __shfl_xor_sync(0xffffffffu, give, 1);
            sv[i] = __uint_as_float(half ? sr[16 + i] : sr[i]) + got;
          }
          // a_t = S_t sigma_t / s_r * scale * log2(e); b_t = a_t + E_t
          const float4* sg4 = reinterpret_cast<const float4*>(&misc->sigma[st][tok0]);
          const float4* lg4 = reinterpret_cast<const float4*>(&misc->lge[st][tok0]);
          float b[16];
#pragma unroll
          for (int a4 = 0; a4 < 4; ++a4) {
            const float4 g = sg4[a4], l = lg4[a4];
            sg[4 * a4] = g.x;
            sg[4 * a4 + 1] = g.y;
            sg[4 * a4 + 2] = g.z;
            sg[4 * a4 + 3] = g.w;
            a[4 * a4] = sv[4 * a4] * g.x * qs;
            a[4 * a4 + 1] = sv[4 * a4 + 1] * g.y * qs;
            a[4 * a4 + 2] = sv[4 * a4 + 2] * g.z * qs;
            a[4 * a4 + 3] = sv[4 * a4 + 3] * g.w * qs;
            b[4 * a4] = a[4 * a4] + l.x;
            b[4 * a4 + 1] = a[4 * a4 + 1] + l.y;
            b[4 * a4 + 2] = a[4 * a4 + 2] + l.z;
            b[4 * a4 + 3] = a[4 * a4 + 3] + l.w;
          }
          if (!full) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int t = slot_token<kLocal>(pd, x, j, tok0 + i);
              const bool vis = slot_valid(pd, x, t) && (!pd.causal || t <= vis_limit);
              if (!vis) {
                a[i] = -CUDART_INF_F;
                b[i] = -CUDART_INF_F;
                vis_mask &= ~(1u << i);
              }
            }
          }
          float m4[4] = {b[0], b[1], b[2], b[3]};
#pragma unroll
          for (int i = 4; i < 16; i += 4) {
            m4[0] = fmaxf(m4[0], b[i]);
            m4[1] = fmaxf(m4[1], b[i + 1]);
            m4[2] = fmaxf(m4[2], b[i + 2]);
            m4[3] = fmaxf(m4[3], b[i + 3]);
          }
          mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          if (half == 0) misc->xmax[gt & 1][grp][r] = mx;
        }
        // both groups reach this reduction every tile: it publishes the
        // groups' row maxima and ends the piece for all of them if any
        // thread's wait failed
        if (named_bar_or(kBarSoftmax, kSoftmaxThreads, !ok_s)) { ok = false; break; }
        const float m_tile = fmaxf(mx, misc->xmax[gt & 1][grp ^ 1][r]);
        const float m_new = fmaxf(m_run, m_tile);
        float alpha = 1.0f;
        bool resc = false;
        if (m_new > m_run + kRescaleThreshold || (j == t0 && m_new > -CUDART_INF_F)) {
          alpha = (m_run == -CUDART_INF_F) ? 0.0f : ex2_approx(m_run - m_new);
          l_run *= alpha;
          m_run = m_new;
          resc = owner && (j != t0);
        }
        if (owner && half == 0) misc->alpha[grp][r] = alpha;
        bool waited_pv = false;
        // both groups see the same maxima, so they take the same decision
        if (named_bar_or(kBarGroup0 + grp, 128, resc)) {
          // some row's running max grew: rescale this group's half of O^T
          // (latent blocks 2 grp, 2 grp + 1) once the previous P.V landed
          const bool ok_pv = __all_sync(
              0xffffffffu, (gt == 0) || mbar_wait(b_pv_done + 8 * ((gt - 1) & 1),
                                                  ((gt - 1) >> 1) & 1, tmo, abort_flag));
          ok = ok_pv;
          waited_pv = true;
          if (!ok_pv) continue;  // caught by the next reduction (or the epilogue's)
          tc_fence_after();
#pragma unroll 1
          for (int blk = 2 * grp; blk < 2 * grp + 2; ++blk) {
#pragma unroll 1
            for (int h2 = 0; h2 < 2; ++h2) {
              uint32_t v[32];
              const uint32_t ta = tmem + lane_off + kColO + 64 * blk + 32 * h2;
              tmem_ld32(ta, v);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c)
                v[c] = __float_as_uint(__uint_as_float(v[c]) * misc->alpha[grp][32 * h2 + c]);
              tmem_st32(ta, v);
            }
          }
          tmem_wait_st();
        }
        // u_t = 2^(a_t - m); P'_t = u_t sigma_t (a masked slot's scale may be
        // garbage, even NaN: select, no branch)
        const float m_use = (m_run == -CUDART_INF_F) ? 0.0f : m_run;
        uint32_t phi[4], plo[4];
        {
          float ls4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4) {
            float pv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int i = 4 * i4 + k;
              const float u = ex2_approx(a[i] - m_use);
              ls4[k] += u;
              pv[k] = ((vis_mask >> i) & 1u) ? u * sg[i] : 0.0f;
            }
            const uint32_t s01 = split_e4m3x2(pv[0], pv[1]);
            const uint32_t s23 = split_e4m3x2(pv[2], pv[3]);
            phi[i4] = (s01 & 0xFFFFu) | (s23 << 16);
            plo[i4] = (s01 >> 16) | (s23 & 0xFFFF0000u);
          }
          l_run += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
        }
        // P_lo has one buffer: the previous tile's P_lo terms must have run
        if (!waited_pv && gt > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->plo_free[(gt - 1) & 1]),
                                                 ((gt - 1) >> 1) & 1, tmo, abort_flag));
          if (!ok) continue;
        }
        uint8_t* stage = smem + kSmemKV + st * kStageBytes;
        if (owner) {
          // this thread's 16 tokens are 16-byte unit tok0 / 16 of the row
          const int u = tok0 >> 4;
          uint8_t* hrow = stage + (r >> 3) * kGroupBytes + kRopeAtom + (r & 7) * 64;
          *reinterpret_cast<uint4*>(hrow + ((u ^ sw) << 4)) =
              make_uint4(phi[0], phi[1], phi[2], phi[3]);
          *reinterpret_cast<uint4*>(plo_row + ((u ^ sw) << 4)) =
              make_uint4(plo[0], plo[1], plo[2], plo[3]);
        }
        if (!full) {
          // zero the value codes of slots that hold no valid token of this
          // shard, so that garbage (even NaN codes) cannot reach O
          for (int e = tid; e < kTile * 32; e += kSoftmaxThreads) {
            const int a2 = e >> 5, c = (e >> 2) & 7, u = e & 3;
            const int t = slot_token<kLocal>(pd, x, j, a2);
            if (!slot_valid(pd, x, t))
              *reinterpret_cast<uint4*>(stage + (a2 >> 3) * kGroupBytes + c * kAtom +
                                        (a2 & 7) * 64 + u * 16) = make_uint4(0, 0, 0, 0);
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
      {
        const float l_grp = l_run + __shfl_xor_sync(0xffffffffu, l_run, 1);
        if (half == 0) misc->xl[grp][r] = l_grp;
      }
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
      if (grp == 0 && owner && half == 0) {
        const float l_tot = misc->xl[0][r] + misc->xl[1][r];
        float lse = (l_tot > 0.0f) ? (m_run + __log2f(l_tot)) * 0.69314718055994530942f
                                   : -CUDART_INF_F;
        misc->inv_l[r] = (l_tot > 0.0f) ? 1.0f / l_tot : 0.0f;
        lbase[dst_row(r)] = lse;
      }
      if (whole) {
        for (int e = tid; e < (x.rows_out - x.rows) * (kDv / 4); e += kSoftmaxThreads)
          reinterpret_cast<float4*>(obase + dst_row(x.rows + e / (kDv / 4)) * kDv)[e % (kDv / 4)] =
              make_float4(0.f, 0.f, 0.f, 0.f);
        for (int rr = x.rows + tid; rr < x.rows_out; rr += kSoftmaxThreads)
          lbase[dst_row(rr)] = -CUDART_INF_F;
      }
      named_bar_sync(kBarSoftmax, kSoftmaxThreads);
      {
        // this group's latent blocks 2 grp, 2 grp + 1: block k / 2, rows
        // 32 (k % 2) .. of this thread's latent dim, two TMEM loads in flight
        const uint32_t o_base = tmem + lane_off + kColO + 128 * grp;
        auto store32 = [&](int k, const uint32_t (&v)[32]) {
          const int dim = 128 * (2 * grp + (k >> 1)) + 32 * quad + lane;
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
        for (int k = 0; k < 4; k += 2) {
          tmem_ld32(o_base + 32 * (k + 1), vb);
          tmem_wait_ld();
          store32(k, va);
          if (k + 2 < 4) tmem_ld32(o_base + 32 * (k + 2), va);
          store32(k + 1, vb);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_o_free);
      named_bar_sync(kBarSoftmax, kSoftmaxThreads);  // inv_l and xl reused by the next piece
      ++pc;
    }
    if (!ok && tid == 0) set_error(p, misc, kErrTimeout);
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // After a failure, let this CTA's own MMAs and copies complete before
    // TMEM is freed and the CTA exits (one commit drains every earlier MMA
    // of the issuing thread).
    int never = 0;
    if (lane == 0 && (warp == 1 || warp == 6 || warp == 7)) {
      mma_commit(smem_u32(&misc->drain));
      mbar_wait(smem_u32(&misc->drain), 0, kDrainNs, &never);
    }
    // the query copy is issued by thread 0 of softmax group 1 (warp 8, lane 0)
    if (warp == 8 && lane == 0 && armed_q >= 0) mbar_wait(b_q_full, armed_q & 1, kDrainNs, &never);
    if (warp == 0 && lane == 0) {
      for (int st = 0; st < kStages; ++st)
        if (armed_kv[st] >= 0)
          mbar_wait(b_kv_full + 8 * st, (armed_kv[st] >> 2) & 1, kDrainNs, &never);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int kLocal, bool kRankIo = false>
static cudaError_t launch_partial_fp8_impl(const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                                           const PartialParams& p, int grid, cudaStream_t stream) {
  const cudaError_t e = host::ensure_dynamic_smem(
      reinterpret_cast<const void*>(&mla_partial_fp8_kernel<kLocal, kRankIo>), kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr = pdl_attribute();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_partial_fp8_kernel<kLocal, kRankIo>, tm_q, tm_kv, p);
}

cudaError_t launch_partial_fp8(const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                               const PartialParams& p, int grid, cudaStream_t stream) {
  // the DCP rank-major I/O (local caches only) is an instantiation of its own
  if (p.pd.rank_heads != 0) return launch_partial_fp8_impl<1, true>(tm_q, tm_kv, p, grid, stream);
  return p.pd.local ? launch_partial_fp8_impl<1>(tm_q, tm_kv, p, grid, stream)
         : p.pd.pad   ? launch_partial_fp8_impl<2>(tm_q, tm_kv, p, grid, stream)
                      : launch_partial_fp8_impl<0>(tm_q, tm_kv, p, grid, stream);
}

}  // namespace mla
