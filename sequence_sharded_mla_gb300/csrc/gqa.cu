// Sequence-sharded grouped-query attention (GQA) decode: the second backend
// of "Decode Context Parallelism" (section 5.4).  The cache stores Hkv KV
// heads of width 128 in separate K and V caches; every KV head serves a
// group of G = H / Hkv consecutive query heads ("tensor broadcast"); the
// sequence is sharded as for the latent cache and the shards' partials are
// merged by their LSEs.
//
// Work unit: (request b, shard s, KV head kh, group g of 64 query rows).  A
// group holds 64 / G query positions x G heads, row r = i_local * G + j for
// query head kh * G + j.  Persistent CTAs walk a stream-K list of 64-token
// tiles as the latent-cache kernel does, with four K/V stages:
//   warp 0      producer: TMA loads of the query group and of K and V tiles
//               (one box per page and shard; group-major layout, 2 chunks)
//   warp 1      QK^T issue: S = Q K^T (M=64 rows, N=64 tokens, K=128) into
//               one TMEM accumulator per stage
//   warp 6      P.V issue: O^T += V^T P^T (M=128 dims, N=rows rounded to 16,
//               K=64 tokens), as soon as a tile's probabilities are ready.
//               With one warp issuing both kinds, a ready P.V waited behind
//               the next QK^T's issue and the stages were released late
//               (4.91 against 6.50 TB/s on the agentic GQA batch).
//   warps 2..5  softmax (two threads per row), P in the stage's P buffer,
//               lazy O^T rescale, epilogue o = O/l, lse = m + ln l.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "host_util.h"
#include "mla_dcp.h"
#include "ptx.cuh"

namespace mla {
namespace gqa {

constexpr int kD = 128;                          // head width
constexpr int kGChunks = kD / 64;                // 2 swizzle chunks per row
constexpr int kGroupB = kGChunks * 1024;         // 2048: one 8-slot group of a tile
constexpr int kKVTile = 8 * kGroupB;             // 16384: 64 tokens of one KV head
constexpr int kPBytes = kRows * 128;             // 8192: P, 64 rows x 64 tokens bf16
constexpr int kStages = 4;
constexpr int kStageBytes = 2 * kKVTile + kPBytes;   // K, V, P
constexpr int kQBytes = kGChunks * kRows * 128;      // 16384
constexpr int kSmemQ = 0;
constexpr int kSmemStage = kQBytes;
constexpr int kSmemMisc = kSmemStage + kStages * kStageBytes;
constexpr int kSmemBytes = kSmemMisc + 2048 + 1024;  // + misc + alignment slack
constexpr int kThreads = 224;
constexpr int kSoftmaxWarps = 4, kSoftmaxThreads = 128;
constexpr uint32_t kBarSoftmax = 1;
constexpr float kRescaleThreshold = 8.0f;        // log2 units
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                    // stage st: S at columns 64 * st
constexpr uint32_t kColO = 256;                  // O^T: 64 columns
constexpr int kMinTilesPerCta = 4;
constexpr int kUnitCost = 2;
constexpr unsigned long long kTimeoutNs = 2000000000ull;
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Desc {
  int B, q_len, H, Hkv, G;   // G = H / Hkv, a power of two <= 64
  int lg;                    // log2(G)
  int ni;                    // query positions per 64-row group (64 / G)
  int Gq;                    // row groups per (request, KV head)
  int num_shards, shard_first, n_out, layout, causal, num_pages, max_pages;
  float scale_log2;
  const int32_t* block_table;
  const int32_t* seq_lens;
};

struct Params {
  Desc d;
  float* out_partial;   // [n_out, B, q_len, H, 128]
  float* lse_partial;   // [n_out, B, q_len, H]
  WsHeader* hdr;
  int* prefix;
  float* ws_o;          // [grid * 2, 64, 128]
  float* ws_lse;        // [grid * 2, 64]
  unsigned long long timeout_ns;
};

struct Unit {
  int b, so, s, kh, g, i0, L, rows, tiles, tstart, tend, p0;
};

__device__ __forceinline__ Unit make_unit(const Desc& d, int u) {
  Unit x;
  x.g = u % d.Gq;
  int t = u / d.Gq;
  x.kh = t % d.Hkv;
  t /= d.Hkv;
  x.so = t % d.n_out;
  x.b = t / d.n_out;
  x.s = d.shard_first + x.so;
  x.L = d.seq_lens[x.b];
  x.i0 = x.g * d.ni;
  x.rows = min(kRows, (d.q_len - x.i0) * d.G);
  x.tstart = x.tend = x.p0 = 0;
  const int L = x.L > 0 ? x.L : 0;
  if (d.layout == kInterleaved) {
    const int n_local = L > x.s ? (L - 1 - x.s) / d.num_shards + 1 : 0;
    x.tiles = ceil_div(n_local, kTile);
  } else {
    const int c = ceil_div(L, d.num_shards);
    x.tstart = x.s * c;
    x.tend = min(x.tstart + c, L);
    if (x.tstart < x.tend) {
      x.p0 = x.tstart / kPage;
      x.tiles = (x.tend - 1) / kPage - x.p0 + 1;
    } else {
      x.tiles = 0;
    }
  }
  return x;
}

// Global position of slot a of tile j (the latent kernel's tile geometry).
__device__ __forceinline__ int slot_token(const Desc& d, const Unit& x, int j, int a) {
  if (d.layout == kInterleaved) return (j * kTile + a) * d.num_shards + x.s;
  return (x.p0 + j) * kPage + a;
}

__device__ __forceinline__ bool slot_valid(const Desc& d, const Unit& x, int t) {
  if (d.layout == kInterleaved) return t < x.L;
  return t >= x.tstart && t < x.tend;
}

__device__ __forceinline__ bool tile_full(const Desc& d, const Unit& x, int j) {
  const int first = slot_token(d, x, j, 0), last = slot_token(d, x, j, kTile - 1);
  bool ok = slot_valid(d, x, first) && slot_valid(d, x, last);
  if (d.causal) ok = ok && last <= x.L - d.q_len + x.i0;
  return ok;
}

// Output row of row r (< x.rows) of unit x: query position x.i0 + r / G,
// head kh * G + r % G, in [n_out, B, q_len, H].  G is a power of two.
__device__ __forceinline__ size_t out_row(const Desc& d, const Unit& x, int r) {
  const int i = x.i0 + (r >> d.lg), h = (x.kh << d.lg) + (r & (d.G - 1));
  return (((size_t)x.so * d.B + x.b) * d.q_len + i) * d.H + h;
}

struct Misc {
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[kStages], s_empty[kStages];
  uint64_t p_full[kStages], pv_done[kStages];
  uint64_t q_full, q_empty, o_free;
  uint64_t drain;  // teardown after a failure: MMAs in flight
  uint32_t tmem_base;
  int abort;
  float alpha[2][kRows];
  alignas(16) float inv_l[kRows];
};
static_assert(sizeof(Misc) <= 2048, "misc block");

__device__ __forceinline__ void set_error(const Params& p, Misc* misc, unsigned bits) {
  atomicOr(&p.hdr->err, bits);
  if (bits & kErrTimeout) *(volatile int*)&misc->abort = 1;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(1024) gqa_plan_kernel(Desc d, WsHeader* hdr, int* prefix,
                                                        int grid) {
  griddep_launch_dependents();
  plan_units(d.B * d.n_out * d.Hkv * d.Gq, [&](int u) { return make_unit(d, u).tiles; }, hdr,
             prefix, grid, kMinTilesPerCta, kUnitCost, 0u);
}

__global__ void __launch_bounds__(kThreads, 1)
    gqa_partial_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Misc* misc = reinterpret_cast<Misc*>(smem + kSmemMisc);
  const Desc& d = p.d;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();
  griddep_launch_dependents();

  const int W = p.hdr->total_cost, per = p.hdr->per_cta;
  const int lo = blockIdx.x * per;
  if (lo >= W) return;
  const int hi = min(lo + per, W);
  const int U = p.hdr->num_units;

  const uint32_t sQ = smem_u32(smem + kSmemQ);
  const uint32_t sSt = smem_u32(smem + kSmemStage);
  auto bar = [&](const uint64_t* b) { return smem_u32(b); };
  volatile int* abort_flag = &misc->abort;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(bar(&misc->kv_full[st]), 1);
      mbar_init(bar(&misc->kv_empty[st]), 1);
      mbar_init(bar(&misc->s_full[st]), 1);
      mbar_init(bar(&misc->s_empty[st]), kSoftmaxWarps);
      mbar_init(bar(&misc->p_full[st]), kSoftmaxWarps);
      mbar_init(bar(&misc->pv_done[st]), 1);
    }
    mbar_init(bar(&misc->q_full), 1);
    mbar_init(bar(&misc->q_empty), 1);
    mbar_init(bar(&misc->o_free), kSoftmaxWarps);
    mbar_init(bar(&misc->drain), 2);  // the two MMA-issuing threads
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
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  const uint64_t tmo = p.timeout_ns;

  PieceIter it;
  it.init(p.prefix, U, lo, hi, p.hdr->unit_cost);
  int armed_kv[kStages], armed_q = -1;
  for (int st = 0; st < kStages; ++st) armed_kv[st] = -1;
  int unit, t0, t1, slot;
  bool whole;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const int nv = d.layout == kInterleaved ? d.num_shards : 1;   // page boxes per tile
    const int box_bytes = kKVTile / nv;
    int gt = 0, pc = 0;
    bool ok = true;
    while (ok && it.next(unit, t0, t1, whole, slot)) {
      const Unit x = make_unit(d, unit);
      const int npages_b = ceil_div(x.L, kPage);
      const int32_t* bt = d.block_table + (size_t)x.b * d.max_pages;
      const int res = nv > 1 ? x.s : 0;
      for (int j = t0; j < t1 && ok; ++j, ++gt) {
        const int st = gt % kStages, round = gt / kStages;
        const int first_slot = nv > 1 ? j * nv : x.p0 + j;
        const int idx = first_slot + lane;
        int page = -1;
        if (lane < nv && idx < npages_b) {
          page = idx < d.max_pages ? __ldg(bt + idx) : -1;
          if (page < 0 || page >= d.num_pages) {
            set_error(p, misc, kErrBadPage);
            page = d.num_pages;
          }
        }
        if (idx >= npages_b) page = d.num_pages;   // past the context: TMA fills zeros
        if (round >= 1) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(&misc->kv_empty[st]), (round - 1) & 1, tmo,
                                                 abort_flag));
          if (!ok) break;
        }
        const uint32_t full = bar(&misc->kv_full[st]);
        if (lane == 0) {
          mbar_arrive_expect_tx(full, 2 * kKVTile);
          armed_kv[st] = gt;
        }
        __syncwarp();
        if (lane < nv) {
          const uint32_t dst = sSt + st * kStageBytes + lane * box_bytes;
          const int crow = (page * kPage + res) * d.Hkv + x.kh;   // cache row of this head
          tma_load_5d(dst, &tm_k, full, 0, 0, 0, 0, crow);
          tma_load_5d(dst + kKVTile, &tm_v, full, 0, 0, 0, 0, crow);
        }
        __syncwarp();
        if (j == t0) {
          if (pc >= 1) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(bar(&misc->q_empty), (pc - 1) & 1, tmo, abort_flag));
            if (!ok) break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(&misc->q_full), kQBytes);
            armed_q = pc;
            tma_load_5d(sQ, &tm_q, bar(&misc->q_full), 0, 0, x.b * d.q_len + x.i0, 0, x.kh);
          }
          __syncwarp();
        }
      }
      ++pc;
    }
    if (!ok && lane == 0) set_error(p, misc, kErrTimeout);
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK^T issue
    const uint32_t id_qk = idesc_bf16_f32(64, 64, false, false);
    const uint64_t dq0 = sw128_desc(sQ, 16, 1024);
    const uint64_t dk0 = sw128_desc(sSt, 16, kGroupB);                 // K: groups 2048 apart
    int gbase = 0, pc = 0;
    bool ok = true;
    while (ok && it.next(unit, t0, t1, whole, slot)) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(&misc->q_full), pc & 1, tmo, abort_flag));
      for (int j = t0; ok && j < t1; ++j) {
        const int g = gbase + (j - t0), st = g % kStages, round = g / kStages;
        bool w = mbar_wait(bar(&misc->kv_full[st]), round & 1, tmo, abort_flag);
        if (round >= 1) w = w && mbar_wait(bar(&misc->s_empty[st]), (round - 1) & 1, tmo, abort_flag);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t off = (uint32_t)(st * kStageBytes) >> 4;
#pragma unroll
          for (int c = 0; c < kGChunks; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16_ss(tmem + kColS + 64 * st,
                          dq0 + (uint32_t)((c * kRows * 128 + 32 * k) >> 4),
                          dk0 + off + (uint32_t)((c * 1024 + 32 * k) >> 4), id_qk,
                          (c != 0 || k != 0) ? 1u : 0u);
          mma_commit(bar(&misc->s_full[st]));
          if (j == t1 - 1) mma_commit(bar(&misc->q_empty));
        }
        __syncwarp();
      }
      gbase += t1 - t0;
      ++pc;
    }
    if (!ok && lane == 0) set_error(p, misc, kErrTimeout);
  } else if (warp == 6) {
    // ------------------------------------------------------------ P.V issue
    const uint64_t dv0 = sw128_desc(sSt + kKVTile, 1024, kGroupB);     // V^T: MN-major
    const uint64_t dp0 = sw128_desc(sSt + 2 * kKVTile, 16, 1024);      // P: 8-row groups
    int gbase = 0, pc = 0;
    bool ok = true;
    while (ok && it.next(unit, t0, t1, whole, slot)) {
      const Unit x = make_unit(d, unit);
      const int npv = (x.rows + 15) & ~15;
      const uint32_t id_pv = idesc_bf16_f32(128, npv, true, false);
      for (int j = t0; ok && j < t1; ++j) {
        const int g = gbase + (j - t0), st = g % kStages, round = g / kStages;
        bool w = mbar_wait(bar(&misc->p_full[st]), round & 1, tmo, abort_flag);
        if (j == t0 && pc >= 1) w = w && mbar_wait(bar(&misc->o_free), (pc - 1) & 1, tmo, abort_flag);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t off = (uint32_t)(st * kStageBytes) >> 4;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss(tmem + kColO, dv0 + off + (uint32_t)((kk * 2 * kGroupB) >> 4),
                        dp0 + off + (uint32_t)((32 * kk) >> 4), id_pv,
                        (j == t0 && kk == 0) ? 0u : 1u);
          mma_commit(bar(&misc->kv_empty[st]));
          mma_commit(bar(&misc->pv_done[st]));
        }
        __syncwarp();
      }
      gbase += t1 - t0;
      ++pc;
    }
    if (!ok && lane == 0) set_error(p, misc, kErrTimeout);
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int tid = threadIdx.x - 64;    // 0..127
    const int half = lane >> 4;
    const int r = 16 * quad + (lane & 15);
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
    int gt = 0, pc = 0;
    bool ok = true;
    while (ok && it.next(unit, t0, t1, whole, slot)) {
      const Unit x = make_unit(d, unit);
      const bool owner = r < x.rows;
      const int vis_limit = x.L - d.q_len + x.i0 + (r >> d.lg);   // causal: t <= vis_limit
      float m_run = -CUDART_INF_F, l_run = 0.0f;
      for (int j = t0; j < t1; ++j, ++gt) {
        const int st = gt % kStages, round = gt / kStages;
        const bool ok_s = __all_sync(
            0xffffffffu, ok && mbar_wait(bar(&misc->s_full[st]), round & 1, tmo, abort_flag));
        bool resc = false;
        uint32_t pk[16];
        const bool full = tile_full(d, x, j);
        if (ok_s) {
          tc_fence_after();
          uint32_t sr[32];
          tmem_ld16x2_32(tmem + lane_off + kColS + 64 * st, sr);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(&misc->s_empty[st]));
          float s[32];
#pragma unroll
          for (int a = 0; a < 32; ++a) s[a] = __uint_as_float(sr[a]);
          if (!full) {
#pragma unroll
            for (int a = 0; a < 32; ++a) {
              const int t = slot_token(d, x, j, 32 * half + a);
              if (!(slot_valid(d, x, t) && (!d.causal || t <= vis_limit))) s[a] = -CUDART_INF_F;
            }
          }
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
          const float m_new = fmaxf(m_run, mx * d.scale_log2);
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
            const float p0 = ex2_approx(fmaf(s[2 * a], d.scale_log2, -m_use));
            const float p1 = ex2_approx(fmaf(s[2 * a + 1], d.scale_log2, -m_use));
            pk[a] = pack_bf16x2(p0, p1);
            ls4[a & 3] += p0 + p1;
          }
          l_run += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
        }
        if (named_bar_or(kBarSoftmax, kSoftmaxThreads, resc || !ok_s)) {
          if (named_bar_or(kBarSoftmax, kSoftmaxThreads, !ok_s)) { ok = false; break; }
          // a running max grew: rescale O^T once the previous P.V has landed
          const bool ok_pv = __all_sync(
              0xffffffffu,
              (gt == 0) || mbar_wait(bar(&misc->pv_done[(gt - 1) % kStages]),
                                     ((gt - 1) / kStages) & 1, tmo, abort_flag));
          ok = ok_pv;
          if (!ok_pv) continue;
          tc_fence_after();
#pragma unroll 1
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t v[32];
            const uint32_t ta = tmem + lane_off + kColO + 32 * h2;
            tmem_ld32(ta, v);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c)
              v[c] = __float_as_uint(__uint_as_float(v[c]) * misc->alpha[gt & 1][32 * h2 + c]);
            tmem_st32(ta, v);
          }
          tmem_wait_st();
        }
        uint8_t* stage = smem + kSmemStage + st * kStageBytes;
        if (owner) {
          uint8_t* prow = stage + 2 * kKVTile + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int ch = 4 * half + c;
            *reinterpret_cast<uint4*>(prow + ((ch ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          }
        }
        if (!full) {
          // zero V rows of slots that hold no valid token (NaN cannot reach O)
          for (int e = tid; e < kTile * kGChunks * 8; e += kSoftmaxThreads) {
            const int a = e / (kGChunks * 8), c = (e / 8) % kGChunks, ch = e % 8;
            const int t = slot_token(d, x, j, a);
            if (!slot_valid(d, x, t))
              *reinterpret_cast<uint4*>(stage + kKVTile + (a >> 3) * kGroupB + c * 1024 +
                                        (a & 7) * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(&misc->p_full[st]));
      }
      // ---------------------------------------------------------- epilogue
      const bool ok_e = __all_sync(
          0xffffffffu, ok && mbar_wait(bar(&misc->pv_done[(gt - 1) % kStages]),
                                       ((gt - 1) / kStages) & 1, tmo, abort_flag));
      if (named_bar_or(kBarSoftmax, kSoftmaxThreads, !ok_e)) { ok = false; break; }
      tc_fence_after();
      const size_t sl = 2 * (size_t)blockIdx.x + slot;
      const float l_tot = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
      if (owner && half == 0) {
        const float lse = (l_tot > 0.0f) ? (m_run + __log2f(l_tot)) * 0.69314718055994530942f
                                         : -CUDART_INF_F;
        misc->inv_l[r] = (l_tot > 0.0f) ? 1.0f / l_tot : 0.0f;
        if (whole) p.lse_partial[out_row(d, x, r)] = lse;
        else p.ws_lse[sl * kRows + r] = lse;
      }
      named_bar_sync(kBarSoftmax, kSoftmaxThreads);
      // thread (quad, lane) holds latent dim 32*quad + lane of every row
      const int dim = 32 * quad + lane;
#pragma unroll 1
      for (int h2 = 0; h2 < 2 && 32 * h2 < x.rows; ++h2) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + kColO + 32 * h2, v);
        tmem_wait_ld();
        float il[32];
        const float4* il4 = reinterpret_cast<const float4*>(misc->inv_l + 32 * h2);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 t = il4[c4];
          il[4 * c4] = t.x;
          il[4 * c4 + 1] = t.y;
          il[4 * c4 + 2] = t.z;
          il[4 * c4 + 3] = t.w;
        }
        // rows 32*h2 + c go to out_partial rows base + (c >> lg) * H + (c & (G-1))
        // (whole unit) or to consecutive workspace rows (piece of a split unit)
        float* base = whole ? p.out_partial + out_row(d, x, 32 * h2) * kD
                            : p.ws_o + (sl * kRows + 32 * h2) * kD;
        const size_t pos_stride = whole ? (size_t)d.H * kD : (size_t)d.G * kD;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (32 * h2 + c < x.rows)
            base[(size_t)(c >> d.lg) * pos_stride + (size_t)(c & (d.G - 1)) * kD + dim] =
                __uint_as_float(v[c]) * il[c];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(&misc->o_free));
      named_bar_sync(kBarSoftmax, kSoftmaxThreads);   // inv_l reused by the next piece
      ++pc;
    }
    if (!ok && tid == 0) set_error(p, misc, kErrTimeout);
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // after a failure, let this CTA's own MMAs and copies complete first
    int never = 0;
    if (lane == 0 && (warp == 1 || warp == 6)) {
      mma_commit(bar(&misc->drain));
      mbar_wait(bar(&misc->drain), 0, kDrainNs, &never);
    }
    if (warp == 0 && lane == 0) {
      for (int st = 0; st < kStages; ++st)
        if (armed_kv[st] >= 0)
          mbar_wait(bar(&misc->kv_full[st]), (armed_kv[st] / kStages) & 1, kDrainNs, &never);
      if (armed_q >= 0) mbar_wait(bar(&misc->q_full), armed_q & 1, kDrainNs, &never);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Units not written by the partial kernel: no token in the shard (o = 0,
// lse = -inf) and units split across CTAs (their pieces merged by LSE).
// Block u, warp w handles rows w, w + 4, ...; lane: dims 4*lane..4*lane+3.
__global__ void __launch_bounds__(128) gqa_merge_kernel(Desc d, const WsHeader* hdr,
                                                        const int* prefix, const float* ws_o,
                                                        const float* ws_lse, float* out_partial,
                                                        float* lse_partial) {
  griddep_wait();
  griddep_launch_dependents();
  const int u = blockIdx.x;
  const Unit x = make_unit(d, u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ps = prefix[u], ue = prefix[u + 1];
  const int us = unit_tile_start(prefix, u, hdr->unit_cost);
  const int per = hdr->per_cta;
  const bool empty = us == ue;
  const int c0 = empty ? 0 : us / per, c1 = empty ? 0 : (ue - 1) / per;
  if (!empty && c0 == c1) return;   // written by the partial kernel
  auto slot_of = [&](int c) -> size_t {
    return (c == c0 && c0 * per < ps) ? 2 * (size_t)c + 1 : 2 * (size_t)c;
  };
  const int np = c1 - c0 + 1;
  for (int r = warp; r < x.rows; r += 4) {
    float4* dst = reinterpret_cast<float4*>(out_partial + out_row(d, x, r) * kD);
    if (empty) {
      dst[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane == 0) lse_partial[out_row(d, x, r)] = -CUDART_INF_F;
      continue;
    }
    float M = -CUDART_INF_F;
    for (int k = lane; k < np; k += 32) M = fmaxf(M, ws_lse[slot_of(c0 + k) * kRows + r]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M > -CUDART_INF_F) {
      for (int k = 0; k < np; ++k) {
        const size_t s = slot_of(c0 + k);
        const float w = __expf(ws_lse[s * kRows + r] - M);
        wsum += w;
        const float4 o = reinterpret_cast<const float4*>(ws_o + (s * kRows + r) * kD)[lane];
        acc.x += w * o.x;
        acc.y += w * o.y;
        acc.z += w * o.z;
        acc.w += w * o.w;
      }
    }
    const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
    dst[lane] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (lane == 0) lse_partial[out_row(d, x, r)] = wsum > 0.f ? M + __logf(wsum) : -CUDART_INF_F;
  }
}

// LSE combine of N shard partials of width 128: one warp per row.
__global__ void __launch_bounds__(256) gqa_combine_kernel(const float* __restrict__ partials,
                                                          const float* __restrict__ lses,
                                                          int num_shards, int rows,
                                                          uint16_t* __restrict__ out,
                                                          float* __restrict__ lse_out) {
  griddep_wait();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float M = -CUDART_INF_F;
  for (int s = 0; s < num_shards; ++s) M = fmaxf(M, __ldg(lses + (size_t)s * rows + row));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (M > -CUDART_INF_F) {
    for (int s = 0; s < num_shards; ++s) {
      const float w = __expf(__ldg(lses + (size_t)s * rows + row) - M);
      wsum += w;
      const float4 o = __ldg(reinterpret_cast<const float4*>(partials + ((size_t)s * rows + row) * kD) + lane);
      acc.x += w * o.x;
      acc.y += w * o.y;
      acc.z += w * o.z;
      acc.w += w * o.w;
    }
  }
  const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
  uint2 packed = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  reinterpret_cast<uint2*>(out + (size_t)row * kD)[lane] = packed;
  if (lse_out != nullptr && lane == 0)
    lse_out[row] = M > -CUDART_INF_F ? M + __logf(wsum) : -CUDART_INF_F;
}

// ------------------------------------------------------------------ host side
bool shape_ok(const gqa_shape* s) {
  if (s == nullptr || s->batch < 1 || s->q_len < 1 || s->num_heads < 1 || s->num_kv_heads < 1)
    return false;
  if (s->causal != 0 && s->causal != 1) return false;
  if (!std::isfinite(s->softmax_scale) || s->softmax_scale <= 0.f) return false;
  return (long long)s->batch * s->q_len * s->num_heads < (1LL << 30);
}

bool shape_supported(const gqa_shape* s) {
  if (s->head_dim != kD || s->num_heads % s->num_kv_heads != 0) return false;
  const int G = s->num_heads / s->num_kv_heads;
  return G <= kRows && (G & (G - 1)) == 0;
}

int units_for(const gqa_shape* s, int num_shards, int shard_id) {
  const int n_out = shard_id == MLA_ALL_SHARDS ? num_shards : 1;
  const int G = s->num_heads / s->num_kv_heads;
  const int Gq = ceil_div(s->q_len, kRows / G);
  return s->batch * n_out * s->num_kv_heads * Gq;
}

struct WsLayout {
  size_t hdr, prefix, ws_o, ws_lse, total;
};

WsLayout ws_layout(int num_units, int grid) {
  auto up = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
  WsLayout w;
  w.hdr = 0;
  w.prefix = up(sizeof(WsHeader));
  w.ws_o = w.prefix + up(sizeof(int) * (size_t)(num_units + 1));
  w.ws_lse = w.ws_o + up(sizeof(float) * (size_t)grid * 2 * kRows * kD);
  w.total = w.ws_lse + up(sizeof(float) * (size_t)grid * 2 * kRows);
  return w;
}

}  // namespace gqa
}  // namespace mla

using namespace mla;

extern "C" {

size_t gqa_workspace_size(const gqa_shape* shape, int num_shards, int shard_id) {
  if (!gqa::shape_ok(shape) || !gqa::shape_supported(shape)) return 0;
  if (num_shards < 1 || num_shards > kMaxShards) return 0;
  if (shard_id != MLA_ALL_SHARDS && (shard_id < 0 || shard_id >= num_shards)) return 0;
  const int grid = std::min(host::device_sm_count(), 512);
  if (grid <= 0) return 0;
  return gqa::ws_layout(gqa::units_for(shape, num_shards, shard_id), grid).total;
}

mla_status gqa_decode_partial(const void* q, const gqa_kv_pages* kv, const int32_t* block_table,
                              int max_pages_per_req, const int32_t* seq_lens,
                              const gqa_shape* shape, int shard_id, int num_shards,
                              mla_layout layout, float* out_partial, float* lse_partial,
                              void* workspace, size_t workspace_bytes, void* stream) {
  using host::aligned16;
  using host::aligned4;
  if (!q || !kv || !block_table || !seq_lens || !out_partial || !lse_partial) return MLA_ERR_INVALID;
  if (!gqa::shape_ok(shape)) return MLA_ERR_INVALID;
  if (num_shards < 1 || num_shards > kMaxShards) return MLA_ERR_INVALID;
  if (shard_id != MLA_ALL_SHARDS && (shard_id < 0 || shard_id >= num_shards)) return MLA_ERR_INVALID;
  if (layout != MLA_LAYOUT_INTERLEAVED && layout != MLA_LAYOUT_CONTIGUOUS) return MLA_ERR_INVALID;
  if (kv->k == nullptr || kv->v == nullptr || kv->num_pages < 1 || max_pages_per_req < 1)
    return MLA_ERR_INVALID;
  if (kv->page_size != kPage || !gqa::shape_supported(shape)) return MLA_ERR_UNSUPPORTED;
  if (layout == MLA_LAYOUT_INTERLEAVED && kPage % num_shards != 0) return MLA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(kv->k) || !aligned16(kv->v) || !aligned16(out_partial) ||
      !aligned16(lse_partial) || !aligned4(block_table) || !aligned4(seq_lens))
    return MLA_ERR_INVALID;
  if (workspace == nullptr || !aligned16(workspace)) return MLA_ERR_WORKSPACE;
  const int grid = std::min(host::device_sm_count(), 512);
  if (grid <= 0) return MLA_ERR_CUDA;
  const int U = gqa::units_for(shape, num_shards, shard_id);
  const gqa::WsLayout wl = gqa::ws_layout(U, grid);
  if (workspace_bytes < wl.total) return MLA_ERR_WORKSPACE;
  host::EncodeTiledFn encode = host::encode_fn();
  if (encode == nullptr) return MLA_ERR_CUDA;

  gqa::Desc d;
  d.B = shape->batch;
  d.q_len = shape->q_len;
  d.H = shape->num_heads;
  d.Hkv = shape->num_kv_heads;
  d.G = d.H / d.Hkv;
  d.lg = 0;
  while ((1 << d.lg) < d.G) ++d.lg;
  d.ni = kRows / d.G;
  d.Gq = ceil_div(d.q_len, d.ni);
  d.num_shards = num_shards;
  d.shard_first = shard_id == MLA_ALL_SHARDS ? 0 : shard_id;
  d.n_out = shard_id == MLA_ALL_SHARDS ? num_shards : 1;
  d.layout = layout == MLA_LAYOUT_INTERLEAVED ? kInterleaved : kContiguous;
  d.causal = shape->causal;
  d.num_pages = kv->num_pages;
  d.max_pages = max_pages_per_req;
  d.scale_log2 = shape->softmax_scale * 1.4426950408889634f;
  d.block_table = block_table;
  d.seq_lens = seq_lens;

  // query [B*q_len, Hkv, G, 128] read as (64 dims, head in group, position,
  // chunk, KV head): one box lands the 64 rows (positions x group heads) of a
  // row group in the [chunk][row][64] shared-memory layout
  const cuuint64_t hb = (cuuint64_t)gqa::kD * 2;   // bytes per head row
  CUtensorMap tm_q, tm_k, tm_v;
  {
    cuuint64_t dims[5] = {64, (cuuint64_t)d.G, (cuuint64_t)d.B * d.q_len, 2, (cuuint64_t)d.Hkv};
    cuuint64_t strides[4] = {hb, hb * d.H, 128, hb * d.G};
    cuuint32_t box[5] = {64, (cuuint32_t)d.G, (cuuint32_t)d.ni, 2, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(q), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MLA_ERR_CUDA;
  }
  // K and V [pages * 64, Hkv, 128] read as (64 dims, row in group, chunk,
  // group, cache row x KV head) from row (page * 64 + residue) * Hkv + kh: a
  // box lands the page's 64/nv rows of one shard, both chunks, group-major
  const int nv = d.layout == kInterleaved ? num_shards : 1;
  for (int which = 0; which < 2; ++which) {
    cuuint64_t dims[5] = {64, 8, 2, (cuuint64_t)(kPage / 8 / nv),
                          (cuuint64_t)kv->num_pages * kPage * d.Hkv};
    cuuint64_t strides[4] = {hb * d.Hkv * nv, 128, hb * d.Hkv * 8 * nv, hb};
    cuuint32_t box[5] = {64, 8, 2, (cuuint32_t)(kPage / 8 / nv), 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (encode(which ? &tm_v : &tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
               const_cast<void*>(which ? kv->v : kv->k), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MLA_ERR_CUDA;
  }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  gqa::Params p;
  p.d = d;
  p.out_partial = out_partial;
  p.lse_partial = lse_partial;
  p.hdr = reinterpret_cast<WsHeader*>(ws + wl.hdr);
  p.prefix = reinterpret_cast<int*>(ws + wl.prefix);
  p.ws_o = reinterpret_cast<float*>(ws + wl.ws_o);
  p.ws_lse = reinterpret_cast<float*>(ws + wl.ws_lse);
  p.timeout_ns = host::wait_budget_ns(gqa::kTimeoutNs);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  gqa::gqa_plan_kernel<<<1, 1024, 0, st>>>(d, p.hdr, p.prefix, grid);
  if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
  if (host::ensure_dynamic_smem(reinterpret_cast<const void*>(&gqa::gqa_partial_kernel),
                                gqa::kSmemBytes) != cudaSuccess)
    return MLA_ERR_CUDA;
  cudaLaunchAttribute attr = pdl_attribute();
  void* ev0 = host::g_ev_before.load();
  void* ev1 = host::g_ev_after.load();
  if (ev0 != nullptr && cudaEventRecord(static_cast<cudaEvent_t>(ev0), st) != cudaSuccess)
    return MLA_ERR_CUDA;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(gqa::kThreads);
    cfg.dynamicSmemBytes = gqa::kSmemBytes;
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gqa::gqa_partial_kernel, tm_q, tm_k, tm_v, p) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  if (ev1 != nullptr && cudaEventRecord(static_cast<cudaEvent_t>(ev1), st) != cudaSuccess)
    return MLA_ERR_CUDA;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(U);
    cfg.blockDim = dim3(128);
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gqa::gqa_merge_kernel, d, (const WsHeader*)p.hdr,
                           (const int*)p.prefix, (const float*)p.ws_o, (const float*)p.ws_lse,
                           out_partial, lse_partial) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

mla_status gqa_shard_combine(const float* partials, const float* lses, int num_shards,
                             const gqa_shape* shape, void* out, float* lse_out, void* stream) {
  using host::aligned16;
  if (!partials || !lses || !out || !gqa::shape_ok(shape)) return MLA_ERR_INVALID;
  if (num_shards < 1 || num_shards > kMaxShards) return MLA_ERR_INVALID;
  if (shape->head_dim != gqa::kD) return MLA_ERR_UNSUPPORTED;
  if (!aligned16(partials) || !aligned16(out)) return MLA_ERR_INVALID;
  const int rows = shape->batch * shape->q_len * shape->num_heads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ceil_div(rows, 8));
  cfg.blockDim = dim3(256);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr = pdl_attribute();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gqa::gqa_combine_kernel, partials, lses, num_shards, rows,
                            static_cast<uint16_t*>(out), lse_out) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // extern "C"
