// Shared definitions of the CUDA path: problem constants, the work-unit
// geometry of a (request, shard, query-row group) and the kernel parameter
// blocks.  Included by the kernels and by the host-side C ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mla {

constexpr int kDqk = 576;        // absorbed query/key width: 512 latent + 64 rope
constexpr int kDv = 512;         // value width (the latent c_kv)
constexpr int kDuv = 128;        // per-head up-projected value width
constexpr int kPage = 64;        // tokens per cache page
constexpr int kTile = 64;        // tokens per pipeline tile (MMA N of QK^T)
constexpr int kRows = 64;        // query rows per work unit (MMA M of QK^T)
constexpr int kChunks = 9;       // 576 / 64: 128-byte swizzle chunks per row
constexpr int kChunkBytes = 64 * 128;            // 64 rows x 64 bf16
constexpr int kTileBytes = kChunks * kChunkBytes;  // 73728
constexpr int kCgChunks = 3;     // bf16 kernel: chunks per KV TMA box (one chunk group)
constexpr int kMaxShards = 8;

// Bound on the waits of a kernel's teardown after another wait gave up: the
// MMAs and copies it still has in flight always complete, so this limit is
// independent of the (possibly very short) budget of the ordinary waits.
constexpr unsigned long long kDrainNs = 2000000000ull;

// Error bits written to the workspace error word.
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrBadPage = 2u;
constexpr unsigned kErrQRange = 4u;   // fp8 caches: a non-finite query value
constexpr unsigned kErrQLens = 8u;    // a per-request query count outside [1, q_len]

enum Layout : int { kInterleaved = 0, kContiguous = 1 };

// Workspace header (first 256 bytes of the caller's workspace).
struct WsHeader {
  unsigned err;        // OR of error bits
  int total_cost;      // C: work positions over all units
  int per_cta;         // work positions per persistent CTA
  int grid;            // persistent CTAs
  int num_units;       // U
  int unit_cost;       // overhead positions charged to every unit that has tiles
  int pad[58];
};

// Work positions: unit u owns [prefix[u], prefix[u+1]) -- unit_cost positions
// standing for its fixed costs (query load, epilogue), then one per tile --
// or nothing when it has no tile.  First position of unit u's tiles:
__host__ __device__ inline int unit_tile_start(const int* prefix, int u, int unit_cost) {
  return prefix[u + 1] > prefix[u] ? prefix[u] + unit_cost : prefix[u];
}
static_assert(sizeof(WsHeader) == 256, "header size");

struct ProblemDesc {
  int B, q_len, H;
  int R;               // q_len * H query rows per request
  int G;               // ceil(R / 64) row groups per request
  int num_shards;      // N
  int shard_first;     // first shard computed by this call
  int n_out;           // shards computed by this call (N, or 1)
  int layout;          // Layout: which global positions shard s owns
  int local;           // 1: the cache holds only the computed shard's tokens,
                       // compactly in order (local position p of request b is
                       // page block_table[b][p / 64], row p % 64)
  int causal;
  int num_pages;
  int max_pages;
  // Interleaved shards of a whole-request cache: a tile of shard s covers
  // ppt consecutive pages of the request, and page k's rows of the shard
  // (r_k, r_k + N, ..., r_k = (s - 64 k) mod N) take 2^spp_log2 slots.  When
  // N divides 64, ppt = N and 2^spp_log2 = 64 / N exactly; otherwise (pad = 1)
  // the slots per page are padded (N = 3: 32 slots, 22 rows; N = 5..7: 16
  // slots, 13..10 rows) and slots past a page's rows hold no token.
  int ppt;
  int spp_log2;
  int pad;
  // DCP rank-major I/O (rank_heads = H / ranks > 0): the query rows are read
  // from the all-gathered buffer [ranks, q_batch_total, q_len, rank_heads,
  // 576] (requests q_batch_first..+B of it), and the outputs are written as
  // head slices [ranks, B, q_len, rank_heads, 512] (and [.., rank_heads]),
  // slice k holding heads k*rank_heads.. -- the all-to-all's send layout.
  // 0: both row-major [B, q_len, H, ...].
  int rank_heads;
  int q_batch_total;
  int q_batch_first;
  float scale_log2;    // softmax scale * log2(e)
  const int32_t* block_table;  // [B, max_pages]
  const int32_t* seq_lens;     // [B]
  const int32_t* q_lens;       // [B] query tokens per request, or null (all q_len)
};

struct PartialParams {
  ProblemDesc pd;
  float* out_partial;  // [n_out, B, q_len, H, 512]
  float* lse_partial;  // [n_out, B, q_len, H]
  WsHeader* hdr;
  int* prefix;         // [U + 1] exclusive tile prefix over units
  float* ws_o;         // [grid * 2, 64, 512] split pieces
  float* ws_lse;       // [grid * 2, 64]
  const float* kv_scale;  // fp8 caches: [num_pages * 64]
  const uint16_t* q;      // bf16 [B * R, 576]: the fp8 kernel reads it directly
  int q_one_box;        // 1: tm_q loads all 9 chunks of a 64-row group per box
  const uint8_t* kv_fp8;  // fp8 caches: [num_pages, 64, 576] codes
  unsigned long long timeout_ns;
  int withhold_query;   // testing aid: 1 = never load the first piece's query rows
};

// Geometry of one work unit u = ((b * n_out) + so) * G + g.
struct Unit {
  int b, so, s, g;
  int L;            // context length of request b
  int qn;           // query tokens of request b (rows i >= qn are padding)
  int rows;         // query rows of this group that attend (multiple of 16)
  int rows_out;     // rows of this group in the output (<= 64)
  int tiles;        // pipeline tiles
  int tstart, tend; // contiguous layout: global token range of the shard
  int p0;           // contiguous layout, global cache: first page slot
};

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Walks the work pieces of one persistent CTA: the units whose tile positions
// intersect the CTA's range [lo, hi) of work positions.
struct PieceIter {
  const int* prefix;
  int U, lo, hi, pos, u, uc;
  bool first;
  __device__ void init(const int* pfx, int num_units, int lo_, int hi_, int unit_cost) {
    prefix = pfx;
    U = num_units;
    lo = lo_;
    hi = hi_;
    pos = lo_;
    uc = unit_cost;
    first = true;
    // last unit with prefix[u] <= lo
    int a = 0, b = num_units - 1;
    while (a < b) {
      int m = (a + b + 1) >> 1;
      if (prefix[m] <= lo_) a = m;
      else b = m - 1;
    }
    u = a;
  }
  // Next piece: unit, tile range [t0, t1), whether it is the whole unit, and
  // the workspace slot of a partial piece (0: the CTA's first piece, 1: its
  // last).  Positions of a unit's fixed-cost part hold no tile.
  __device__ bool next(int& unit, int& t0, int& t1, bool& whole, int& slot) {
    while (pos < hi) {
      while (u < U && prefix[u + 1] <= pos) ++u;
      if (u >= U) return false;
      const int ue = prefix[u + 1];
      const int ts = unit_tile_start(prefix, u, uc);
      const int a = max(pos, ts), b = min(hi, ue);
      const int cur = u;
      pos = b;
      ++u;
      if (a >= b) continue;
      unit = cur;
      t0 = a - ts;
      t1 = b - ts;
      whole = (a == ts) && (b == ue);
      slot = first ? 0 : 1;
      first = false;
      return true;
    }
    return false;
  }
};

// Work plan over U units (one 1024-thread block): charges every unit with
// tiles unit_cost extra positions, writes the exclusive prefix of positions
// and the header (positions per CTA for `grid` persistent CTAs).
template <class TilesFn>
__device__ void plan_units(int U, TilesFn tiles_of, WsHeader* hdr, int* prefix, int grid,
                           int min_tiles, int unit_cost, unsigned err_bits) {
  __shared__ int part[1024];
  const int tid = threadIdx.x;
  const int per_thread = ceil_div(U, 1024);
  const int u0 = tid * per_thread, u1 = min(U, u0 + per_thread);
  auto cost = [&](int u) {
    const int t = tiles_of(u);
    return t > 0 ? t + unit_cost : 0;
  };
  int sum = 0;
  for (int u = u0; u < u1; ++u) sum += cost(u);
  part[tid] = sum;
  __syncthreads();
  // inclusive Hillis-Steele scan of the 1024 partial sums
  for (int off = 1; off < 1024; off <<= 1) {
    int v = tid >= off ? part[tid - off] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int run = part[tid] - sum;  // exclusive
  for (int u = u0; u < u1; ++u) {
    prefix[u] = run;
    run += cost(u);
  }
  if (tid == 1023) {
    const int W = part[1023];
    prefix[U] = W;
    hdr->err = err_bits;
    hdr->total_cost = W;
    hdr->per_cta = max(min_tiles, ceil_div(W, grid));
    hdr->grid = grid;
    hdr->num_units = U;
    hdr->unit_cost = unit_cost;
  }
}

// Launch attribute for programmatic dependent launch: the kernel may be
// scheduled while the previous kernel on the stream finishes; it waits for
// that kernel's results with griddep_wait().
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// kLocal: the cache kind, fixed at compile time in the partial kernels --
// 0: whole requests, 1: a local slice (pd.local), 2: whole requests with
// interleaved shards whose count does not divide the page (pd.pad) -- and
// read at run time (-1) elsewhere.
template <int kLocal>
__device__ __forceinline__ bool is_local(const ProblemDesc& pd) {
  return kLocal < 0 ? pd.local != 0 : kLocal == 1;
}
template <int kLocal>
__device__ __forceinline__ bool is_pad(const ProblemDesc& pd) {
  return kLocal < 0 ? pd.pad != 0 : kLocal == 2;
}

template <int kLocal = -1>
__device__ __forceinline__ Unit make_unit(const ProblemDesc& pd, int u) {
  Unit x;
  x.g = u % pd.G;
  int bs = u / pd.G;
  x.so = bs % pd.n_out;
  x.b = bs / pd.n_out;
  x.s = pd.shard_first + x.so;
  x.L = pd.seq_lens[x.b];
  x.qn = pd.q_lens ? min(max(pd.q_lens[x.b], 0), pd.q_len) : pd.q_len;
  int r0 = x.g * kRows;
  x.rows_out = min(kRows, pd.R - r0);
  x.rows = min(max(x.qn * pd.H - r0, 0), x.rows_out);
  x.tstart = 0;
  x.tend = 0;
  x.p0 = 0;
  int L = x.L > 0 ? x.L : 0;
  if (x.rows == 0) L = 0;   // only padding rows: nothing to attend
  if (pd.layout == kInterleaved) {
    int n_local = L > x.s ? (L - 1 - x.s) / pd.num_shards + 1 : 0;
    if (is_pad<kLocal>(pd)) {
      // tiles up to the page of the shard's last position
      x.tiles = n_local > 0 ? ((x.s + pd.num_shards * (n_local - 1)) / kPage) / pd.ppt + 1 : 0;
    } else {
      x.tiles = ceil_div(n_local, kTile);
    }
  } else {
    int c = ceil_div(L, pd.num_shards);
    x.tstart = x.s * c;
    x.tend = min(x.tstart + c, L);
    if (x.tstart >= x.tend) {
      x.tiles = 0;
    } else if (is_local<kLocal>(pd)) {
      x.tiles = ceil_div(x.tend - x.tstart, kTile);
    } else {
      x.p0 = x.tstart / kPage;
      x.tiles = (x.tend - 1) / kPage - x.p0 + 1;
    }
  }
  return x;
}

// Row of out_partial / lse_partial that holds row `row` (0..63) of unit x's
// query group.
__device__ __forceinline__ size_t out_row(const ProblemDesc& pd, const Unit& x, int row) {
  const int rr = x.g * kRows + row;            // i * H + h within the request
  if (pd.rank_heads == 0) return ((size_t)x.so * pd.B + x.b) * pd.R + rr;
  const int i = rr / pd.H, h = rr - i * pd.H;
  const int k = h / pd.rank_heads, hl = h - k * pd.rank_heads;
  return (((size_t)k * pd.B + x.b) * pd.q_len + i) * pd.rank_heads + hl;
}

// Query rows per TMA box in the rank-major mode: a run of one rank's heads
// of one query position (rank_heads is a multiple of 8 that divides 64 or is
// a multiple of 64), and the gathered-buffer row of row `row` of x's group.
__device__ __forceinline__ int q_run_rows(const ProblemDesc& pd) {
  return pd.rank_heads < kRows ? pd.rank_heads : kRows;
}
__device__ __forceinline__ int q_src_row(const ProblemDesc& pd, const Unit& x, int row) {
  const int rr = x.g * kRows + row;
  const int i = rr / pd.H, h = rr - i * pd.H;
  const int k = h / pd.rank_heads, hl = h - k * pd.rank_heads;
  return ((k * pd.q_batch_total + pd.q_batch_first + x.b) * pd.q_len + i) * pd.rank_heads + hl;
}

// Global token position of slot a (0..63) of tile j of unit x.  Interleaved
// shards: tile j holds the shard's positions 64j..64j+63 (in a local cache,
// exactly local page j).  Contiguous shards: tile j is global page p0 + j, or
// local page j of a local cache.
// The first row of shard s in page `page` of an interleaved whole-request
// cache: (s - 64 page) mod N.
__host__ __device__ __forceinline__ int shard_row0(int s, int page, int n) {
  const int v = (s - (kPage % n) * (page % n)) % n;
  return v < 0 ? v + n : v;
}

// A position past every context: the slot holds no token.
constexpr int kNoToken = 0x3fffffff;

template <int kLocal = -1>
__device__ __forceinline__ int slot_token(const ProblemDesc& pd, const Unit& x, int j, int a) {
  if (pd.layout == kInterleaved) {
    if (is_pad<kLocal>(pd)) {
      const int page = pd.ppt * j + (a >> pd.spp_log2);
      const int row = shard_row0(x.s, page, pd.num_shards) +
                      pd.num_shards * (a & ((1 << pd.spp_log2) - 1));
      return row < kPage ? page * kPage + row : kNoToken;
    }
    return (j * kTile + a) * pd.num_shards + x.s;
  }
  if (is_local<kLocal>(pd)) return x.tstart + j * kTile + a;
  return (x.p0 + j) * kPage + a;
}

__device__ __forceinline__ bool slot_valid(const ProblemDesc& pd, const Unit& x, int t) {
  if (pd.layout == kInterleaved) return t < x.L;
  return t >= x.tstart && t < x.tend;
}

// True when every slot of tile j is a valid token visible to every query row
// of the unit (no masking needed).
template <int kLocal = -1>
__device__ __forceinline__ bool tile_full(const ProblemDesc& pd, const Unit& x, int j) {
  int first = slot_token<kLocal>(pd, x, j, 0), last = slot_token<kLocal>(pd, x, j, kTile - 1);
  bool ok = slot_valid(pd, x, first) && slot_valid(pd, x, last);
  if (pd.causal) {
    int i_min = (x.g * kRows) / pd.H;  // smallest query position in the group
    ok = ok && last <= x.L - x.qn + i_min;
  }
  return ok;
}

}  // namespace mla
