/*
 * mla_dcp.h -- C ABI of the sequence-sharded MLA decode library (sm_103a).
 *
 * The operation is the data-parallel core of Decode Context Parallelism
 * ("Decode Context Parallelism", sections 4 and 4.1): the latent KV cache of
 * a multi-head latent attention (MLA) model is split along the sequence;
 * every shard attends the full query over only its slice and emits a partial
 * output plus a log-sum-exp (LSE); a combine step reweights the partials by
 * their LSEs, optionally fused with the per-head value up-projection
 * ("Kimi K3 in vLLM: Specialized CuTe DSL Decode on NVIDIA GB300",
 * section 1).  On one GPU the N shards are logical partitions of the cache.
 *
 * Conventions for every entry point:
 *   - Pointers named "device" must be device memory of the current CUDA
 *     device, 16-byte aligned (4-byte for the int32 arrays block_table,
 *     seq_lens and q_lens, so that views of a larger batch can be passed).
 *     The caller owns every buffer; the library
 *     keeps no pointer after a call returns and allocates no device memory
 *     at run time (its one static buffer, the scratch of
 *     mla_decode_partial_noalloc, exists from library load to process exit).
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream).  Argument errors are detected on
 *     the host and returned before anything is launched.
 *   - No C++ exception crosses this boundary.
 *   - Results are deterministic: the same inputs give bitwise-identical
 *     outputs (fixed reduction order, no atomics on data).
 *
 * Layouts (row-major, bf16 = IEEE bfloat16 bit patterns in uint16):
 *   q            bf16  [B, q_len, H, 576]  absorbed queries: 512 latent + 64 rope
 *   kv data      bf16  [num_pages, 64, 576]  latent rows [c_kv(512) | k_rope(64)]
 *                e4m3  [num_pages, 64, 576]  (fp8 caches, OCP e4m3 codes)
 *   kv scale     fp32  [num_pages, 64]     fp8 only: value = e4m3(code) * scale
 *   block_table  int32 [B, max_pages_per_req]  page of token t of request b is
 *                                          block_table[b][t / 64], row t % 64
 *   seq_lens     int32 [B]                 context length L_b (>= 1), device
 *   out_partial  fp32  [n_out, B, q_len, H, 512]  normalised partial outputs
 *   lse_partial  fp32  [n_out, B, q_len, H]       natural-log LSE, -inf if empty
 *   w_uv         bf16  [H, 512, 128]       per-head value up-projection
 *   out          bf16  [B, q_len, H, 512]  (or [B, q_len, H, 128] with w_uv)
 *   lse_out      fp32  [B, q_len, H]
 */
#ifndef MLA_DCP_H_
#define MLA_DCP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID = -1,       /* bad argument; nothing was launched */
  MLA_ERR_UNSUPPORTED = -2,   /* well-formed but outside what this build supports */
  MLA_ERR_CUDA = -3,          /* a CUDA runtime or driver call failed */
  MLA_ERR_TIMEOUT = -4,       /* a device-side wait gave up (from mla_get_device_error) */
  MLA_ERR_DEVICE_BOUNDS = -5, /* a block-table entry was outside [0, num_pages) */
  MLA_ERR_WORKSPACE = -6,     /* workspace missing or smaller than mla_workspace_size() */
  MLA_ERR_RANGE = -7          /* fp8 cache: an inf or NaN query value in a row that attends */
} mla_status;

/* Which token positions of a request belong to shard s of N
 * ("Decode Context Parallelism", section 4):
 *   INTERLEAVED  t mod N == s                  (any N <= 8)
 *   CONTIGUOUS   s*c <= t < min((s+1)*c, L),   c = ceil(L / N)
 * The section's worked example (a 200K-token request on 4 GPUs holding
 * 0-50K, 50K-100K, 100K-150K, 150K-200K) is the CONTIGUOUS layout.
 * With these two the cache and block table describe whole requests (every
 * position t at page block_table[b][t / 64], row t % 64).
 *
 * The *_LOCAL layouts are the same shards, stored the way each GPU of a
 * multi-GPU deployment holds its slice (section 4: each GPU stores only its
 * chunk): the cache and block table hold only shard `shard_id`'s positions,
 * in order, compactly -- local position p of request b is page
 * block_table[b][p / 64], row p % 64, and is global position p*N + s
 * (INTERLEAVED_LOCAL, any N <= 8) or s*c + p (CONTIGUOUS_LOCAL).  seq_lens
 * stay the global lengths L_b: they fix the shard's token count and the
 * causal mask.  shard_id must name one shard. */
typedef enum mla_layout {
  MLA_LAYOUT_INTERLEAVED = 0,
  MLA_LAYOUT_CONTIGUOUS = 1,
  MLA_LAYOUT_INTERLEAVED_LOCAL = 2,
  MLA_LAYOUT_CONTIGUOUS_LOCAL = 3
} mla_layout;

typedef enum mla_kv_dtype { MLA_KV_BF16 = 0, MLA_KV_FP8_E4M3 = 1 } mla_kv_dtype;

/* Decode-step shape.  num_heads must be a multiple of 16.  With an fp8
 * cache the tensor cores take each query row as a two-term e4m3 sum under a
 * power-of-two row scale (exact for components within 2^10 of the row's
 * largest; any finite bf16 value is accepted); an inf or NaN component of a
 * row that attends is reported as MLA_ERR_RANGE by mla_get_device_error.
 * With causal != 0
 * (a speculative verify step of q_len = 1 + drafts tokens whose KV is the
 * last q_len entries of the cache), query i sees tokens t <= L - q_len + i. */
typedef struct mla_shape {
  int batch;            /* B >= 1 */
  int q_len;            /* query tokens per request >= 1 (the padded count, see q_lens) */
  int num_heads;        /* H: multiple of 16 */
  int causal;           /* 0 or 1 */
  float softmax_scale;  /* logits = softmax_scale * q . k  (1/sqrt(192) for the workloads here) */
  /* Optional (NULL = every request has q_len query tokens), device int32
   * [B]: request b has q_lens[b] in [1, q_len] query tokens -- a batch of
   * verify steps with different draft counts padded to q_len.  Rows
   * i >= q_lens[b] are padding: their partials are o = 0, lse = -inf and
   * their combined output is 0.  With causal, query i of request b sees
   * t <= L_b - q_lens[b] + i.  A value outside [1, q_len] is clamped and
   * reported as MLA_ERR_INVALID by mla_get_device_error.  Ignored by
   * mla_shard_combine and mla_workspace_size. */
  const int32_t* q_lens;
} mla_shape;

/* The paged latent cache (device memory, not modified). */
typedef struct mla_kv_pages {
  const void* data;     /* [num_pages, page_size, 576] bf16 or e4m3 */
  const float* scale;   /* fp8 only: [num_pages, page_size]; must be NULL for bf16 */
  mla_kv_dtype dtype;
  int num_pages;        /* >= 1 */
  int page_size;        /* must be 64 */
} mla_kv_pages;

/* shard_id value that computes every shard 0..N-1 in one call (n_out = N). */
#define MLA_ALL_SHARDS (-1)

/*
 * Bytes of device workspace mla_decode_partial needs for this shape on the
 * current device (work list, split-piece partials and an error word).
 * Returns 0 for invalid arguments.
 */
size_t mla_workspace_size(const mla_shape* shape, int num_shards, int shard_id);

/*
 * Per-shard partial attention ("Decode Context Parallelism", section 4.1,
 * the "Compute" step; section 5.3: each rank attends over its latent slice).
 * For every request b, query row (i, h) and computed shard s, over the tokens
 * T_s of request b that shard s owns (see mla_layout) and the query may see:
 *     s_t = softmax_scale * q[b,i,h,:] . K_t            (K_t = cache row, 576 wide)
 *     lse_partial = ln sum_{t in T_s} exp(s_t)           (-inf if T_s is empty)
 *     out_partial = sum_{t in T_s} exp(s_t - lse) * K_t[0:512]   (0 if empty)
 * shard_id = MLA_ALL_SHARDS computes all N shards (out_partial holds N
 * slices, shard-major); shard_id in [0, N) computes that shard only
 * (n_out = 1), which is the per-GPU call of a multi-GPU deployment.
 *
 * Arguments: q, block_table, seq_lens, out_partial, lse_partial, workspace:
 * device pointers, layouts above.  max_pages_per_req: row stride of
 * block_table; it must cover the pages of every request (ceil(L_b / 64), or
 * ceil(n_s / 64) for a local layout holding n_s of the request's positions;
 * only those entries are read).  num_shards: 1..8.  workspace_bytes must be at
 * least mla_workspace_size(shape, num_shards, shard_id).
 *
 * Errors: MLA_ERR_INVALID / MLA_ERR_UNSUPPORTED / MLA_ERR_WORKSPACE before
 * any launch; MLA_ERR_CUDA if a launch fails.  Device-side problems (a
 * block-table entry out of range, which then reads as zeros; a wait that
 * timed out) are recorded in the workspace and read with
 * mla_get_device_error.
 */
mla_status mla_decode_partial(const void* q, const mla_kv_pages* kv, const int32_t* block_table,
                              int max_pages_per_req, const int32_t* seq_lens,
                              const mla_shape* shape, int shard_id, int num_shards,
                              mla_layout layout, float* out_partial, float* lse_partial,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * The per-rank call of a multi-GPU DCP step with the exchanges' own layouts
 * ("Decode Context Parallelism", section 4.1: AllGather Q -> Compute -> a
 * combine of the partials; "Kimi K3 Performance Optimizations in vLLM",
 * section "Decode context parallelism": the partial outputs and LSEs travel
 * by an all-to-all).  Computes what mla_decode_partial computes for shard
 * `rank` of `num_ranks` (shard_id = rank, num_shards = num_ranks) with no copy
 * around it:
 *   q_gathered: bf16 [num_ranks, batch_total, q_len, H/num_ranks, 576], the
 *     all-gather of every rank's query heads as it lands (rank k's block
 *     holds heads k*H/num_ranks ..); this call computes requests
 *     batch_first .. batch_first + shape->batch - 1 of it.
 *   block_table, seq_lens (and shape->q_lens): those requests' rows.
 *   out_send: fp32 [num_ranks, shape->batch, q_len, H/num_ranks, 512];
 *   lse_send: fp32 [num_ranks, shape->batch, q_len, H/num_ranks]: slice k
 *     holds this shard's partial of heads k*H/num_ranks .., i.e. the send
 *     buffers of an all-to-all after which rank k holds every shard's
 *     partial of its own heads, shard-major, as mla_shard_combine takes
 *     them.
 * layout: MLA_LAYOUT_INTERLEAVED_LOCAL or MLA_LAYOUT_CONTIGUOUS_LOCAL (the
 * rank's own slice of the cache; else MLA_ERR_INVALID).  H must be a multiple
 * of num_ranks with H/num_ranks a multiple of 8 that divides 64 or is a
 * multiple of 64 (else MLA_ERR_UNSUPPORTED).  Other
 * arguments, the workspace (mla_workspace_size(shape, num_ranks, rank)) and
 * errors as for mla_decode_partial.
 */
mla_status mla_decode_partial_dcp(const void* q_gathered, int batch_total, int batch_first,
                                  const mla_kv_pages* kv, const int32_t* block_table,
                                  int max_pages_per_req, const int32_t* seq_lens,
                                  const mla_shape* shape, int rank, int num_ranks,
                                  mla_layout layout, float* out_send, float* lse_send,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode_partial without a workspace argument, for callers that cannot
 * allocate device memory (for example code running while a serving engine's
 * pool already owns the whole GPU, allocator or out-of-memory callbacks, or
 * loops where an allocation is not allowed).  The pages this library follows
 * have no counterpart of this call; it exists only for such callers.
 *
 * The work list and split partial results live in a fixed scratch buffer
 * that the library keeps in device memory: about 40 MiB on every GPU that
 * loads the library, held until the process exits.  Shapes whose workspace
 * (mla_workspace_size) would exceed it, i.e. more than 8192 work units
 * (batch x computed shards x ceil(q_len * num_heads / 64)) or a GPU with
 * more than 160 SMs, return MLA_ERR_UNSUPPORTED before any launch.
 * Arguments, layouts, results and host-side errors are those of
 * mla_decode_partial.
 *
 * The first call in a CUDA context (normally: on a device) looks up the
 * scratch's device address (cudaGetSymbolAddress) and keeps it for that
 * context; make that first call before any stream capture.  All calls on a
 * device share the one scratch buffer, so calls whose kernels overlap on the
 * GPU (different streams, or different host threads) race: order them on
 * one stream.  Nothing needs clearing between calls; each call rebuilds what
 * it reads.  Device-side errors (a bad block-table page, a wait that timed
 * out) are kept in the scratch's error word: read them with
 * mla_get_device_error_noalloc.
 */
mla_status mla_decode_partial_noalloc(const void* q, const mla_kv_pages* kv,
                                      const int32_t* block_table, int max_pages_per_req,
                                      const int32_t* seq_lens, const mla_shape* shape,
                                      int shard_id, int num_shards, mla_layout layout,
                                      float* out_partial, float* lse_partial, void* stream);

/*
 * The device error word of mla_decode_partial_noalloc's scratch on the
 * current device: synchronises `stream`, reads and clears it, with the
 * results of mla_get_device_error.  Like the entry point it serves, this has
 * no counterpart on the pages; it lets callers that cannot allocate see a
 * bad block-table page or a timed-out wait.  It reads the state left by the
 * last mla_decode_partial_noalloc on the device, whatever its stream.
 */
mla_status mla_get_device_error_noalloc(void* stream);

/*
 * LSE combine of N shard partials ("Decode Context Parallelism", section 4.1:
 * partial outputs reweighted by their LSE and summed into the true output):
 *     M = max_s lse_s,  w_s = exp(lse_s - M),  lse_out = M + ln sum_s w_s
 *     o = sum_s w_s out_s / sum_s w_s                  (fp32)
 *     out = bf16(o)                                    if w_uv == NULL
 *     out = bf16(o . w_uv[h])  ([B,q_len,H,128])       otherwise (the fused
 *           v-projection of "Kimi K3 in vLLM ...", section 1)
 * partials / lses: as written by mla_decode_partial with MLA_ALL_SHARDS (or
 * the N per-shard slices stacked shard-major).  lse_out may be NULL.
 * A row whose shards are all empty gives out = 0 and lse_out = -inf.
 */
mla_status mla_shard_combine(const float* partials, const float* lses, int num_shards,
                             const mla_shape* shape, const void* w_uv, void* out, float* lse_out,
                             void* stream);

/*
 * One whole decode step on one GPU: every shard's partial attention
 * (mla_decode_partial with MLA_ALL_SHARDS) and their LSE combine
 * (mla_shard_combine, optionally fused with W_UV) in one call, with the shard
 * partials kept in the workspace instead of caller buffers.  The N shards are
 * logical partitions of the cache ("Decode Context Parallelism", section 4.1:
 * Compute, then the LSE reweighting of the partials into the true output).
 * A shard's unit that the work split divides between several CTAs leaves one
 * partial per CTA; these pieces are merged together with the other shards'
 * partials in the combine itself (the LSE merge is associative), so no merged
 * per-shard partial is written.  With w_uv and B * q_len >= 64 query rows per
 * head, the combine writes the output o in bf16 into the workspace and the
 * W_UV projection runs as one tensor-core GEMM per head (o rounded to bf16
 * before the product, as when projecting the unfused bf16 output); with
 * fewer rows the combine projects on the fly.
 *
 * Arguments as for mla_decode_partial and mla_shard_combine; layout must be
 * MLA_LAYOUT_INTERLEAVED or MLA_LAYOUT_CONTIGUOUS.  out: bf16
 * [B, q_len, H, 512], or [B, q_len, H, 128] with w_uv; lse_out: fp32
 * [B, q_len, H] or NULL.  workspace_bytes must be at least
 * mla_decode_step_workspace_size(shape, num_shards).  Device-side errors are
 * read with mla_get_device_error(workspace, stream).
 */
size_t mla_decode_step_workspace_size(const mla_shape* shape, int num_shards);
mla_status mla_decode_step(const void* q, const mla_kv_pages* kv, const int32_t* block_table,
                           int max_pages_per_req, const int32_t* seq_lens, const mla_shape* shape,
                           int num_shards, mla_layout layout, const void* w_uv, void* out,
                           float* lse_out, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * Synchronises `stream`, reads and clears the device error word kept in
 * `workspace` by the last mla_decode_partial on it.  Returns MLA_OK,
 * MLA_ERR_TIMEOUT, MLA_ERR_DEVICE_BOUNDS, MLA_ERR_RANGE or MLA_ERR_INVALID (a
 * q_lens entry out of range), in that order of precedence when several
 * occurred, or MLA_ERR_CUDA.
 */
mla_status mla_get_device_error(void* workspace, void* stream);

/*
 * Testing and diagnostic aid (not part of the method): sets the time limit,
 * in nanoseconds, of every device-side wait of the partial-attention kernels
 * launched from now on (process-wide, any thread).  A wait that runs out
 * makes its kernel stop early, with MLA_ERR_TIMEOUT in the error word and
 * its outputs undefined; the kernel still lets its own copies and tensor-core
 * operations finish and releases its tensor memory, so later calls work
 * normally.  0 restores the default of 2 s.  Always MLA_OK.
 */
mla_status mla_set_wait_budget_ns(unsigned long long ns);

/*
 * Testing aid (not part of the method): while `on` is non-zero, the
 * partial-attention kernels of mla_decode_partial launched from now on never
 * load the query rows of each CTA's first piece of work (process-wide).  The
 * waits for those rows cannot succeed, so each CTA stops once its wait
 * budget (mla_set_wait_budget_ns) runs out, and mla_get_device_error then
 * reads MLA_ERR_TIMEOUT; outputs are undefined.  This exercises the
 * time-out path without any fault.  0 turns it off.  Always MLA_OK.
 */
mla_status mla_set_withhold_query(int on);

/*
 * Profiling aid (not part of the method): while set, every later
 * mla_decode_partial call (both entry points, any thread) records
 * `before_partial` and `after_partial` -- two cudaEvent_t handles passed as
 * void*, owned by the caller -- on its stream immediately before and after
 * the launch of its partial-attention kernel, so that kernel's device time
 * can be read without the planning and merge kernels around it.  Pass two
 * NULLs to stop.  Exactly one NULL is MLA_ERR_INVALID.  The caller keeps the
 * events alive while they are set; the setting is process-wide.
 */
mla_status mla_set_profile_events(void* before_partial, void* after_partial);

/*
 * Grouped-query attention (GQA) with the same sequence sharding ("Decode
 * Context Parallelism", section 5.4, the GQA backend): the cache stores
 * num_kv_heads KV heads of width head_dim in separate K and V caches, and
 * query head h attends with KV head h / (num_heads / num_kv_heads) (each KV
 * head broadcast over its group of consecutive query heads).
 *
 *   q            bf16  [B, q_len, H, D]
 *   k, v         bf16  [num_pages, 64, Hkv, D]   (token t of request b at
 *                                                 page block_table[b][t / 64],
 *                                                 row t % 64)
 *   out_partial  fp32  [n_out, B, q_len, H, D]
 *   lse_partial  fp32  [n_out, B, q_len, H]
 *   out          bf16  [B, q_len, H, D]
 *
 * This build supports head_dim = 128 and groups H / Hkv that are powers of
 * two up to 64; layouts INTERLEAVED and CONTIGUOUS.  Everything else matches
 * the MLA calls: logits scaled by softmax_scale (1/sqrt(D) for the workloads
 * here), causal verify steps, shard_id / MLA_ALL_SHARDS, workspace, error
 * reporting through mla_get_device_error, asynchronous on `stream`.
 */
typedef struct gqa_shape {
  int batch;            /* B >= 1 */
  int q_len;            /* query tokens per request >= 1 */
  int num_heads;        /* H */
  int num_kv_heads;     /* Hkv, divides H */
  int head_dim;         /* D: 128 */
  int causal;           /* 0 or 1 */
  float softmax_scale;
} gqa_shape;

typedef struct gqa_kv_pages {
  const void* k;        /* bf16 [num_pages, page_size, Hkv, D] */
  const void* v;        /* bf16 [num_pages, page_size, Hkv, D] */
  int num_pages;        /* >= 1 */
  int page_size;        /* must be 64 */
} gqa_kv_pages;

/* Workspace bytes gqa_decode_partial needs (0 for invalid or unsupported shapes). */
size_t gqa_workspace_size(const gqa_shape* shape, int num_shards, int shard_id);

/* Per-shard partial GQA attention: for every request b, query row (i, h) and
 * computed shard s, over the shard's visible tokens T_s:
 *   s_t = softmax_scale * q[b,i,h,:] . K_t[kh,:],  kh = h / (H / Hkv)
 *   lse_partial = ln sum exp(s_t)  (-inf if empty);
 *   out_partial = sum exp(s_t - lse) V_t[kh,:]  (0 if empty). */
mla_status gqa_decode_partial(const void* q, const gqa_kv_pages* kv, const int32_t* block_table,
                              int max_pages_per_req, const int32_t* seq_lens,
                              const gqa_shape* shape, int shard_id, int num_shards,
                              mla_layout layout, float* out_partial, float* lse_partial,
                              void* workspace, size_t workspace_bytes, void* stream);

/* LSE combine of N GQA shard partials (head_dim wide) into bf16 out
 * [B, q_len, H, D] and lse_out (may be NULL). */
mla_status gqa_shard_combine(const float* partials, const float* lses, int num_shards,
                             const gqa_shape* shape, void* out, float* lse_out, void* stream);

/* Static description of a status code. */
const char* mla_status_string(mla_status status);

/* Library version: major * 10000 + minor * 100 + patch.  0.2.0 added
 * mla_shape.q_lens, the *_LOCAL layouts and MLA_ERR_RANGE. */
int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DCP_H_ */
