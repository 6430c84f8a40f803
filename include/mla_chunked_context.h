/*
 * mla_chunked_context.h -- C ABI of the GB300 (sm_103a) MLA chunked-context
 * prefill library, libmla_gb300.so.
 *
 * The method (three vLLM pull-request reports):
 *   - PR #50613 ("MLA prefill schedules chunks per request"): a host planner
 *     packs each request's cached context into workspace-sized chunks, cutting
 *     an overflowing request at an aligned length; per chunk the context rows
 *     are gathered once into a workspace, attended, and merged into a context
 *     partial (O, LSE) that starts as O=0, LSE=-inf for requests without
 *     context.
 *   - PR #36540 ("Remove trtllm ragged mla prefills"): merge_attn_states takes
 *     prefix_num_tokens; tokens at or past it copy the suffix output.
 *   - PR #49294 ("Ignore empty MLA context chunks during merge"): rows with an
 *     empty context carry LSE=-inf and O=0 and must merge without NaN.
 * The MLA arithmetic (latent cache -> W_kv_b up-projection into K_nope and V,
 * attention over concat(K_nope, k_pe)) is the standard MLA prefill.
 *
 * Conventions for every call
 *   - Return value: MLA_OK (0) or a negative MLA_ERR_* code.  Arguments are
 *     validated on the host before anything is enqueued; on an error nothing
 *     has been enqueued.
 *   - The caller owns all memory.  The library allocates no device memory,
 *     with one exception: the fixed device array behind
 *     mla_context_chunk_attn_noalloc.  Calls that need scratch take a
 *     caller-provided device workspace whose size a *_workspace_bytes query
 *     returns; workspaces must be 16-byte aligned.
 *   - Kernels: bf16 storage with the DeepSeek-V3 head shape (L 512, P 64,
 *     Dn 128, Dv 128) runs on the tcgen05 tensor-core kernels only.  Such a
 *     call needs an sm_103a GPU and 16-byte aligned q, latent / new_latent,
 *     kv_cache, w_kv_b and K/V pointers, else it returns MLA_ERR_UNSUPPORTED
 *     before anything is enqueued; it never falls back to the CUDA-core
 *     kernels.  Those serve float32 storage and all other head shapes.
 *   - "device" pointers are CUDA device pointers of the current device;
 *     work is enqueued on `stream` (a cudaStream_t, NULL = legacy default
 *     stream) and nothing synchronises unless stated.  "host" pointers are
 *     read before the call returns.
 *   - Layouts (row-major, contiguous):
 *       q            [T, H, Dn+P]            (nope first, then rope)
 *       kv_cache     [num_blocks, block_size, L+P]  (c_kv first, then k_pe)
 *       block_table  [R, block_table_stride] int32 physical block ids
 *       new_latent   [T, L+P]                latent rows of the new tokens
 *       w_kv_b       [H*(Dn+Dv), L]          rows h*(Dn+Dv)+[0,Dn) -> K_nope,
 *                                            the next Dv rows -> V
 *       O            [T, H, Dv];  LSE [H, T] float32, natural log
 *     T = number of new tokens, H = heads, L = kv_lora_rank, P = rope dim,
 *     Dn = qk_nope_dim, Dv = v_dim, R = requests.  Tokens of request r are
 *     rows [qsl[r], qsl[r+1]) where qsl is the prefix sum of query lengths.
 *   - dtype (mla_dims_t.dtype) is the storage type of q, kv_cache,
 *     new_latent, w_kv_b and of the final output O.  Arithmetic is float32
 *     (tensor-core products of bf16 operands accumulate in float32).
 *   - dev_status (nullable, device int32): kernels OR MLA_STATUS_* bits into
 *     it; the caller clears it and checks it when it chooses to.
 *       MLA_STATUS_BAD_BLOCK   a block id outside [0, num_blocks) was met;
 *                              that row was read as zeros.
 *       MLA_STATUS_FP16_RANGE  a value rounded to fp16 (q_nope on the
 *                              tensor-core path, or an up-projected K/V
 *                              element stored as fp16) had magnitude >= 65520
 *                              and became +-inf: results that depend on it
 *                              are not valid (bf16 keeps its range, fp16
 *                              does not; the tensor-core path uses fp16 for
 *                              its 3 extra mantissa bits).
 */
#ifndef MLA_CHUNKED_CONTEXT_H
#define MLA_CHUNKED_CONTEXT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

typedef void *mla_stream_t; /* cudaStream_t */

enum {
  MLA_OK = 0,
  MLA_ERR_INVALID = -1,        /* bad argument (null pointer, bad size)        */
  MLA_ERR_TOO_SMALL = -2,      /* output array or workspace too small          */
  MLA_ERR_PLANNER_STUCK = -3,  /* no aligned split fits an empty chunk         */
  MLA_ERR_CUDA = -4,           /* a CUDA launch or runtime call failed         */
  MLA_ERR_UNSUPPORTED = -5     /* dims / dtype combination not supported       */
};

/* Element types.  mla_dims_t.dtype (the inputs and the final output) is F32
 * or BF16; F16 is used for the up-projected K/V workspace (see
 * mla_kv_up_proj). */
enum { MLA_DTYPE_F32 = 0, MLA_DTYPE_BF16 = 1, MLA_DTYPE_F16 = 2 };

/* Bits of the caller's dev_status word (see the conventions above). */
enum { MLA_STATUS_BAD_BLOCK = 1, MLA_STATUS_FP16_RANGE = 2 };

/* Bits of mla_device_error_flags(). */
enum { MLA_DEVICE_ERR_WAIT_TIMEOUT = 1 };

typedef struct {
  int32_t num_heads;     /* H  */
  int32_t kv_lora_rank;  /* L  */
  int32_t qk_rope_dim;   /* P  */
  int32_t qk_nope_dim;   /* Dn */
  int32_t v_dim;         /* Dv */
  int32_t block_size;    /* rows per paged-cache block */
  float softmax_scale;   /* score = scale * (q_nope.k_nope + q_pe.k_pe) */
  int32_t dtype;         /* MLA_DTYPE_* storage type, see above */
} mla_dims_t;

/* One chunk of the plan (PR #50613 report, key source snippet
 * _ContextChunkPlan): requests [request_start, request_end); their entries
 * are starts[entry_offset + i] / seq_lens[entry_offset + i]. */
typedef struct {
  int32_t request_start;
  int32_t request_end;
  int32_t entry_offset;
  int32_t rows;            /* padded workspace rows the chunk uses */
  int32_t is_continuation; /* 1 when starts[entry_offset] > 0 */
} mla_chunk_t;

/* ---------------------------------------------------------------------------
 * mla_plan_context_chunks  (host only; PR #50613 report, "implementation
 * breakdown" item 2 and key source snippet plan_mla_context_chunks /
 * aligned_split_len)
 *
 * Packs the context rows of requests 0..num_requests-1, in order, into chunks
 * of at most row_budget padded rows.  Requests with context_lens[r] == 0 are
 * in no chunk.  A request that overflows the chunk is cut at the largest
 * multiple of split_alignment that is <= max_context_chunk, < its remaining
 * rows, and fits; the chunk then closes (also when no such length exists, in
 * which case the request opens the next chunk).
 *   context_lens   host [num_requests], >= 0
 *   padded_rows    optional callback mapping a context offset to padded
 *                  workspace rows (non-decreasing); NULL = identity
 *   chunks, starts, seq_lens: host outputs.  Call with all three NULL (and
 *                  caps 0) to get *num_chunks / *num_entries only.
 * Errors: MLA_ERR_INVALID (negative length, budget/alignment < 1),
 *         MLA_ERR_PLANNER_STUCK (a request cannot be placed even in an empty
 *         chunk: row_budget smaller than one aligned split),
 *         MLA_ERR_TOO_SMALL (caps below the counts; the counts are still set).
 */
int mla_plan_context_chunks(const int32_t *context_lens, int32_t num_requests,
                            int32_t row_budget, int32_t max_context_chunk,
                            int32_t split_alignment,
                            int64_t (*padded_rows)(int64_t, void *),
                            void *padded_rows_ctx, mla_chunk_t *chunks,
                            int32_t chunks_cap, int32_t *starts,
                            int32_t *seq_lens, int32_t entries_cap,
                            int32_t *num_chunks, int32_t *num_entries);

/* ---------------------------------------------------------------------------
 * merge_attn_states  (PR #36540 report, "implementation breakdown", CUDA
 * kernel layer; PR #49294 report, test_merge_attn_states_both_empty)
 *
 * Per token t < num_tokens and head h:
 *   t >= prefix_num_tokens       -> out = suffix (prefix never read)
 *   both LSE = -inf              -> out O = 0, LSE = -inf
 *   one LSE = -inf               -> the other side (the empty side's O is
 *                                   never read)
 *   otherwise                    -> LSE-weighted average, new LSE =
 *                                   m + ln(e^(pL-m) + e^(sL-m))
 *   out, prefix_o, suffix_o  device [T, H, D]; in_dtype for the two inputs,
 *                            out_dtype for out (bf16 output is rounded to
 *                            nearest even)
 *   prefix_lse, suffix_lse   device float32 [H, T];  out_lse nullable
 *   head_dim must be a multiple of 8.  out, prefix_o and suffix_o must be
 *   16-byte aligned and the LSE arrays 4-byte aligned (O moves as 16-byte
 *   vectors), else MLA_ERR_INVALID.  out may alias either input O (each
 *   element is read before it is written, by the same thread); out_lse must
 *   not alias an input LSE (one LSE is read by all threads of its row).
 */
int merge_attn_states(void *out, float *out_lse, const void *prefix_o,
                      const float *prefix_lse, const void *suffix_o,
                      const float *suffix_lse, int32_t num_tokens,
                      int32_t num_heads, int32_t head_dim,
                      int32_t prefix_num_tokens, int32_t in_dtype,
                      int32_t out_dtype, mla_stream_t stream);

/* ---------------------------------------------------------------------------
 * Per-step calls of the chunk pipeline.  They exist so that every step can be
 * tested and timed on its own; mla_context_chunk_attn and mla_chunked_prefill
 * run them in order.
 *
 * mla_gather_context_rows  (PR #50613 report, item 2: every context row of a
 * chunk is gathered exactly once)
 *   For seq i < num_seqs (request seq_request[i], rows [seq_start[i],
 *   seq_start[i] + cu_rows[i+1] - cu_rows[i]) of its context) copies cache row
 *   j = kv_cache[block_table[r][j / bs]][j % bs][0 : L+P] to latent_ws row
 *   cu_rows[i] + (j - seq_start[i]).
 *   seq_request, seq_start device [num_seqs]; cu_rows device [num_seqs+1];
 *   latent_ws device [total_rows, L+P] in dtype.  (L+P)*elem must be a
 *   multiple of 16 bytes and kv_cache, latent_ws 16-byte aligned (rows move
 *   as 16-byte pieces), else MLA_ERR_UNSUPPORTED / MLA_ERR_INVALID.
 */
int mla_gather_context_rows(const mla_dims_t *d, const void *kv_cache,
                            int32_t num_blocks, const int32_t *block_table,
                            int32_t block_table_stride, int32_t num_seqs,
                            const int32_t *seq_request,
                            const int32_t *seq_start, const int32_t *cu_rows,
                            int32_t total_rows, void *latent_ws,
                            int32_t *dev_status, mla_stream_t stream);

/* mla_kv_up_proj: kv[h, row, c] = latent[row, 0:L] . w_kv_b[h*(Dn+Dv) + c, :]
 *   latent device [rows, latent_ld] in dtype (latent_ld >= L); w_kv_b in
 *   dtype; kv device, HEAD-MAJOR [H, rows, Dn+Dv] in kv_dtype (F32, BF16 or
 *   F16; accumulation is float32, the result is rounded once to kv_dtype):
 *   columns [0, Dn) of head h are K_nope, [Dn, Dn+Dv) are V.  Head-major
 *   keeps every output tile of the GEMM and every key tile of the attention
 *   one contiguous block of HBM.  The tensor-core shape (see the
 *   conventions) runs on the 2-SM tcgen05 GEMM, which writes F16 or BF16
 *   (F32 output: MLA_ERR_UNSUPPORTED; latent_ld*2 a multiple of 16 bytes).
 *   The chunked path stores K/V as F16 there: bf16 keeps 8 significant bits
 *   and its rounding of K_nope alone moves a one-key LSE by ~5e-4 (1 sigma),
 *   fp16 keeps 11.  An F16 result of magnitude >= 65520 sets
 *   MLA_STATUS_FP16_RANGE in dev_status (nullable). */
int mla_kv_up_proj(const mla_dims_t *d, const void *latent, int64_t latent_ld,
                   int32_t rows, const void *w_kv_b, void *kv, int32_t kv_dtype,
                   int32_t *dev_status, mla_stream_t stream);

/* mla_varlen_attn: softmax attention per sequence, returning (O, LSE).
 *   Sequence i owns query tokens [q_loc[i], q_loc[i+1]) (rows of q, o, lse)
 *   and key rows [k_loc[i], k_loc[i+1]) of kv (the head-major up-projection
 *   output [H, kv_rows, Dn+Dv] of mla_kv_up_proj, kv_rows >= k_loc[num_seqs])
 *   and of latent (k_pe = latent[row][L:L+P]).
 *   causal = 0: every query sees all of its sequence's keys (context chunk).
 *   causal = 1: keys are the sequence's own new tokens and query i sees keys
 *               0..i (requires equal query and key counts).
 *   accumulate (device [num_seqs], nullable): where nonzero, the result is
 *   LSE-merged into the (o, lse) already stored for those tokens instead of
 *   overwriting them (PR #50613 report, item 3, accumulate_mla_context_chunk).
 *   q_loc, k_loc device [num_seqs+1]; max_q / max_k: upper bounds of the
 *   per-sequence counts.  o device float32 [T, H, Dv]; lse float32 [H, T];
 *   num_tokens = T (the row count of q, o and lse).  kv is in kv_dtype
 *   (F32, BF16 or F16); q and latent in d->dtype.  The tensor-core shape
 *   (see the conventions) runs on the tcgen05 kernels, which take F16 kv
 *   only (other K/V types: MLA_ERR_UNSUPPORTED); they convert q_nope to
 *   fp16 on chip (exact for bf16 values of magnitude 2^-14 .. 65504; beyond
 *   65504 sets MLA_STATUS_FP16_RANGE in dev_status, nullable).
 *   A row that sees no key gets O = 0, LSE = -inf. */
int mla_varlen_attn(const mla_dims_t *d, int32_t causal, int32_t num_seqs,
                    const int32_t *q_loc, const int32_t *k_loc,
                    const int32_t *q_loc_host, const int32_t *k_loc_host,
                    int32_t num_tokens, const void *q, const void *kv,
                    int32_t kv_dtype, int32_t kv_rows, const void *latent,
                    int64_t latent_ld,
                    const int32_t *accumulate, float *o, float *lse,
                    int32_t *dev_status, mla_stream_t stream);

/* mla_fused_context_attn: the context attention of mla_varlen_attn
 *   (causal = 0, PR #50613 report, items 3-4) with the W_kv_b up-projection
 *   fused in (the report's Triton/CUDA kernels are prior art; this is the
 *   same arithmetic as mla_kv_up_proj followed by mla_varlen_attn, K_nope and
 *   V rounded to F16 as that path stores them): the keys and values of each
 *   128-key tile are computed on chip from latent[row][0:L] and w_kv_b and
 *   never written to memory.
 *   Sequence i owns query tokens [q_loc[i], q_loc[i+1]) and latent rows
 *   [k_loc[i], k_loc[i+1]) of latent (device [latent_rows, latent_ld],
 *   bf16; k_pe = latent[row][L:L+P]); w_kv_b device [H*(Dn+Dv), L] bf16; q
 *   device [T, H, Dn+P] bf16 (T = num_tokens); o float32 [T, H, Dv]; lse
 *   float32 [H, T]; accumulate as in mla_varlen_attn.  Every sequence with
 *   both queries and keys may have at most 128 queries (one query tile: more
 *   would repeat the up-projection per tile); rows of sequences without keys
 *   are left untouched.
 *   workspace: device, 16-byte aligned, mla_fused_attn_workspace_bytes()
 *   bytes (the queries head-major with q_nope in F16, and key-split scratch);
 *   owned by the caller, reusable once the stream has passed the call.
 *   Runs for the DeepSeek-V3 head shape (L 512, P 64, Dn 128, Dv 128) on a
 *   tcgen05 GPU with q, latent, w_kv_b and workspace 16-byte aligned;
 *   MLA_ERR_UNSUPPORTED otherwise or when a sequence has more than 128
 *   queries.  dev_status (nullable) as in mla_varlen_attn / mla_kv_up_proj.
 *   Needs no K/V workspace; on GB300 it is slower than the two-step path
 *   (mla_chunked_prefill does not use it). */
int mla_fused_attn_workspace_bytes(const mla_dims_t *d, int32_t num_tokens,
                                   size_t *bytes);
int mla_fused_context_attn(const mla_dims_t *d, int32_t num_seqs,
                           const int32_t *q_loc, const int32_t *k_loc,
                           const int32_t *q_loc_host, const int32_t *k_loc_host,
                           int32_t num_tokens, const void *q, const void *latent,
                           int64_t latent_ld, int32_t latent_rows,
                           const void *w_kv_b, const int32_t *accumulate,
                           float *o, float *lse, void *workspace,
                           size_t workspace_bytes, int32_t *dev_status,
                           mla_stream_t stream);

/* mla_fused_attn_plan (host only, no GPU needed): how mla_fused_context_attn
 *   splits its work over `clusters` 2-SM clusters.  items[4*i .. 4*i+3] =
 *   (sequence, key tiles of 128, first tile in a head's order, slot info =
 *   (first scratch slot + 1) | slots << 16, or 0 when the item is never cut),
 *   one per sequence with queries and keys; cluster c takes the flattened
 *   (head, item, key tile) positions [bounds[c], bounds[c+1]), head-major.
 *   A (head, item) unit cut between clusters writes each piece to a key-split
 *   scratch slot; when that would take more than split_slots slots or 16 cut
 *   items, the ranges end on unit boundaries instead.  num_clusters (at most
 *   min(clusters, 128)), num_items and num_groups (cut items) are returned;
 *   pass bounds = items = NULL for those counts alone, else capacities of at
 *   least num_clusters + 1 and num_items (MLA_ERR_TOO_SMALL otherwise).
 *   MLA_ERR_UNSUPPORTED when a sequence has more than 128 queries. */
int mla_fused_attn_plan(int32_t num_heads, int32_t num_seqs,
                        const int32_t *q_loc_host, const int32_t *k_loc_host,
                        int32_t clusters, int32_t split_slots, int32_t *bounds,
                        int32_t bounds_cap, int32_t *items, int32_t items_cap,
                        int32_t *num_clusters, int32_t *num_items,
                        int32_t *num_groups);

/* mla_fill_empty_rows  (PR #50613 report, item 3, init_mla_context_partial):
 *   o[t, :, :] = 0 and lse[:, t] = -inf for t in each [slices[2k],
 *   slices[2k+1]).  slices device int32 [2*num_slices]; o float32 [T, H, Dv];
 *   lse float32 [H, T]. */
int mla_fill_empty_rows(float *o, float *lse, int32_t num_tokens,
                        int32_t num_heads, int32_t v_dim, int32_t num_slices,
                        const int32_t *slices, mla_stream_t stream);

/* mla_mask_empty_context  (PR #49294 report, mask_empty_context): the old
 *   scheme's fix-up.  For every request r whose context length in the chunk,
 *   context_start_loc[r+1] - context_start_loc[r], is 0, rows
 *   [query_start_loc[r], query_start_loc[r+1]) get lse = -inf and o = 0 (o in
 *   dtype, [T, H, D]); all other rows are left untouched.  Both loc arrays
 *   device int32 [num_requests+1]. */
int mla_mask_empty_context(float *lse, void *o, int32_t dtype,
                           int32_t num_tokens, int32_t num_heads,
                           int32_t head_dim, int32_t num_requests,
                           const int32_t *query_start_loc,
                           const int32_t *context_start_loc,
                           mla_stream_t stream);

/* mla_chunk_kv_dtype: the K/V workspace element type (MLA_DTYPE_*) that
 *   mla_context_chunk_attn and mla_chunked_prefill use on the current device
 *   for these dims: F16 where the tcgen05 kernels run, F32 otherwise.  For
 *   callers that compose the per-step calls themselves. */
int mla_chunk_kv_dtype(const mla_dims_t *d, int32_t *kv_dtype);

/* ---------------------------------------------------------------------------
 * Chunk-level and whole-prefill calls.
 *
 * mla_chunk_workspace_bytes: device bytes mla_context_chunk_attn needs for a
 *   chunk of up to max_rows context rows and max_entries requests.
 */
int mla_chunk_workspace_bytes(const mla_dims_t *d, int32_t max_rows,
                              int32_t max_entries, size_t *bytes);

/* mla_context_chunk_attn  (PR #50613 report, items 2-4: one ContextChunk)
 *   Gathers the chunk's rows, up-projects them, attends each of its
 *   requests' new tokens to its rows, and accumulates into the context
 *   partial: requests whose entry starts at 0 overwrite their rows, the
 *   continued request (start > 0) is LSE-merged into what earlier chunks
 *   stored.
 *   chunk, starts, seq_lens: the planner's host outputs (starts/seq_lens
 *     indexed from chunk->entry_offset); query_start_loc host [R+1].  The
 *     library builds the chunk's device descriptor (request ids, starts,
 *     workspace row offsets, query offsets) from them; whether a request
 *     accumulates follows from its start, as on the page: start > 0 (the
 *     request continues from an earlier chunk) merges, start 0 writes.
 *   o_partial device float32 [T, H, Dv]; lse_partial device float32 [H, T].
 *   workspace: device, 16-byte aligned, at least mla_chunk_workspace_bytes
 *   bytes.  The metadata is uploaded from pageable host memory with
 *   cudaMemcpyAsync, so the call is not for stream capture. */
int mla_context_chunk_attn(const mla_dims_t *d, const mla_chunk_t *chunk,
                           const int32_t *starts, const int32_t *seq_lens,
                           const int32_t *query_start_loc, int32_t num_tokens,
                           const void *q, const void *kv_cache,
                           int32_t num_blocks, const int32_t *block_table,
                           int32_t block_table_stride, const void *w_kv_b,
                           void *workspace, size_t workspace_bytes,
                           float *o_partial, float *lse_partial,
                           int32_t *dev_status, mla_stream_t stream);

/* mla_context_chunk_attn_noalloc: mla_context_chunk_attn without a caller
 *   workspace.  (Not a step of the method; it serves callers that cannot
 *   allocate device memory themselves, e.g. a plugin whose host framework
 *   owns every device allocation and hands it no workspace, or a path where a
 *   cudaMalloc, which can synchronise the device, is not allowed.)
 *   The scratch is a library-owned device array of MLA_NOALLOC_SCRATCH_BYTES
 *   (64 MiB) that every GPU which loads the library holds until the process
 *   exits.  The call allocates nothing.  A chunk whose workspace
 *   (mla_chunk_workspace_bytes for its rows and requests) exceeds that size
 *   is rejected with MLA_ERR_TOO_SMALL before anything is enqueued.
 *   The first call on a device, with that device current, looks up the
 *   array's device address (cudaGetSymbolAddress) and keeps it for the
 *   process; after a cudaDeviceReset of that device the kept address is
 *   stale, so do not call this entry point again on a device the process
 *   has reset.  Like mla_context_chunk_attn it uploads its metadata from
 *   pageable host memory, so it is not for stream capture.  All calls share
 *   the one array and it keeps the last call's contents; nothing in it needs
 *   to start at zero (each call writes all it reads), but calls that overlap
 *   on the GPU race on it and must be serialised by the caller.  Other
 *   arguments and results as for mla_context_chunk_attn. */
#define MLA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int mla_context_chunk_attn_noalloc(const mla_dims_t *d, const mla_chunk_t *chunk,
                                   const int32_t *starts, const int32_t *seq_lens,
                                   const int32_t *query_start_loc,
                                   int32_t num_tokens, const void *q,
                                   const void *kv_cache, int32_t num_blocks,
                                   const int32_t *block_table,
                                   int32_t block_table_stride,
                                   const void *w_kv_b, float *o_partial,
                                   float *lse_partial, int32_t *dev_status,
                                   mla_stream_t stream);

/* mla_prefill_workspace_bytes: device bytes mla_chunked_prefill needs for
 *   these lengths and planner settings (it runs the planner).
 * mla_prefill_pinned_bytes: host bytes of the metadata that
 *   mla_chunked_prefill uploads for them (the size of its optional pinned
 *   scratch). */
int mla_prefill_workspace_bytes(const mla_dims_t *d,
                                const int32_t *context_lens,
                                const int32_t *query_lens,
                                int32_t num_requests, int32_t row_budget,
                                int32_t max_context_chunk,
                                int32_t split_alignment, size_t *bytes);
int mla_prefill_pinned_bytes(const mla_dims_t *d, const int32_t *context_lens,
                             const int32_t *query_lens, int32_t num_requests,
                             int32_t row_budget, int32_t max_context_chunk,
                             int32_t split_alignment, size_t *bytes);

/* mla_chunked_prefill  (the whole path: plan, init partial, per chunk
 *   gather + up-projection + attention + accumulate, new-token up-projection
 *   and causal attention, final merge_attn_states with prefix_num_tokens)
 *   context_lens, query_lens: host [num_requests].
 *   prefix_num_tokens = end of the last request with context (tokens of a
 *   context-free tail copy the suffix result).
 *   out device [T, H, Dv] in dtype; out_lse device float32 [H, T], nullable.
 *   workspace: device, 16-byte aligned, >= mla_prefill_workspace_bytes.
 *   Metadata (the plan's chunk descriptors, the empty-token slices and the
 *   query offsets; the host lengths avoid any device-to-host read, PR #36540
 *   report, comments) goes to the device in one cudaMemcpyAsync.
 *   pinned_scratch (nullable): caller-owned page-locked host memory of at
 *   least mla_prefill_pinned_bytes bytes (else MLA_ERR_TOO_SMALL); the
 *   library writes the metadata there and copies it from there, so the copy
 *   is a true asynchronous DMA.  Before rewriting pinned scratch a call waits
 *   on the host until the previous call's copy out of pinned scratch on this
 *   device has run, so one buffer can serve call after call; the library
 *   never frees it.  NULL: the copy is made from pageable memory.
 *   On the tensor-core path the workspace keeps K/V in fp16 (see
 *   mla_kv_up_proj); on the CUDA-core path in float32.  There, when the
 *   last execution group's units with the new tokens' causal tiles suit
 *   the looping or the persistent attention kernel (on average at most 16
 *   key tiles of 128 per (request, query tile, head) and more units than
 *   SMs, or at most 64 and at least two units per SM), its context
 *   attention and the new-token attention run as one launch: each (request, query tile, head) walks the request's
 *   context rows of that group and then its own new tokens, and merges with
 *   the context partial only where an earlier group left one.  The result
 *   is the same composition, one LSE merge order apart.
 *   Streams: the chunks run as a two-buffer pipeline.  Gathers and
 *   up-projections go to two library-owned side streams of the highest
 *   priority (one pair per device, made on first use); attention, merges
 *   and every write of out/out_lse stay on `stream`.  All of it is ordered
 *   after the work already on `stream` (an event recorded there), and
 *   `stream` waits for all of it before the call's last kernel, so to the
 *   caller the call behaves like work enqueued on `stream` alone.  (Not for
 *   stream capture.)  Calls on one device from several host threads are
 *   serialised while they enqueue (a lock per device); calls on different
 *   devices are independent.  The workspace holds two chunk buffer sets and
 *   the key-split scratch of the context attention.
 */
int mla_chunked_prefill(const mla_dims_t *d, const int32_t *context_lens,
                        const int32_t *query_lens, int32_t num_requests,
                        int32_t row_budget, int32_t max_context_chunk,
                        int32_t split_alignment, const void *q,
                        const void *new_latent, const void *kv_cache,
                        int32_t num_blocks, const int32_t *block_table,
                        int32_t block_table_stride, const void *w_kv_b,
                        void *workspace, size_t workspace_bytes, void *out,
                        float *out_lse, void *pinned_scratch, size_t pinned_bytes,
                        int32_t *dev_status, mla_stream_t stream);

/* ---------------------------------------------------------------------------
 * The old scheme, kept as a comparator (PR #50613 report, motivation: the
 * workspace was divided evenly among the requests with context and every
 * iteration processed the same context window of every request; PR #49294
 * report: per chunk, rows of requests whose window is empty are fixed up with
 * mask_empty_context before the merge).
 *
 * mla_plan_equal_window_chunks (host only): window = row_budget / (requests
 *   with context), rounded down to split_alignment; chunk c covers rows
 *   [c*window, (c+1)*window) of every request, clipped to its length;
 *   *num_chunks = ceil(max context / window).  MLA_ERR_PLANNER_STUCK when the
 *   window rounds to 0.
 * mla_chunked_prefill_equal_window: the whole prefill under that plan: per
 *   chunk gather + up-projection + attention over every request, the
 *   empty-window fix-up, and a merge over the whole batch into the running
 *   partial; then the new-token attention and the final merge.  Same
 *   arguments, layouts and result as mla_chunked_prefill (no
 *   max_context_chunk); workspace from
 *   mla_prefill_equal_window_workspace_bytes. */
int mla_plan_equal_window_chunks(const int32_t *context_lens,
                                 int32_t num_requests, int32_t row_budget,
                                 int32_t split_alignment, int32_t *window,
                                 int32_t *num_chunks);
int mla_prefill_equal_window_workspace_bytes(
    const mla_dims_t *d, const int32_t *context_lens, const int32_t *query_lens,
    int32_t num_requests, int32_t row_budget, int32_t split_alignment,
    size_t *bytes);
int mla_chunked_prefill_equal_window(
    const mla_dims_t *d, const int32_t *context_lens, const int32_t *query_lens,
    int32_t num_requests, int32_t row_budget, int32_t split_alignment,
    const void *q, const void *new_latent, const void *kv_cache,
    int32_t num_blocks, const int32_t *block_table, int32_t block_table_stride,
    const void *w_kv_b, void *workspace, size_t workspace_bytes, void *out,
    float *out_lse, int32_t *dev_status, mla_stream_t stream);

/* 1 when the current device runs the tcgen05 (sm_103a) kernels of this
 * library. */
int mla_has_tcgen05(void);

/* Number of kernels this library has enqueued since it was loaded, over all
 * threads and devices (each launcher counts its launch as it enqueues it).
 * Host-only, no synchronisation: a caller brackets a region with two reads
 * to count the kernels that region launched.  Errors: MLA_ERR_INVALID for a
 * NULL count. */
int mla_kernel_launches(uint64_t *count);

/* Per-launch timing, for looking inside a call's pipeline in place.
 * mla_profile_begin: from now on this host thread records a CUDA event on
 *   the launching stream right before and right after every kernel the
 *   library enqueues (for the calls this thread makes).
 * mla_profile_end: stops, waits for those events, and returns one record per
 *   launch in launch order: the kernel's name, the step of the method it
 *   serves inside mla_chunked_prefill ("a4 gather", "a5 up-projection",
 *   "a6-a7 context attention", ...; empty for the other calls), the stream
 *   it ran on (numbered from 0 in order of first appearance), its start
 *   relative to the first record's start and its duration, both in ms
 *   (kernels that run side by side on different streams each show their
 *   own span).
 *   *count = number of launches; MLA_ERR_TOO_SMALL when it exceeds cap (the
 *   first cap records are filled).  The events are freed either way.
 *   Profiling adds two event records per launch: time a call with it off. */
typedef struct {
  char kernel[40];
  char role[40];
  int32_t stream;
  float start_ms;
  float ms;
} mla_launch_record_t;
int mla_profile_begin(void);
int mla_profile_end(mla_launch_record_t *records, int32_t cap, int32_t *count);

/* Overlap of the chunk pipeline (mla_chunked_prefill and
 * mla_chunked_prefill_equal_window): on (1, the default), the gathers and
 * up-projections run on two library-owned side streams, one chunk ahead of
 * the attention on the caller's stream; off (0), every kernel of the call
 * runs on the caller's stream, one after another in the same order, with
 * identical results.  Off lets each kernel be timed alone inside a real
 * prefill (per-launch profile above).  Process-wide, read when a call is
 * enqueued; returns the previous setting.  No errors. */
int32_t mla_set_pipeline_overlap(int32_t on);

/* Failure-detection self test: launches one thread that waits on an
 * mbarrier nothing arrives on, with the same bounded wait the tensor-core
 * kernels use but a limit of limit_us microseconds (1 .. 10^6).  The wait
 * gives up, sets MLA_DEVICE_ERR_WAIT_TIMEOUT (read with
 * mla_device_error_flags) and writes 1 to gave_up (device int32); the kernel
 * returns normally and the context stays usable.  MLA_ERR_UNSUPPORTED off
 * sm_103a. */
int mla_selftest_bounded_wait(int32_t limit_us, int32_t *gave_up,
                              mla_stream_t stream);

/* Reads and clears the device-side error bits of the tensor-core kernels
 * (MLA_DEVICE_ERR_*; nonzero means a kernel gave up waiting on one of its
 * own barriers and its output is not valid).  Synchronises the device. */
int mla_device_error_flags(int32_t *flags);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif

#endif /* MLA_CHUNKED_CONTEXT_H */
