// C-ABI entry points: argument checks, workspace carving, metadata upload and
// the order of the steps (PR #50613 report, items 2-4; PR #36540 report).
//
// Step order of mla_chunked_prefill:
//   plan (host), chunks grouped for execution -> one metadata upload -> fill
//   of context-free rows of the partial, query preparation -> per execution
//   group { gather, up-projection (side streams), attention + accumulate } as
//   a two-buffer pipeline -> new-token up-projection -> causal new-token
//   attention with the final merge (tensor-core path; else attention, merge).
//   Everything that writes the partial or the output runs on the caller's
//   stream, which waits for the side streams before the last kernel.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "planner.h"

namespace mla {

// kernels (merge.cu, gather.cu, generic.cu, sm103_gemm.cu, sm103_attn.cu)
int launch_merge(void *out, float *out_lse, const void *prefix_o, const float *prefix_lse,
                 const void *suffix_o, const float *suffix_lse, int T, int H, int D,
                 int pnt, int in_dtype, int out_dtype, cudaStream_t s);
int launch_fill_empty_rows(float *o, float *lse, int T, int H, int Dv, int num_slices,
                           const int32_t *slices, cudaStream_t s);
int launch_mask_empty_context(float *lse, void *o, int dtype, int T, int H, int D, int R,
                              const int32_t *qsl, const int32_t *csl, cudaStream_t s);
int launch_gather(const void *cache, int num_blocks, int block_size, int row_bytes,
                  const int32_t *block_table, int bt_stride, int num_seqs,
                  const int32_t *seq_request, const int32_t *seq_start,
                  const int32_t *cu_rows, int total_rows, void *ws, int32_t *status,
                  cudaStream_t s);
bool generic_dims_ok(const mla_dims_t &d);
int launch_up_proj_simt(int dtype, int kv_dtype, const void *latent, int64_t lda, int rows,
                        const void *w, void *kv, int N, int K, int hd, int32_t *status,
                        cudaStream_t s);
int launch_attn_simt(const mla_dims_t &d, int causal, int num_seqs, const int32_t *q_loc,
                     const int32_t *k_loc, int num_q_rows, int T, int kv_rows, const void *q,
                     const void *kv, int kv_dtype, const void *latent, int64_t latent_ld,
                     const int32_t *accumulate, float *o, float *lse, cudaStream_t s);
bool tc_gemm_ok(const mla_dims_t &d, int kv_dtype, int64_t lda, const void *latent,
                const void *w, const void *kv);
int launch_up_proj_tc(const mla_dims_t &d, int kv_dtype, const void *latent, int64_t lda,
                      int rows, const void *w, void *kv, int32_t *status, cudaStream_t s);
bool tc_attn_ok(const mla_dims_t &d, int kv_dtype, int64_t latent_ld);
int gemm_take_errors();
int attn_take_errors();
int launch_bounded_wait_selftest(long long limit_cycles, int32_t *gave_up, cudaStream_t s);
int launch_attn_tc(const mla_dims_t &d, int causal, int num_seqs, const int32_t *q_loc,
                   const int32_t *k_loc, const int32_t *q_loc_host,
                   const int32_t *k_loc_host, int T, int kv_rows, const void *q, const void *kv,
                   const void *latent, int64_t latent_ld, const int32_t *accumulate,
                   float *o, float *lse, void *final_out, float *final_lse, int final_dtype,
                   int pnt, const SplitScratch *split, bool skip_keyless, bool q_prepared,
                   int32_t *status, cudaStream_t s, const NewKeySource *new_keys = nullptr);
bool attn_tc_new_keys_ok(int num_seqs, const int32_t *q_loc_host, const int32_t *k_loc_host,
                         int H);
int launch_prepare_q(const void *q, void *qh, int T, int H, int32_t *status, cudaStream_t s);
bool fused_attn_ok(const mla_dims_t &d, int64_t latent_ld);
bool fused_attn_fits(int num_seqs, const int32_t *q_loc_host, const int32_t *k_loc_host,
                     int min_tiles);
int launch_attn_fused(const mla_dims_t &d, int num_seqs, const int32_t *q_loc,
                      const int32_t *k_loc, const int32_t *q_loc_host, const int32_t *k_loc_host,
                      int T, const void *q_prep, const void *latent, int64_t latent_ld, int rows,
                      const void *w, const int32_t *acc, float *o, float *lse,
                      const SplitScratch *split, int32_t *status, cudaStream_t s);
int fused_take_errors();
int gather_take_errors();
bool tc_available();

namespace {

constexpr size_t kAlign = 256;

struct Carve {
  char *base;
  size_t off = 0;
  explicit Carve(void *b) : base(static_cast<char *>(b)) {}
  void *take(size_t bytes) {
    off = (off + kAlign - 1) / kAlign * kAlign;
    void *p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
};

int check_dims(const mla_dims_t *d) {
  if (!d) return MLA_ERR_INVALID;
  if (d->num_heads < 1 || d->kv_lora_rank < 1 || d->qk_rope_dim < 0 || d->qk_nope_dim < 1 ||
      d->v_dim < 1 || d->block_size < 1 || !valid_dtype(d->dtype))
    return MLA_ERR_INVALID;
  if (!(d->softmax_scale > 0.f)) return MLA_ERR_INVALID;
  const int es = elem_bytes(d->dtype);
  if (((d->kv_lora_rank + d->qk_rope_dim) * es) % 16 != 0) return MLA_ERR_UNSUPPORTED;
  if (d->v_dim % 8 != 0) return MLA_ERR_UNSUPPORTED;
  if (!generic_dims_ok(*d)) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

inline int kv_width(const mla_dims_t &d) { return d.num_heads * (d.qk_nope_dim + d.v_dim); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

// The tensor-core kernels serve bf16 storage with the DeepSeek-V3 head shape
// (latent 512, rope 64, nope 128, v 128); the CUDA-core kernels serve float32
// storage and every other head shape.  A call of the tensor-core shape runs
// on the tensor-core kernels or fails with MLA_ERR_UNSUPPORTED (no tcgen05
// GPU, an operand not 16-byte aligned, a K/V type they do not take): it is
// never handed to the CUDA-core kernels, which are 10-100x slower.
bool tc_shape(const mla_dims_t &d) {
  return d.dtype == MLA_DTYPE_BF16 && d.kv_lora_rank == 512 && d.qk_rope_dim == 64 &&
         d.qk_nope_dim == 128 && d.v_dim == 128;
}

// K/V workspace type of the chunked path: fp16 for the tensor-core kernels,
// float32 for the CUDA-core kernels.
int path_kv_dtype(const mla_dims_t &d) {
  return tc_shape(d) ? MLA_DTYPE_F16 : MLA_DTYPE_F32;
}

int up_proj(const mla_dims_t &d, const void *latent, int64_t lda, int rows, const void *w,
            void *kv, int kv_dtype, int32_t *status, cudaStream_t s) {
  if (rows == 0) return MLA_OK;
  if (tc_shape(d)) {
    if (!tc_gemm_ok(d, kv_dtype, lda, latent, w, kv) || !tc_available())
      return MLA_ERR_UNSUPPORTED;
    return launch_up_proj_tc(d, kv_dtype, latent, lda, rows, w, kv, status, s);
  }
  return launch_up_proj_simt(d.dtype, kv_dtype, latent, lda, rows, w, kv, kv_width(d),
                             d.kv_lora_rank, d.qk_nope_dim + d.v_dim, status, s);
}

int attention(const mla_dims_t &d, int causal, int n, const int32_t *q_loc,
              const int32_t *k_loc, const int32_t *q_loc_host, const int32_t *k_loc_host,
              int T, const void *q, const void *kv, int kv_dtype, int kv_rows,
              const void *latent, int64_t latent_ld, const int32_t *acc, float *o, float *lse,
              int32_t *status, cudaStream_t s, const SplitScratch *split = nullptr,
              bool skip_keyless = false, const void *q_prep = nullptr) {
  const int nq = q_loc_host[n] - q_loc_host[0];
  if (n == 0 || nq == 0) return MLA_OK;
  // q_prep: the same queries head-major with q_nope in fp16 (prepare_q), for
  // the tensor-core kernel
  if (tc_shape(d)) {
    if (!tc_attn_ok(d, kv_dtype, latent_ld) || !aligned16(q) || !aligned16(kv) ||
        !aligned16(latent) || (q_prep && !aligned16(q_prep)) || !tc_available())
      return MLA_ERR_UNSUPPORTED;
    return launch_attn_tc(d, causal, n, q_loc, k_loc, q_loc_host, k_loc_host, T, kv_rows,
                          q_prep ? q_prep : q, kv, latent, latent_ld, acc, o, lse, nullptr,
                          nullptr, 0, 0, split, skip_keyless, q_prep != nullptr, status, s);
  }
  return launch_attn_simt(d, causal, n, q_loc, k_loc, nq, T, kv_rows, q, kv, kv_dtype, latent,
                          latent_ld, acc, o, lse, s);
}

// Device metadata of one chunk, in this order (n = number of requests):
//   seq_request[n] seq_start[n] cu_rows[n+1] q_loc[n+1] accumulate[n]
struct ChunkMetaHost {
  int n = 0, rows = 0;
  std::vector<int32_t> ints;
  std::vector<int32_t> q_loc, cu_rows;  // host copies for launch sizing
};

size_t chunk_meta_ints(int n) { return size_t(5) * n + 2; }

void build_chunk_meta(const mla_chunk_t &c, const int32_t *starts, const int32_t *lens,
                      const int32_t *qsl, ChunkMetaHost &m) {
  const int n = c.request_end - c.request_start;
  m.n = n;
  m.ints.assign(chunk_meta_ints(n), 0);
  m.q_loc.assign(n + 1, 0);
  m.cu_rows.assign(n + 1, 0);
  int32_t *req = m.ints.data(), *st = req + n, *cu = st + n, *ql = cu + n + 1,
          *acc = ql + n + 1;
  for (int i = 0; i < n; ++i) {
    const int e = c.entry_offset + i;
    req[i] = c.request_start + i;
    st[i] = starts[e];
    cu[i + 1] = cu[i] + lens[e];
    acc[i] = starts[e] > 0 ? 1 : 0;
  }
  for (int i = 0; i <= n; ++i) ql[i] = qsl[c.request_start + i];
  m.rows = cu[n];
  std::memcpy(m.q_loc.data(), ql, sizeof(int32_t) * (n + 1));
  std::memcpy(m.cu_rows.data(), cu, sizeof(int32_t) * (n + 1));
}

// Execution group: consecutive chunks [c0, c1) whose requests are all new
// (no chunk after the first continues a request) and whose rows fit the
// budget together.  The zero-context requests between them become sequences
// without rows, so the group's sequences are the contiguous request range
// and q_loc stays a prefix sum of query counts; the attention skips them
// (their partial rows are initialised to O=0, LSE=-inf).
void build_group_meta(const std::vector<mla_chunk_t> &chunks, size_t c0, size_t c1,
                      const int32_t *starts, const int32_t *lens, const int32_t *qsl,
                      ChunkMetaHost &m) {
  const int r0 = chunks[c0].request_start, r1 = chunks[c1 - 1].request_end;
  const int n = r1 - r0;
  m.n = n;
  m.ints.assign(chunk_meta_ints(n), 0);
  m.q_loc.assign(n + 1, 0);
  m.cu_rows.assign(n + 1, 0);
  int32_t *req = m.ints.data(), *st = req + n, *cu = st + n, *ql = cu + n + 1,
          *acc = ql + n + 1;
  std::vector<int32_t> rows(n, 0);
  for (size_t c = c0; c < c1; ++c)
    for (int i = 0; i < chunks[c].request_end - chunks[c].request_start; ++i) {
      const int e = chunks[c].entry_offset + i, k = chunks[c].request_start + i - r0;
      st[k] = starts[e];
      rows[k] = lens[e];
      acc[k] = starts[e] > 0 ? 1 : 0;
    }
  for (int k = 0; k < n; ++k) {
    req[k] = r0 + k;
    cu[k + 1] = cu[k] + rows[k];
  }
  for (int k = 0; k <= n; ++k) ql[k] = qsl[r0 + k];
  m.rows = cu[n];
  std::memcpy(m.q_loc.data(), ql, sizeof(int32_t) * (n + 1));
  std::memcpy(m.cu_rows.data(), cu, sizeof(int32_t) * (n + 1));
}

struct ChunkBuffers {
  void *latent_ws;
  void *kv_ws;
  int kv_dtype;
};

int run_chunk(const mla_dims_t &d, const ChunkMetaHost &m, const int32_t *meta_dev, int T,
              const void *q, const void *kv_cache, int num_blocks, const int32_t *block_table,
              int bt_stride, const void *w, const ChunkBuffers &b, float *o, float *lse,
              int32_t *status, cudaStream_t s) {
  const int n = m.n;
  const int32_t *req = meta_dev, *st = req + n, *cu = st + n, *ql = cu + n + 1,
                *acc = ql + n + 1;
  const int LP = d.kv_lora_rank + d.qk_rope_dim;
  const int es = elem_bytes(d.dtype);
  int rc = launch_gather(kv_cache, num_blocks, d.block_size, LP * es, block_table, bt_stride,
                         n, req, st, cu, m.rows, b.latent_ws, status, s);
  if (rc) return rc;
  rc = up_proj(d, b.latent_ws, LP, m.rows, w, b.kv_ws, b.kv_dtype, status, s);
  if (rc) return rc;
  return attention(d, 0, n, ql, cu, m.q_loc.data(), m.cu_rows.data(), T, q, b.kv_ws, b.kv_dtype,
                   m.rows, b.latent_ws, LP, acc, o, lse, status, s);
}

void carve_chunk_buffers(Carve &cv, const mla_dims_t &d, int64_t rows, ChunkBuffers &b) {
  const int es = elem_bytes(d.dtype);
  const int LP = d.kv_lora_rank + d.qk_rope_dim;
  b.kv_dtype = path_kv_dtype(d);
  b.latent_ws = cv.take(size_t(rows) * LP * es);
  b.kv_ws = cv.take(size_t(rows) * kv_width(d) * elem_bytes(b.kv_dtype));
}

int upload(void *dst, const std::vector<int32_t> &src, cudaStream_t s) {
  if (src.empty()) return MLA_OK;
  return cudaMemcpyAsync(dst, src.data(), src.size() * sizeof(int32_t),
                         cudaMemcpyHostToDevice, s) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int merge_attn_states(void *out, float *out_lse, const void *prefix_o,
                                 const float *prefix_lse, const void *suffix_o,
                                 const float *suffix_lse, int32_t num_tokens,
                                 int32_t num_heads, int32_t head_dim,
                                 int32_t prefix_num_tokens, int32_t in_dtype,
                                 int32_t out_dtype, mla_stream_t stream) {
  if (num_tokens < 0 || num_heads < 1 || head_dim < 8 || head_dim % 8 != 0 ||
      !valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return MLA_ERR_INVALID;
  if (num_tokens == 0) return MLA_OK;
  if (!out || !suffix_o || !suffix_lse) return MLA_ERR_INVALID;
  if (prefix_num_tokens > 0 && (!prefix_o || !prefix_lse)) return MLA_ERR_INVALID;
  // the kernel moves O as 16-byte vectors and LSEs as 4-byte words
  if (!aligned16(out) || !aligned16(suffix_o) || !aligned4(suffix_lse) ||
      (out_lse && !aligned4(out_lse)) ||
      (prefix_num_tokens > 0 && (!aligned16(prefix_o) || !aligned4(prefix_lse))))
    return MLA_ERR_INVALID;
  return launch_merge(out, out_lse, prefix_o, prefix_lse, suffix_o, suffix_lse, num_tokens,
                      num_heads, head_dim, prefix_num_tokens < 0 ? 0 : prefix_num_tokens,
                      in_dtype, out_dtype, static_cast<cudaStream_t>(stream));
}

extern "C" int mla_gather_context_rows(const mla_dims_t *d, const void *kv_cache,
                                       int32_t num_blocks, const int32_t *block_table,
                                       int32_t block_table_stride, int32_t num_seqs,
                                       const int32_t *seq_request, const int32_t *seq_start,
                                       const int32_t *cu_rows, int32_t total_rows,
                                       void *latent_ws, int32_t *dev_status,
                                       mla_stream_t stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (num_seqs < 0 || total_rows < 0 || num_blocks < 0 || block_table_stride < 1)
    return MLA_ERR_INVALID;
  if (total_rows == 0) return MLA_OK;
  if (!kv_cache || !block_table || !seq_request || !seq_start || !cu_rows || !latent_ws ||
      num_seqs == 0)
    return MLA_ERR_INVALID;
  if (!aligned16(kv_cache) || !aligned16(latent_ws)) return MLA_ERR_INVALID;  // 16-byte copies
  return launch_gather(kv_cache, num_blocks, d->block_size,
                       (d->kv_lora_rank + d->qk_rope_dim) * elem_bytes(d->dtype), block_table,
                       block_table_stride, num_seqs, seq_request, seq_start, cu_rows,
                       total_rows, latent_ws, dev_status, static_cast<cudaStream_t>(stream));
}

extern "C" int mla_kv_up_proj(const mla_dims_t *d, const void *latent, int64_t latent_ld,
                              int32_t rows, const void *w_kv_b, void *kv, int32_t kv_dtype,
                              int32_t *dev_status, mla_stream_t stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (rows < 0 || latent_ld < d->kv_lora_rank || !valid_kv_dtype(kv_dtype))
    return MLA_ERR_INVALID;
  if (rows == 0) return MLA_OK;
  if (!latent || !w_kv_b || !kv) return MLA_ERR_INVALID;
  return up_proj(*d, latent, latent_ld, rows, w_kv_b, kv, kv_dtype, dev_status,
                 static_cast<cudaStream_t>(stream));
}

extern "C" int mla_varlen_attn(const mla_dims_t *d, int32_t causal, int32_t num_seqs,
                               const int32_t *q_loc, const int32_t *k_loc,
                               const int32_t *q_loc_host, const int32_t *k_loc_host,
                               int32_t num_tokens, const void *q, const void *kv,
                               int32_t kv_dtype, int32_t kv_rows, const void *latent,
                               int64_t latent_ld, const int32_t *accumulate, float *o,
                               float *lse, int32_t *dev_status, mla_stream_t stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (num_seqs < 0 || num_tokens < 0 || !valid_kv_dtype(kv_dtype)) return MLA_ERR_INVALID;
  if (num_seqs == 0) return MLA_OK;
  if (!q_loc || !k_loc || !q_loc_host || !k_loc_host || !q || !kv || !latent || !o || !lse)
    return MLA_ERR_INVALID;
  if (latent_ld < d->kv_lora_rank + d->qk_rope_dim) return MLA_ERR_INVALID;
  for (int i = 0; i < num_seqs; ++i) {
    const int nq = q_loc_host[i + 1] - q_loc_host[i], nk = k_loc_host[i + 1] - k_loc_host[i];
    if (nq < 0 || nk < 0) return MLA_ERR_INVALID;
    if (causal && nq != nk) return MLA_ERR_INVALID;
  }
  if (q_loc_host[0] < 0 || q_loc_host[num_seqs] > num_tokens) return MLA_ERR_INVALID;
  if (k_loc_host[0] < 0 || kv_rows < k_loc_host[num_seqs]) return MLA_ERR_INVALID;
  return attention(*d, causal ? 1 : 0, num_seqs, q_loc, k_loc, q_loc_host, k_loc_host,
                   num_tokens, q, kv, kv_dtype, kv_rows, latent, latent_ld, accumulate, o, lse,
                   dev_status, static_cast<cudaStream_t>(stream));
}

extern "C" int mla_fill_empty_rows(float *o, float *lse, int32_t num_tokens, int32_t num_heads,
                                   int32_t v_dim, int32_t num_slices, const int32_t *slices,
                                   mla_stream_t stream) {
  if (num_tokens < 0 || num_heads < 1 || v_dim < 1 || num_slices < 0) return MLA_ERR_INVALID;
  if (num_slices == 0) return MLA_OK;
  if (!o || !lse || !slices) return MLA_ERR_INVALID;
  return launch_fill_empty_rows(o, lse, num_tokens, num_heads, v_dim, num_slices, slices,
                                static_cast<cudaStream_t>(stream));
}

extern "C" int mla_mask_empty_context(float *lse, void *o, int32_t dtype, int32_t num_tokens,
                                      int32_t num_heads, int32_t head_dim,
                                      int32_t num_requests, const int32_t *query_start_loc,
                                      const int32_t *context_start_loc, mla_stream_t stream) {
  if (num_tokens < 0 || num_heads < 1 || head_dim < 1 || num_requests < 0 ||
      !valid_dtype(dtype))
    return MLA_ERR_INVALID;
  if (num_tokens == 0 || num_requests == 0) return MLA_OK;
  if (!lse || !o || !query_start_loc || !context_start_loc) return MLA_ERR_INVALID;
  return launch_mask_empty_context(lse, o, dtype, num_tokens, num_heads, head_dim,
                                   num_requests, query_start_loc, context_start_loc,
                                   static_cast<cudaStream_t>(stream));
}

extern "C" int mla_chunk_kv_dtype(const mla_dims_t *d, int32_t *kv_dtype) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!kv_dtype) return MLA_ERR_INVALID;
  *kv_dtype = path_kv_dtype(*d);
  return MLA_OK;
}

extern "C" int mla_chunk_workspace_bytes(const mla_dims_t *d, int32_t max_rows,
                                         int32_t max_entries, size_t *bytes) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (max_rows < 0 || max_entries < 0 || !bytes) return MLA_ERR_INVALID;
  Carve cv(nullptr);
  cv.take(chunk_meta_ints(max_entries) * sizeof(int32_t));
  ChunkBuffers b;
  carve_chunk_buffers(cv, *d, max_rows, b);
  *bytes = cv.off;
  return MLA_OK;
}

extern "C" int mla_context_chunk_attn(const mla_dims_t *d, const mla_chunk_t *chunk,
                                      const int32_t *starts, const int32_t *seq_lens,
                                      const int32_t *query_start_loc, int32_t num_tokens,
                                      const void *q, const void *kv_cache, int32_t num_blocks,
                                      const int32_t *block_table, int32_t block_table_stride,
                                      const void *w_kv_b, void *workspace,
                                      size_t workspace_bytes, float *o_partial,
                                      float *lse_partial, int32_t *dev_status,
                                      mla_stream_t stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!chunk || !starts || !seq_lens || !query_start_loc || !q || !kv_cache || !block_table ||
      !w_kv_b || !workspace || !o_partial || !lse_partial)
    return MLA_ERR_INVALID;
  if (!aligned16(workspace) || !aligned16(kv_cache)) return MLA_ERR_INVALID;
  const int n = chunk->request_end - chunk->request_start;
  if (n < 1 || chunk->request_start < 0 || chunk->entry_offset < 0 || block_table_stride < 1)
    return MLA_ERR_INVALID;
  for (int i = 0; i < n; ++i) {
    const int e = chunk->entry_offset + i;
    if (starts[e] < 0 || seq_lens[e] < 1 ||
        int64_t(starts[e]) + seq_lens[e] > int64_t(block_table_stride) * d->block_size)
      return MLA_ERR_INVALID;
  }
  if (query_start_loc[chunk->request_end] > num_tokens) return MLA_ERR_INVALID;
  ChunkMetaHost m;
  build_chunk_meta(*chunk, starts, seq_lens, query_start_loc, m);
  size_t need = 0;
  mla_chunk_workspace_bytes(d, m.rows, n, &need);
  if (workspace_bytes < need) return MLA_ERR_TOO_SMALL;
  Carve cv(workspace);
  int32_t *meta = static_cast<int32_t *>(cv.take(m.ints.size() * sizeof(int32_t)));
  ChunkBuffers b;
  carve_chunk_buffers(cv, *d, m.rows, b);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = upload(meta, m.ints, s);
  if (rc) return rc;
  return run_chunk(*d, m, meta, num_tokens, q, kv_cache, num_blocks, block_table,
                   block_table_stride, w_kv_b, b, o_partial, lse_partial, dev_status, s);
}

namespace {

// Side streams and events of the chunk pipeline, one set per device, made on
// first use and kept for the life of the process, with the device's lock: a
// prefill enqueues its whole pipeline (and its metadata upload) holding the
// lock of its device, so concurrent callers never interleave their records
// and waits on these streams.  Calls on different devices do not wait for
// one another.
struct Pipeline {
  std::mutex mu;
  cudaStream_t gather = nullptr, gemm = nullptr;
  std::vector<cudaEvent_t> ev;
  // the last metadata copy out of a caller's pinned scratch: the next call
  // waits for it on the host before rewriting pinned memory
  cudaEvent_t upload = nullptr;
  bool upload_pending = false;
};
constexpr int kMaxDevices = 64;
Pipeline g_pipelines[kMaxDevices];

// Locks the current device's pipeline and makes its streams and at least
// `events` events.
int lock_pipeline(size_t events, std::unique_lock<std::mutex> &lock, Pipeline **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  Pipeline &pl = g_pipelines[dev];
  lock = std::unique_lock<std::mutex>(pl.mu);
  if (!pl.gemm) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&pl.gather, cudaStreamNonBlocking, greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&pl.gemm, cudaStreamNonBlocking, greatest) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  if (!pl.upload && cudaEventCreateWithFlags(&pl.upload, cudaEventDisableTiming) != cudaSuccess)
    return MLA_ERR_CUDA;
  while (pl.ev.size() < events) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return MLA_ERR_CUDA;
    pl.ev.push_back(e);
  }
  *out = &pl;
  return MLA_OK;
}

bool record(cudaEvent_t e, cudaStream_t s) { return cudaEventRecord(e, s) == cudaSuccess; }
bool wait_on(cudaStream_t s, cudaEvent_t e) { return cudaStreamWaitEvent(s, e, 0) == cudaSuccess; }

// One metadata upload: from the caller's pinned scratch when given (the
// ints are written there first, after the previous copy out of pinned
// scratch on this device has run), else from the pageable vector.  Called
// with the device's pipeline locked.
int upload_meta(Pipeline &pl, void *dst, const std::vector<int32_t> &src, void *pinned,
                size_t pinned_bytes, cudaStream_t s) {
  if (src.empty()) return MLA_OK;
  const size_t bytes = src.size() * sizeof(int32_t);
  if (!pinned) return upload(dst, src, s);
  if (pinned_bytes < bytes) return MLA_ERR_TOO_SMALL;
  if (pl.upload_pending && cudaEventSynchronize(pl.upload) != cudaSuccess) return MLA_ERR_CUDA;
  pl.upload_pending = false;
  std::memcpy(pinned, src.data(), bytes);
  if (cudaMemcpyAsync(dst, pinned, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      !record(pl.upload, s))
    return MLA_ERR_CUDA;
  pl.upload_pending = true;
  return MLA_OK;
}

// The two-buffer pipeline of the chunked paths, enqueued with the device's
// pipeline `pl` locked.  First pre(s) on the caller's stream `s` (work only
// the consumers need, beside the first gather and up-projection); then for
// units c = 0..n-1: gather(c, stream) on the gather side stream once
// consume(c-2) has released buffer set c % 2, up(c, stream) on the GEMM side
// stream after it, and consume(c, stream) on `s` after that; then
// tail(stream) on the GEMM side stream (the new tokens' up-projection,
// beside the last consume; or, with tail_before = k < n, on that stream
// just before unit k's gather is waited for and its up-projection
// enqueued).  Both side streams start after the work already
// on `s` and are joined back into `s` before returning, also after an error
// (the caller may free the workspace once `s` has passed this point).  The
// side streams run at the highest priority, so a GEMM takes SMs as soon as
// attention CTAs retire.
// With the overlap switched off (mla_set_pipeline_overlap) every step runs
// on `s` in the same order, one kernel after another.
std::atomic<int> g_overlap{1};

template <class Pre, class Gather, class Up, class Consume, class Tail>
int run_pipeline(Pipeline &pl, cudaStream_t s, size_t n, Pre pre, Gather gather, Up up,
                 Consume consume, Tail tail, size_t tail_before = SIZE_MAX) {
  if (pl.ev.size() < 3 * n + 3) return MLA_ERR_INVALID;
  cudaEvent_t *ev = pl.ev.data();
  const bool overlap = g_overlap.load() != 0;
  const cudaStream_t sg = overlap ? pl.gather : s, sm = overlap ? pl.gemm : s;
  auto ev_lat = [&](size_t c) { return ev[1 + 3 * c]; };
  auto ev_kv = [&](size_t c) { return ev[2 + 3 * c]; };
  auto ev_used = [&](size_t c) { return ev[3 + 3 * c]; };
  cudaEvent_t ev_tail = ev[1 + 3 * n], ev_join = ev[2 + 3 * n];
  if (!record(ev[0], s) || !wait_on(sg, ev[0]) || !wait_on(sm, ev[0])) return MLA_ERR_CUDA;
  int rc = pre(s);
  bool tail_done = false;
  for (size_t c = 0; c < n && rc == MLA_OK; ++c) {
    if (c >= 2 && !wait_on(sg, ev_used(c - 2))) rc = MLA_ERR_CUDA;
    if (!rc) rc = gather(c, sg);
    if (!rc && c == tail_before) {
      rc = tail(sm);
      tail_done = true;
    }
    if (!rc && (!record(ev_lat(c), sg) || !wait_on(sm, ev_lat(c)))) rc = MLA_ERR_CUDA;
    if (!rc) rc = up(c, sm);
    if (!rc && (!record(ev_kv(c), sm) || !wait_on(s, ev_kv(c)))) rc = MLA_ERR_CUDA;
    if (!rc) rc = consume(c, s);
    if (!rc && !record(ev_used(c), s)) rc = MLA_ERR_CUDA;
  }
  if (!rc && !tail_done) rc = tail(sm);
  const bool joined = record(ev_tail, sm) && record(ev_join, sg) && wait_on(s, ev_tail) &&
                      wait_on(s, ev_join);
  if (rc) return rc;
  return joined ? MLA_OK : MLA_ERR_CUDA;
}

struct PrefillLayout {
  std::vector<mla_chunk_t> chunks;
  std::vector<int32_t> starts, lens, qsl;
  std::vector<ChunkMetaHost> metas;        // one per execution group
  std::vector<size_t> meta_off;            // int offset of each group's metadata
  std::vector<std::pair<int, int>> empty;  // token slices of context-free requests
  // the last group's context rows per request (prefix sums over all
  // requests: rows of the group's workspace) and, per request, whether its
  // context partial holds an earlier group's result -- for the final
  // launch that attends the last group's context and the new tokens at once
  std::vector<int32_t> last_rows, last_merge;
  size_t slices_off = 0, suffix_off = 0, last_off = 0, meta_total = 0;
  int T = 0, pnt = 0, max_rows = 0;
};

int build_prefill(const mla_dims_t &d, const int32_t *ctx, const int32_t *ql, int R,
                  int budget, int max_chunk, int align, PrefillLayout &p) {
  for (int r = 0; r < R; ++r)
    if (ql[r] < 0 || ctx[r] < 0) return MLA_ERR_INVALID;
  int rc = plan_chunks(ctx, R, budget, max_chunk, align, nullptr, nullptr, p.chunks, p.starts,
                       p.lens);
  if (rc) return rc;
  p.qsl.assign(R + 1, 0);
  for (int r = 0; r < R; ++r) p.qsl[r + 1] = p.qsl[r] + ql[r];
  p.T = p.qsl[R];
  int last = -1;
  for (int r = 0; r < R; ++r)
    if (ctx[r] > 0) last = r;
  p.pnt = last >= 0 ? p.qsl[last + 1] : 0;
  for (int r = 0; r < R; ++r) {
    const int lo = p.qsl[r], hi = std::min(p.qsl[r + 1], p.pnt);
    if (ctx[r] == 0 && lo < hi) p.empty.emplace_back(lo, hi);
  }
  size_t off = 0;
  for (size_t c0 = 0; c0 < p.chunks.size();) {
    // a group ends before a continuation (its first request must see the
    // previous chunk's result) and before the budget would overflow
    size_t c1 = c0 + 1;
    int64_t rows = p.chunks[c0].rows;
    while (c1 < p.chunks.size() && !p.chunks[c1].is_continuation &&
           rows + p.chunks[c1].rows <= budget)
      rows += p.chunks[c1++].rows;
    p.metas.emplace_back();
    build_group_meta(p.chunks, c0, c1, p.starts.data(), p.lens.data(), p.qsl.data(),
                     p.metas.back());
    p.meta_off.push_back(off);
    off += p.metas.back().ints.size();
    p.max_rows = std::max(p.max_rows, p.metas.back().rows);
    c0 = c1;
  }
  p.slices_off = off;
  off += 2 * p.empty.size();
  p.suffix_off = off;
  off += R + 1;
  p.last_rows.assign(R + 1, 0);
  p.last_merge.assign(R, 0);
  if (!p.metas.empty()) {
    // the last group's sequences are requests r0 .. r0+n-1 (build_group_meta)
    const ChunkMetaHost &m = p.metas.back();
    const int32_t *req = m.ints.data(), *acc = req + 4 * m.n + 2;  // req st cu ql acc
    const int r0 = m.n > 0 ? req[0] : R;
    for (int r = 0; r < R; ++r) {
      const int k = r - r0;
      const int rows = (k >= 0 && k < m.n) ? m.cu_rows[k + 1] - m.cu_rows[k] : 0;
      p.last_rows[r + 1] = p.last_rows[r] + rows;
      p.last_merge[r] = (k >= 0 && k < m.n) ? acc[k] : (k < 0 && ctx[r] > 0 ? 1 : 0);
    }
  }
  p.last_off = off;
  off += 2 * size_t(R) + 1;
  p.meta_total = off;
  return MLA_OK;
}

// Key-split scratch slots of the context attention (a few (sequence, query
// tile) units of a chunk, split over their keys when the chunk has too few
// units to fill the GPU).
constexpr int kSplitSlots = 16;

struct PrefillBuffers {
  int32_t *meta;
  ChunkBuffers chunk[2];  // chunk c uses set c % 2
  void *q_prep;           // queries head-major, q_nope in fp16 (tensor-core path)
  void *kv_suffix;
  float *o_part, *lse_part, *o_suf, *lse_suf;
  SplitScratch split;
};

size_t carve_prefill(void *base, const mla_dims_t &d, const PrefillLayout &p,
                     PrefillBuffers &b) {
  Carve cv(base);
  b.meta = static_cast<int32_t *>(cv.take(p.meta_total * sizeof(int32_t)));
  const int sets = p.metas.size() > 1 ? 2 : 1;
  for (int k = 0; k < 2; ++k) {
    if (k < sets)
      carve_chunk_buffers(cv, d, p.max_rows, b.chunk[k]);
    else
      b.chunk[k] = b.chunk[0];
  }
  b.q_prep = cv.take(size_t(p.T) * d.num_heads * (d.qk_nope_dim + d.qk_rope_dim) * 2);
  b.kv_suffix = cv.take(size_t(p.T) * kv_width(d) * elem_bytes(b.chunk[0].kv_dtype));
  const size_t rows_split = size_t(kSplitSlots) * d.num_heads * 128;
  b.split.o = static_cast<float *>(cv.take(rows_split * d.v_dim * sizeof(float)));
  b.split.lse = static_cast<float *>(cv.take(rows_split * sizeof(float)));
  b.split.slots = kSplitSlots;
  b.split.target_ctas = 4 * num_sms();
  const size_t o_bytes = size_t(p.T) * d.num_heads * d.v_dim * sizeof(float);
  const size_t l_bytes = size_t(p.T) * d.num_heads * sizeof(float);
  b.o_part = static_cast<float *>(cv.take(o_bytes));
  b.lse_part = static_cast<float *>(cv.take(l_bytes));
  b.o_suf = static_cast<float *>(cv.take(o_bytes));
  b.lse_suf = static_cast<float *>(cv.take(l_bytes));
  return cv.off;
}

}  // namespace

extern "C" int mla_prefill_workspace_bytes(const mla_dims_t *d, const int32_t *context_lens,
                                           const int32_t *query_lens, int32_t num_requests,
                                           int32_t row_budget, int32_t max_context_chunk,
                                           int32_t split_alignment, size_t *bytes) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!bytes || num_requests < 0 || (num_requests > 0 && (!context_lens || !query_lens)))
    return MLA_ERR_INVALID;
  PrefillLayout p;
  rc = build_prefill(*d, context_lens, query_lens, num_requests, row_budget, max_context_chunk,
                     split_alignment, p);
  if (rc) return rc;
  PrefillBuffers b;
  *bytes = carve_prefill(nullptr, *d, p, b);
  return MLA_OK;
}

extern "C" int mla_prefill_pinned_bytes(const mla_dims_t *d, const int32_t *context_lens,
                                        const int32_t *query_lens, int32_t num_requests,
                                        int32_t row_budget, int32_t max_context_chunk,
                                        int32_t split_alignment, size_t *bytes) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!bytes || num_requests < 0 || (num_requests > 0 && (!context_lens || !query_lens)))
    return MLA_ERR_INVALID;
  PrefillLayout p;
  rc = build_prefill(*d, context_lens, query_lens, num_requests, row_budget, max_context_chunk,
                     split_alignment, p);
  if (rc) return rc;
  *bytes = p.meta_total * sizeof(int32_t);
  return MLA_OK;
}

extern "C" int mla_chunked_prefill(const mla_dims_t *d, const int32_t *context_lens,
                                   const int32_t *query_lens, int32_t num_requests,
                                   int32_t row_budget, int32_t max_context_chunk,
                                   int32_t split_alignment, const void *q,
                                   const void *new_latent, const void *kv_cache,
                                   int32_t num_blocks, const int32_t *block_table,
                                   int32_t block_table_stride, const void *w_kv_b,
                                   void *workspace, size_t workspace_bytes, void *out,
                                   float *out_lse, void *pinned_scratch, size_t pinned_bytes,
                                   int32_t *dev_status, mla_stream_t stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (num_requests < 0 || (num_requests > 0 && (!context_lens || !query_lens)))
    return MLA_ERR_INVALID;
  PrefillLayout p;
  rc = build_prefill(*d, context_lens, query_lens, num_requests, row_budget, max_context_chunk,
                     split_alignment, p);
  if (rc) return rc;
  if (p.T == 0) return MLA_OK;
  if (!q || !new_latent || !w_kv_b || !workspace || !out) return MLA_ERR_INVALID;
  if (!p.chunks.empty() && (!kv_cache || !block_table || block_table_stride < 1))
    return MLA_ERR_INVALID;
  for (int r = 0; r < num_requests; ++r)
    if (int64_t(context_lens[r]) > int64_t(block_table_stride) * d->block_size)
      return MLA_ERR_INVALID;
  // buffers carved from the workspace keep its alignment (offsets are
  // multiples of 256); the gather moves 16-byte pieces of the cache
  if (!aligned16(workspace) || (kv_cache && !aligned16(kv_cache))) return MLA_ERR_INVALID;
  if (pinned_scratch && pinned_bytes < p.meta_total * sizeof(int32_t)) return MLA_ERR_TOO_SMALL;
  PrefillBuffers b;
  const size_t need = carve_prefill(nullptr, *d, p, b);
  if (workspace_bytes < need) return MLA_ERR_TOO_SMALL;
  // the tensor-core shape runs on the tensor-core kernels only (see tc_shape)
  const bool tc = tc_shape(*d);
  if (tc && (!aligned16(q) || !aligned16(new_latent) || !aligned16(w_kv_b) || !tc_available()))
    return MLA_ERR_UNSUPPORTED;
  carve_prefill(workspace, *d, p, b);

  std::vector<int32_t> meta(p.meta_total, 0);
  for (size_t c = 0; c < p.metas.size(); ++c)
    std::memcpy(meta.data() + p.meta_off[c], p.metas[c].ints.data(),
                p.metas[c].ints.size() * sizeof(int32_t));
  for (size_t k = 0; k < p.empty.size(); ++k) {
    meta[p.slices_off + 2 * k] = p.empty[k].first;
    meta[p.slices_off + 2 * k + 1] = p.empty[k].second;
  }
  std::memcpy(meta.data() + p.suffix_off, p.qsl.data(), p.qsl.size() * sizeof(int32_t));
  std::memcpy(meta.data() + p.last_off, p.last_rows.data(),
              p.last_rows.size() * sizeof(int32_t));
  std::memcpy(meta.data() + p.last_off + p.last_rows.size(), p.last_merge.data(),
              p.last_merge.size() * sizeof(int32_t));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::unique_lock<std::mutex> lock;
  Pipeline *pl = nullptr;
  rc = lock_pipeline(3 * p.metas.size() + 3, lock, &pl);
  if (rc) return rc;
  rc = upload_meta(*pl, b.meta, meta, pinned_scratch, pinned_bytes, s);
  if (rc) return rc;

  const int H = d->num_heads, Dv = d->v_dim, T = p.T;
  const int LP = d->kv_lora_rank + d->qk_rope_dim;
  const int es = elem_bytes(d->dtype);
  const int kv_dtype = b.chunk[0].kv_dtype;
  // the tensor-core attention reads the queries head-major with q_nope
  // already fp16: one pass (in the pipeline's pre step) instead of a strided
  // load and an fp16 conversion in every attention CTA
  const void *q_prep = tc ? b.q_prep : nullptr;
  // The last group's context attention and the new-token attention as one
  // launch of the looping or the persistent kernel (when the units suit
  // one of them):
  // each (request, query tile, head) unit walks the request's context rows
  // of that group, then its own new tokens causally, and merges with the
  // context partial only where an earlier group left one -- no second Q
  // load, no partial written and read back between the two.
  const size_t n_groups = p.metas.size();
  const bool merged = tc && n_groups > 0 &&
                      attn_tc_new_keys_ok(num_requests, p.qsl.data(), p.last_rows.data(),
                                          d->num_heads);

  // The chunk pipeline (run_pipeline) over execution groups: consecutive
  // chunks with no continuation between them and rows within the budget
  // together run as one gather, one up-projection and one attention (the
  // seven small chunks of the hetero batch cost 0.67 ms as separate
  // launches).  Group c uses buffer set c % 2, so the up-projection of group
  // c+1 fills the SMs that the attention of group c leaves idle (its tail, or
  // a long request's few CTAs, which is also why that attention is split over
  // its keys).  (Capping the GEMM at a share of the SMs, to run the two side
  // by side, was slower: its per-SM rate does not grow when fewer SMs share
  // HBM.)
  auto meta_of = [&](size_t c, const int32_t *&req, const int32_t *&st, const int32_t *&cu,
                     const int32_t *&ql, const int32_t *&acc) {
    const int n = p.metas[c].n;
    req = b.meta + p.meta_off[c];
    st = req + n;
    cu = st + n;
    ql = cu + n + 1;
    acc = ql + n + 1;
  };
  rc = run_pipeline(
      *pl, s, p.metas.size(),
      // the partial's context-free rows and the prepared queries, beside the
      // first gather and up-projection
      [&](cudaStream_t st_) {
        int r;
        {
          ProfRole role("a3 init partial");
          r = launch_fill_empty_rows(b.o_part, b.lse_part, T, H, Dv, int(p.empty.size()),
                                     b.meta + p.slices_off, st_);
        }
        ProfRole role("query preparation");
        if (!r && q_prep) r = launch_prepare_q(q, b.q_prep, T, H, dev_status, st_);
        return r;
      },
      [&](size_t c, cudaStream_t st_) {
        ProfRole role("a4 gather");
        const int32_t *req, *st, *cu, *ql, *acc;
        meta_of(c, req, st, cu, ql, acc);
        return launch_gather(kv_cache, num_blocks, d->block_size, LP * es, block_table,
                             block_table_stride, p.metas[c].n, req, st, cu, p.metas[c].rows,
                             b.chunk[c & 1].latent_ws, dev_status, st_);
      },
      [&](size_t c, cudaStream_t st_) {
        ProfRole role("a5 up-projection");
        return up_proj(*d, b.chunk[c & 1].latent_ws, LP, p.metas[c].rows, w_kv_b,
                       b.chunk[c & 1].kv_ws, kv_dtype, dev_status, st_);
      },
      [&](size_t c, cudaStream_t st_) {
        if (merged && c + 1 == n_groups) return int(MLA_OK);  // in the final launch
        ProfRole role("a6-a7 context attention");
        const ChunkMetaHost &m = p.metas[c];
        const int32_t *req, *st, *cu, *ql, *acc;
        meta_of(c, req, st, cu, ql, acc);
        return attention(*d, 0, m.n, ql, cu, m.q_loc.data(), m.cu_rows.data(), T, q,
                         b.chunk[c & 1].kv_ws, kv_dtype, m.rows, b.chunk[c & 1].latent_ws, LP,
                         acc, b.o_part, b.lse_part, dev_status, st_, &b.split, true, q_prep);
      },
      // new-token up-projection, beside the last group's attention (or,
      // when that attention is in the final launch, before the last
      // group's up-projection, so that the final launch waits on neither)
      [&](cudaStream_t st_) {
        ProfRole role("a8 new-token up-projection");
        return up_proj(*d, new_latent, LP, T, w_kv_b, b.kv_suffix, kv_dtype, dev_status, st_);
      },
      merged ? n_groups - 1 : SIZE_MAX);
  if (rc) return rc;

  const int32_t *sq = b.meta + p.suffix_off;
  if (merged) {
    ProfRole role("a6-a10 last context group + new tokens");
    const ChunkBuffers &cb = b.chunk[(n_groups - 1) & 1];
    const int32_t *lrows = b.meta + p.last_off, *lmerge = lrows + num_requests + 1;
    NewKeySource nks;
    nks.kv = b.kv_suffix;
    nks.latent = new_latent;
    nks.latent_ld = LP;
    return launch_attn_tc(*d, 0, num_requests, sq, lrows, p.qsl.data(), p.last_rows.data(), T,
                          p.metas.back().rows, q_prep, cb.kv_ws, cb.latent_ws, LP, lmerge,
                          b.o_part, b.lse_part, out, out_lse, d->dtype, p.pnt, nullptr, false,
                          true, dev_status, s, &nks);
  }
  ProfRole role("a9-a10 new-token attention + merge");
  if (tc) {
    // new-token attention with the final merge in its epilogue (row f3): the
    // context partial is read where needed, the output written once
    return launch_attn_tc(*d, 1, num_requests, sq, sq, p.qsl.data(), p.qsl.data(), T, T, q_prep,
                          b.kv_suffix, new_latent, LP, nullptr, b.o_part, b.lse_part, out,
                          out_lse, d->dtype, p.pnt, nullptr, false, true, dev_status, s);
  }
  rc = attention(*d, 1, num_requests, sq, sq, p.qsl.data(), p.qsl.data(), T, q, b.kv_suffix,
                 kv_dtype, T, new_latent, LP, nullptr, b.o_suf, b.lse_suf, dev_status, s);
  if (rc) return rc;
  return launch_merge(out, out_lse, b.o_part, b.lse_part, b.o_suf, b.lse_suf, T, H, Dv, p.pnt,
                      MLA_DTYPE_F32, d->dtype, s);
}

namespace mla {
namespace {
size_t fused_workspace(const mla_dims_t &d, int T, void *base, PrefillBuffers *b) {
  Carve cv(base);
  void *qp = cv.take(size_t(T) * d.num_heads * (d.qk_nope_dim + d.qk_rope_dim) * 2);
  const size_t rows_split = size_t(kSplitSlots) * d.num_heads * 128;
  void *so = cv.take(rows_split * d.v_dim * sizeof(float));
  void *sl = cv.take(rows_split * sizeof(float));
  if (b) {
    b->q_prep = qp;
    b->split.o = static_cast<float *>(so);
    b->split.lse = static_cast<float *>(sl);
    b->split.slots = kSplitSlots;
  }
  return cv.off;
}
}  // namespace
}  // namespace mla

extern "C" int mla_fused_attn_workspace_bytes(const mla_dims_t *d, int32_t num_tokens,
                                              size_t *bytes) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!bytes || num_tokens < 0) return MLA_ERR_INVALID;
  *bytes = fused_workspace(*d, num_tokens, nullptr, nullptr);
  return MLA_OK;
}

extern "C" int mla_fused_context_attn(const mla_dims_t *d, int32_t num_seqs,
                                      const int32_t *q_loc, const int32_t *k_loc,
                                      const int32_t *q_loc_host, const int32_t *k_loc_host,
                                      int32_t num_tokens, const void *q, const void *latent,
                                      int64_t latent_ld, int32_t latent_rows,
                                      const void *w_kv_b, const int32_t *accumulate, float *o,
                                      float *lse, void *workspace, size_t workspace_bytes,
                                      int32_t *dev_status, mla_stream_t stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (num_seqs < 0 || num_tokens < 0 || latent_rows < 0) return MLA_ERR_INVALID;
  if (num_seqs == 0) return MLA_OK;
  if (!q_loc || !k_loc || !q_loc_host || !k_loc_host || !q || !latent || !w_kv_b || !o ||
      !lse || !workspace)
    return MLA_ERR_INVALID;
  if (latent_ld < d->kv_lora_rank + d->qk_rope_dim) return MLA_ERR_INVALID;
  for (int i = 0; i < num_seqs; ++i)
    if (q_loc_host[i + 1] < q_loc_host[i] || k_loc_host[i + 1] < k_loc_host[i])
      return MLA_ERR_INVALID;
  if (q_loc_host[0] < 0 || q_loc_host[num_seqs] > num_tokens) return MLA_ERR_INVALID;
  if (k_loc_host[0] < 0 || latent_rows < k_loc_host[num_seqs]) return MLA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(latent) || !aligned16(w_kv_b) || !aligned16(workspace) ||
      !tc_available() || !fused_attn_ok(*d, latent_ld) ||
      !fused_attn_fits(num_seqs, q_loc_host, k_loc_host, 1))
    return MLA_ERR_UNSUPPORTED;
  PrefillBuffers b{};
  if (workspace_bytes < fused_workspace(*d, num_tokens, nullptr, nullptr))
    return MLA_ERR_TOO_SMALL;
  fused_workspace(*d, num_tokens, workspace, &b);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = launch_prepare_q(q, b.q_prep, num_tokens, d->num_heads, dev_status, s);
  if (rc) return rc;
  return launch_attn_fused(*d, num_seqs, q_loc, k_loc, q_loc_host, k_loc_host, num_tokens,
                           b.q_prep, latent, latent_ld, latent_rows, w_kv_b, accumulate, o, lse,
                           &b.split, dev_status, s);
}

extern "C" int mla_has_tcgen05(void) { return tc_available() ? 1 : 0; }

extern "C" int mla_kernel_launches(uint64_t *count) {
  if (!count) return MLA_ERR_INVALID;
  *count = g_kernel_launches.load(std::memory_order_relaxed);
  return MLA_OK;
}

namespace {
// the records' events go back to the thread's pool
void drop_profile() {
  for (const ProfRecord &r : g_prof.recs) {
    g_prof.pool.push_back(r.start);
    g_prof.pool.push_back(r.stop);
  }
  g_prof.recs.clear();
  if (g_prof.pending) g_prof.pool.push_back(g_prof.pending);
  g_prof.pending = nullptr;
}
}  // namespace

extern "C" int32_t mla_set_pipeline_overlap(int32_t on) {
  return g_overlap.exchange(on != 0 ? 1 : 0);
}

extern "C" int mla_profile_begin(void) {
  drop_profile();
  g_prof.on = true;
  return MLA_OK;
}

extern "C" int mla_profile_end(mla_launch_record_t *records, int32_t cap, int32_t *count) {
  if (!count || cap < 0 || (cap > 0 && !records)) return MLA_ERR_INVALID;
  g_prof.on = false;
  const int n = int(g_prof.recs.size());
  *count = n;
  int rc = MLA_OK;
  std::vector<cudaStream_t> streams;  // in order of first appearance
  for (int i = 0; i < n && i < cap && rc == MLA_OK; ++i) {
    const ProfRecord &r = g_prof.recs[i];
    float ms = 0.f, at = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess ||
        cudaEventElapsedTime(&at, g_prof.recs[0].start, r.start) != cudaSuccess) {
      rc = MLA_ERR_CUDA;
      break;
    }
    int sid = 0;
    while (sid < int(streams.size()) && streams[sid] != r.stream) ++sid;
    if (sid == int(streams.size())) streams.push_back(r.stream);
    mla_launch_record_t &o = records[i];
    std::memset(&o, 0, sizeof(o));
    std::strncpy(o.kernel, r.name, sizeof(o.kernel) - 1);
    std::strncpy(o.role, r.role, sizeof(o.role) - 1);
    o.stream = sid;
    o.start_ms = at;
    o.ms = ms;
  }
  drop_profile();
  if (rc) return rc;
  return n > cap ? MLA_ERR_TOO_SMALL : MLA_OK;
}

extern "C" int mla_selftest_bounded_wait(int32_t limit_us, int32_t *gave_up,
                                         mla_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000 || !gave_up) return MLA_ERR_INVALID;
  if (!tc_available()) return MLA_ERR_UNSUPPORTED;
  int dev = 0, khz = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev);
  if (khz <= 0) khz = 2000000;
  return launch_bounded_wait_selftest(static_cast<long long>(limit_us) * khz / 1000, gave_up,
                                      static_cast<cudaStream_t>(stream));
}

extern "C" int mla_device_error_flags(int32_t *flags) {
  if (!flags) return MLA_ERR_INVALID;
  if (cudaDeviceSynchronize() != cudaSuccess) return MLA_ERR_CUDA;
  const int a = gemm_take_errors(), b = attn_take_errors(), c = fused_take_errors(),
            e = gather_take_errors();
  if (a < 0 || b < 0 || c < 0 || e < 0) return MLA_ERR_CUDA;
  *flags = a | b | c | e;
  return MLA_OK;
}

// ---------------------------------------------------------------------------
// The old scheme, kept as a comparator: equal context windows for every
// request with context (PR #50613 report, motivation; PR #49294 report,
// build_mla_chunked_context_metadata and mask_empty_context).  Each chunk
// runs the gather, up-projection and attention over the whole batch, fixes
// the rows of requests whose window is empty, and merges into the running
// partial.
namespace mla {
namespace {

int plan_equal_window(const int32_t *ctx, int R, int budget, int align, int &window,
                      int &n_chunks) {
  if (R < 0 || budget < 1 || align < 1 || (R > 0 && !ctx)) return MLA_ERR_INVALID;
  int with_ctx = 0, mx = 0;
  for (int r = 0; r < R; ++r) {
    if (ctx[r] < 0) return MLA_ERR_INVALID;
    if (ctx[r] > 0) ++with_ctx;
    mx = std::max(mx, int(ctx[r]));
  }
  window = n_chunks = 0;
  if (with_ctx == 0) return MLA_OK;
  window = budget / with_ctx / align * align;
  if (window <= 0) return MLA_ERR_PLANNER_STUCK;
  n_chunks = (mx + window - 1) / window;
  return MLA_OK;
}

struct EqualWindowLayout {
  int window = 0, n_chunks = 0, T = 0, pnt = 0, max_rows = 0, R = 0;
  std::vector<int32_t> qsl;
  std::vector<ChunkMetaHost> metas;  // every chunk lists every request
  std::vector<size_t> meta_off;
  std::vector<char> has_empty;
  size_t slice_off = 0, suffix_off = 0, meta_total = 0;
};

int build_equal_window(const int32_t *ctx, const int32_t *ql, int R, int budget, int align,
                       EqualWindowLayout &p) {
  for (int r = 0; r < R; ++r)
    if (ql[r] < 0) return MLA_ERR_INVALID;
  int rc = plan_equal_window(ctx, R, budget, align, p.window, p.n_chunks);
  if (rc) return rc;
  p.R = R;
  p.qsl.assign(R + 1, 0);
  for (int r = 0; r < R; ++r) p.qsl[r + 1] = p.qsl[r] + ql[r];
  p.T = p.qsl[R];
  int last = -1;
  for (int r = 0; r < R; ++r)
    if (ctx[r] > 0) last = r;
  p.pnt = last >= 0 ? p.qsl[last + 1] : 0;
  std::vector<int32_t> st(R), ln(R);
  size_t off = 0;
  p.metas.resize(p.n_chunks);
  for (int c = 0; c < p.n_chunks; ++c) {
    bool empty = false;
    int rows = 0;
    for (int r = 0; r < R; ++r) {
      const int64_t lo = std::min<int64_t>(int64_t(c) * p.window, ctx[r]);
      const int64_t hi = std::min<int64_t>(int64_t(c + 1) * p.window, ctx[r]);
      st[r] = int32_t(lo);
      ln[r] = int32_t(hi - lo);
      rows += ln[r];
      empty = empty || ln[r] == 0;
    }
    const mla_chunk_t chunk{0, R, 0, rows, 0};
    build_chunk_meta(chunk, st.data(), ln.data(), p.qsl.data(), p.metas[c]);
    // the old scheme writes every chunk's result in full: no accumulate flags
    std::fill(p.metas[c].ints.begin() + 4 * R + 2, p.metas[c].ints.end(), 0);
    p.meta_off.push_back(off);
    off += p.metas[c].ints.size();
    p.has_empty.push_back(empty ? 1 : 0);
    p.max_rows = std::max(p.max_rows, rows);
  }
  p.slice_off = off;
  off += 2;
  p.suffix_off = off;
  off += R + 1;
  p.meta_total = off;
  return MLA_OK;
}

struct EqualWindowBuffers {
  int32_t *meta;
  ChunkBuffers chunk[2];  // chunk c uses set c % 2 (the same pipeline as the new path)
  void *q_prep;           // as in the new path
  void *kv_suffix;
  float *o_run[2], *lse_run[2];  // running partial, ping-ponged per chunk
  float *o_chunk, *lse_chunk, *o_suf, *lse_suf;
};

size_t carve_equal_window(void *base, const mla_dims_t &d, const EqualWindowLayout &p,
                          EqualWindowBuffers &b) {
  Carve cv(base);
  b.meta = static_cast<int32_t *>(cv.take(p.meta_total * sizeof(int32_t)));
  const int sets = p.n_chunks > 1 ? 2 : 1;
  for (int k = 0; k < 2; ++k) {
    if (k < sets)
      carve_chunk_buffers(cv, d, p.max_rows, b.chunk[k]);
    else
      b.chunk[k] = b.chunk[0];
  }
  b.q_prep = cv.take(size_t(p.T) * d.num_heads * (d.qk_nope_dim + d.qk_rope_dim) * 2);
  b.kv_suffix = cv.take(size_t(p.T) * kv_width(d) * elem_bytes(b.chunk[0].kv_dtype));
  const size_t o_bytes = size_t(p.T) * d.num_heads * d.v_dim * sizeof(float);
  const size_t l_bytes = size_t(p.T) * d.num_heads * sizeof(float);
  for (int k = 0; k < 2; ++k) {
    b.o_run[k] = static_cast<float *>(cv.take(o_bytes));
    b.lse_run[k] = static_cast<float *>(cv.take(l_bytes));
  }
  b.o_chunk = static_cast<float *>(cv.take(o_bytes));
  b.lse_chunk = static_cast<float *>(cv.take(l_bytes));
  b.o_suf = static_cast<float *>(cv.take(o_bytes));
  b.lse_suf = static_cast<float *>(cv.take(l_bytes));
  return cv.off;
}

}  // namespace
}  // namespace mla

extern "C" int mla_plan_equal_window_chunks(const int32_t *context_lens, int32_t num_requests,
                                            int32_t row_budget, int32_t split_alignment,
                                            int32_t *window, int32_t *num_chunks) {
  if (!window || !num_chunks) return MLA_ERR_INVALID;
  int w = 0, n = 0;
  const int rc = plan_equal_window(context_lens, num_requests, row_budget, split_alignment, w, n);
  if (rc) return rc;
  *window = w;
  *num_chunks = n;
  return MLA_OK;
}

extern "C" int mla_prefill_equal_window_workspace_bytes(const mla_dims_t *d,
                                                        const int32_t *context_lens,
                                                        const int32_t *query_lens,
                                                        int32_t num_requests, int32_t row_budget,
                                                        int32_t split_alignment, size_t *bytes) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!bytes || num_requests < 0 || (num_requests > 0 && (!context_lens || !query_lens)))
    return MLA_ERR_INVALID;
  EqualWindowLayout p;
  rc = build_equal_window(context_lens, query_lens, num_requests, row_budget, split_alignment, p);
  if (rc) return rc;
  EqualWindowBuffers b;
  *bytes = carve_equal_window(nullptr, *d, p, b);
  return MLA_OK;
}

extern "C" int mla_chunked_prefill_equal_window(
    const mla_dims_t *d, const int32_t *context_lens, const int32_t *query_lens,
    int32_t num_requests, int32_t row_budget, int32_t split_alignment, const void *q,
    const void *new_latent, const void *kv_cache, int32_t num_blocks, const int32_t *block_table,
    int32_t block_table_stride, const void *w_kv_b, void *workspace, size_t workspace_bytes,
    void *out, float *out_lse, int32_t *dev_status, mla_stream_t stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (num_requests < 0 || (num_requests > 0 && (!context_lens || !query_lens)))
    return MLA_ERR_INVALID;
  EqualWindowLayout p;
  rc = build_equal_window(context_lens, query_lens, num_requests, row_budget, split_alignment, p);
  if (rc) return rc;
  if (p.T == 0) return MLA_OK;
  if (!q || !new_latent || !w_kv_b || !workspace || !out) return MLA_ERR_INVALID;
  if (p.n_chunks > 0 && (!kv_cache || !block_table || block_table_stride < 1))
    return MLA_ERR_INVALID;
  for (int r = 0; r < num_requests; ++r)
    if (int64_t(context_lens[r]) > int64_t(block_table_stride) * d->block_size)
      return MLA_ERR_INVALID;
  if (!aligned16(workspace) || (kv_cache && !aligned16(kv_cache))) return MLA_ERR_INVALID;
  EqualWindowBuffers b;
  if (workspace_bytes < carve_equal_window(nullptr, *d, p, b)) return MLA_ERR_TOO_SMALL;
  const bool tc = tc_shape(*d);
  if (tc && (!aligned16(q) || !aligned16(new_latent) || !aligned16(w_kv_b) || !tc_available()))
    return MLA_ERR_UNSUPPORTED;
  carve_equal_window(workspace, *d, p, b);
  std::vector<int32_t> meta(p.meta_total, 0);
  for (int c = 0; c < p.n_chunks; ++c)
    std::memcpy(meta.data() + p.meta_off[c], p.metas[c].ints.data(),
                p.metas[c].ints.size() * sizeof(int32_t));
  meta[p.slice_off] = 0;
  meta[p.slice_off + 1] = p.T;
  std::memcpy(meta.data() + p.suffix_off, p.qsl.data(), p.qsl.size() * sizeof(int32_t));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::unique_lock<std::mutex> lock;
  Pipeline *pl = nullptr;
  rc = lock_pipeline(3 * size_t(p.n_chunks) + 3, lock, &pl);
  if (rc) return rc;
  rc = upload(b.meta, meta, s);
  if (rc) return rc;
  const int H = d->num_heads, Dv = d->v_dim, T = p.T, R = p.R;
  const int LP = d->kv_lora_rank + d->qk_rope_dim;
  const int es = elem_bytes(d->dtype);
  const int kv_dtype = b.chunk[0].kv_dtype;
  const void *q_prep = tc ? b.q_prep : nullptr;
  // the chunks run through the same two-buffer pipeline as the new path, so
  // the two schemes differ in their chunks, not in how a chunk is executed
  rc = run_pipeline(
      *pl, s, size_t(p.n_chunks),
      // the running partial starts empty (O = 0, LSE = -inf); the prepared
      // queries
      [&](cudaStream_t st_) {
        int r = launch_fill_empty_rows(b.o_run[0], b.lse_run[0], T, H, Dv, 1,
                                       b.meta + p.slice_off, st_);
        if (!r && q_prep) r = launch_prepare_q(q, b.q_prep, T, H, dev_status, st_);
        return r;
      },
      [&](size_t c, cudaStream_t st_) {
        const ChunkMetaHost &m = p.metas[c];
        const int32_t *req = b.meta + p.meta_off[c], *st = req + R, *cu = st + R;
        if (m.rows == 0) return int(MLA_OK);
        return launch_gather(kv_cache, num_blocks, d->block_size, LP * es, block_table,
                             block_table_stride, R, req, st, cu, m.rows,
                             b.chunk[c & 1].latent_ws, dev_status, st_);
      },
      [&](size_t c, cudaStream_t st_) {
        return up_proj(*d, b.chunk[c & 1].latent_ws, LP, p.metas[c].rows, w_kv_b,
                       b.chunk[c & 1].kv_ws, kv_dtype, dev_status, st_);
      },
      [&](size_t c, cudaStream_t st_) {
        const ChunkMetaHost &m = p.metas[c];
        const int32_t *req = b.meta + p.meta_off[c], *st = req + R, *cu = st + R,
                      *ql = cu + R + 1;
        int r = attention(*d, 0, R, ql, cu, m.q_loc.data(), m.cu_rows.data(), T, q,
                          b.chunk[c & 1].kv_ws, kv_dtype, m.rows, b.chunk[c & 1].latent_ws, LP,
                          nullptr, b.o_chunk, b.lse_chunk, dev_status, st_, nullptr, false,
                          q_prep);
        if (!r && p.has_empty[c])
          r = launch_mask_empty_context(b.lse_chunk, b.o_chunk, MLA_DTYPE_F32, T, H, Dv, R, ql,
                                        cu, st_);
        if (!r)
          r = launch_merge(b.o_run[(c + 1) & 1], b.lse_run[(c + 1) & 1], b.o_run[c & 1],
                           b.lse_run[c & 1], b.o_chunk, b.lse_chunk, T, H, Dv, T, MLA_DTYPE_F32,
                           MLA_DTYPE_F32, st_);
        return r;
      },
      [&](cudaStream_t st_) {
        return up_proj(*d, new_latent, LP, T, w_kv_b, b.kv_suffix, kv_dtype, dev_status, st_);
      });
  if (rc) return rc;
  const int32_t *sq = b.meta + p.suffix_off;
  rc = attention(*d, 1, R, sq, sq, p.qsl.data(), p.qsl.data(), T, q, b.kv_suffix,
                 kv_dtype, T, new_latent, LP, nullptr, b.o_suf, b.lse_suf, dev_status, s,
                 nullptr, false, q_prep);
  if (rc) return rc;
  const int fin = p.n_chunks & 1;  // the buffer the last chunk merged into
  return launch_merge(out, out_lse, b.o_run[fin], b.lse_run[fin], b.o_suf, b.lse_suf, T, H, Dv,
                      p.pnt, MLA_DTYPE_F32, d->dtype, s);
}
