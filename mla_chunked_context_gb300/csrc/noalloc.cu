// mla_context_chunk_attn_noalloc: the chunk pipeline (gather, up-projection,
// attention + accumulate) with its scratch in a library-owned device array, for
// callers that cannot allocate device memory themselves -- for example a
// plugin whose host framework owns every device allocation and hands it no
// workspace, or a caller on a path where a cudaMalloc (which can synchronise
// the device) is not allowed.
//
// The scratch is one file-scope device array of MLA_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  Host
// code never passes the array's name to a kernel (in host code that name is a
// host-side stand-in, not a device address): the first call on a device,
// with that device current, looks up the array's device address with
// cudaGetSymbolAddress and keeps it for later calls on that device.
//
// All calls share the array and it keeps the last call's contents.  Nothing
// in it has to start at zero: each call writes every byte it later reads
// (metadata upload, gathered rows, up-projected K/V).  Calls that overlap on
// the GPU (different streams, or threads without ordering between them) race
// on the array and must be serialised by the caller.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of this device's scratch array (looked up once per device).
int scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MLA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" int mla_context_chunk_attn_noalloc(
    const mla_dims_t *d, const mla_chunk_t *chunk, const int32_t *starts,
    const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_tokens, const void *q,
    const void *kv_cache, int32_t num_blocks, const int32_t *block_table,
    int32_t block_table_stride, const void *w_kv_b, float *o_partial, float *lse_partial,
    int32_t *dev_status, mla_stream_t stream) {
  if (!d || !chunk || !starts || !seq_lens) return MLA_ERR_INVALID;
  const int n = chunk->request_end - chunk->request_start;
  if (n < 1 || chunk->entry_offset < 0) return MLA_ERR_INVALID;
  int64_t rows = 0;
  for (int i = 0; i < n; ++i) rows += seq_lens[chunk->entry_offset + i];
  if (rows > INT32_MAX) return MLA_ERR_TOO_SMALL;
  size_t need = 0;
  int rc = mla_chunk_workspace_bytes(d, int32_t(rows), n, &need);
  if (rc) return rc;
  if (need > MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_TOO_SMALL;  // chunk too large
  void *scratch = nullptr;
  rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  return mla_context_chunk_attn(d, chunk, starts, seq_lens, query_start_loc, num_tokens, q,
                                kv_cache, num_blocks, block_table, block_table_stride, w_kv_b,
                                scratch, MLA_NOALLOC_SCRATCH_BYTES, o_partial, lse_partial,
                                dev_status, stream);
}
