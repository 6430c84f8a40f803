// Paged-cache gather of a chunk's context rows into the dense latent
// workspace (PR #50613 report, item 2: every context row of a chunk is
// gathered exactly once, at the workspace offsets cu_seq_lens).
//
// HBM-bound copy: one warp per workspace row.  The warp resolves the row's
// sequence (binary search on cu_rows, one broadcast load per step), its
// logical context position and the physical block once, then its 32 lanes
// move the row's (L+P)*elem bytes as coalesced 16-byte vectors.  A block id
// outside [0, num_blocks) is not dereferenced: the row is written as zeros
// and a status bit is set for the host.
#include "common.cuh"

namespace mla {
namespace {

__global__ void __launch_bounds__(256) gather_rows_kernel(
    const uint4 *__restrict__ cache, int num_blocks, int block_size, int vec_per_row,
    const int32_t *__restrict__ block_table, int bt_stride, int num_seqs,
    const int32_t *__restrict__ seq_request, const int32_t *__restrict__ seq_start,
    const int32_t *__restrict__ cu_rows, int total_rows, uint4 *__restrict__ ws,
    int32_t *status) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < total_rows;
       row += warps) {
    const int i = find_seq(cu_rows, num_seqs, row);
    const int j = __ldg(seq_start + i) + (row - __ldg(cu_rows + i));
    const int r = __ldg(seq_request + i);
    const int blk = __ldg(block_table + int64_t(r) * bt_stride + j / block_size);
    uint4 *dst = ws + int64_t(row) * vec_per_row;
    if (blk < 0 || blk >= num_blocks) {
      for (int v = lane; v < vec_per_row; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
      if (lane == 0 && status) atomicOr(status, MLA_STATUS_BAD_BLOCK);
      continue;
    }
    const uint4 *src =
        cache + (int64_t(blk) * block_size + (j % block_size)) * vec_per_row;
    for (int v = lane; v < vec_per_row; v += 32) __stcg(dst + v, __ldcs(src + v));
  }
}

}  // namespace

int launch_gather(const void *cache, int num_blocks, int block_size, int row_bytes,
                  const int32_t *block_table, int bt_stride, int num_seqs,
                  const int32_t *seq_request, const int32_t *seq_start,
                  const int32_t *cu_rows, int total_rows, void *ws, int32_t *status,
                  cudaStream_t s) {
  if (total_rows == 0) return MLA_OK;
  const int vec_per_row = row_bytes / 16;
  const int64_t warps_needed = total_rows;
  int64_t blocks = (warps_needed * 32 + 255) / 256;
  const int64_t cap = int64_t(num_sms()) * 16;
  if (blocks > cap) blocks = cap;
  gather_rows_kernel<<<int(blocks), 256, 0, s>>>(
      static_cast<const uint4 *>(cache), num_blocks, block_size, vec_per_row, block_table,
      bt_stride, num_seqs, seq_request, seq_start, cu_rows, total_rows,
      static_cast<uint4 *>(ws), status);
  return launch_status();
}

}  // namespace mla
