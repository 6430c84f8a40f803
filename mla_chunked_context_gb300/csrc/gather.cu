// Paged-cache gather of a chunk's context rows into the dense latent
// workspace (PR #50613 report, item 2: every context row of a chunk is
// gathered exactly once, at the workspace offsets cu_seq_lens).
//
// HBM-bound copy: a warp takes four workspace rows at a time.  It resolves
// each row's sequence (binary search on cu_rows, one broadcast load per
// step), logical context position and physical block, then its 32 lanes move
// the rows' (L+P)*elem bytes as coalesced 16-byte vectors, all loads of the
// four rows issued before the stores.  A block id outside [0, num_blocks) is
// not dereferenced: the row is written as zeros and a status bit is set for
// the host.
#include "common.cuh"

namespace mla {
namespace {

constexpr int ROWS_PER_WARP = 4;  // rows a warp moves at once
constexpr int VEC_PER_LANE = 3;   // 16-byte pieces per lane and row (rows <= 1536 B)

__device__ __forceinline__ bool row_source(const int32_t *__restrict__ block_table, int bt_stride,
                                           int num_blocks, int block_size, int num_seqs,
                                           const int32_t *__restrict__ seq_request,
                                           const int32_t *__restrict__ seq_start,
                                           const int32_t *__restrict__ cu_rows, int row,
                                           int64_t *src_row) {
  const int i = find_seq(cu_rows, num_seqs, row);
  const int j = __ldg(seq_start + i) + (row - __ldg(cu_rows + i));
  const int r = __ldg(seq_request + i);
  const int blk = __ldg(block_table + int64_t(r) * bt_stride + j / block_size);
  if (blk < 0 || blk >= num_blocks) return false;
  *src_row = int64_t(blk) * block_size + (j % block_size);
  return true;
}

// One warp per ROWS_PER_WARP workspace rows: the rows' sources are resolved
// first (sequence by binary search on cu_rows, logical position, physical
// block), then every lane issues all of its 16-byte loads for those rows
// before any store, so each lane keeps up to 12 loads in flight.
__global__ void __launch_bounds__(256) gather_rows_kernel(
    const uint4 *__restrict__ cache, int num_blocks, int block_size, int vec_per_row,
    const int32_t *__restrict__ block_table, int bt_stride, int num_seqs,
    const int32_t *__restrict__ seq_request, const int32_t *__restrict__ seq_start,
    const int32_t *__restrict__ cu_rows, int total_rows, uint4 *__restrict__ ws,
    int32_t *status) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int w0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int row0 = w0 * ROWS_PER_WARP; row0 < total_rows; row0 += warps * ROWS_PER_WARP) {
    int64_t src[ROWS_PER_WARP];
    bool ok[ROWS_PER_WARP];
#pragma unroll
    for (int r = 0; r < ROWS_PER_WARP; ++r) {
      const int row = row0 + r;
      ok[r] = row < total_rows &&
              row_source(block_table, bt_stride, num_blocks, block_size, num_seqs, seq_request,
                         seq_start, cu_rows, row, &src[r]);
      if (row < total_rows && !ok[r] && lane == 0 && status)
        atomicOr(status, MLA_STATUS_BAD_BLOCK);
    }
    if (vec_per_row <= 32 * VEC_PER_LANE) {
      uint4 v[ROWS_PER_WARP][VEC_PER_LANE];
#pragma unroll
      for (int r = 0; r < ROWS_PER_WARP; ++r)
#pragma unroll
        for (int k = 0; k < VEC_PER_LANE; ++k) {
          const int c = lane + 32 * k;
          v[r][k] = (ok[r] && c < vec_per_row) ? __ldcs(cache + src[r] * vec_per_row + c) : zero;
        }
#pragma unroll
      for (int r = 0; r < ROWS_PER_WARP; ++r) {
        if (row0 + r >= total_rows) break;
        uint4 *dst = ws + int64_t(row0 + r) * vec_per_row;
#pragma unroll
        for (int k = 0; k < VEC_PER_LANE; ++k) {
          const int c = lane + 32 * k;
          if (c < vec_per_row) __stcg(dst + c, v[r][k]);
        }
      }
    } else {  // wider rows: plain strided copy
      for (int r = 0; r < ROWS_PER_WARP && row0 + r < total_rows; ++r) {
        uint4 *dst = ws + int64_t(row0 + r) * vec_per_row;
        for (int c = lane; c < vec_per_row; c += 32)
          __stcg(dst + c, ok[r] ? __ldcs(cache + src[r] * vec_per_row + c) : zero);
      }
    }
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
  const int64_t warps_needed = (int64_t(total_rows) + ROWS_PER_WARP - 1) / ROWS_PER_WARP;
  int64_t blocks = (warps_needed * 32 + 255) / 256;
  const int64_t cap = int64_t(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  launch_begin(s);
  gather_rows_kernel<<<int(blocks), 256, 0, s>>>(
      static_cast<const uint4 *>(cache), num_blocks, block_size, vec_per_row, block_table,
      bt_stride, num_seqs, seq_request, seq_start, cu_rows, total_rows,
      static_cast<uint4 *>(ws), status);
  return launch_status(s, "gather_rows_kernel");
}

}  // namespace mla
