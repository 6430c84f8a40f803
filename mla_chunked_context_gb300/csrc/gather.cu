// Paged-cache gather of a chunk's context rows into the dense latent
// workspace (PR #50613 report, item 2: every context row of a chunk is
// gathered exactly once, at the workspace offsets cu_seq_lens), staged in
// shared memory by the bulk-copy (TMA) engine.
//
// The workspace is cut into windows of 32 rows.  For each window one warp
// resolves the source of its 32 rows (lane = row: sequence by binary search
// on cu_rows, logical context position, physical block from the block
// table), splits them into runs of rows that are consecutive in the cache
// (a run never crosses a cache block unless the next physical block follows
// in memory), and every lane that starts a run issues one bulk copy of the
// whole run into the window's shared-memory stage.  When the window's bytes
// have landed (mbarrier transaction count) one bulk copy writes the stage to
// the workspace, which is contiguous for the window.  Three stages: the
// loads of window k run while the store of window k-1 drains, and the next
// window's sources are resolved while the loads are in flight.  A block id
// outside [0, num_blocks) is not dereferenced: the row is written as zeros
// and a status bit is set for the host.  Every wait is bounded.
#include <algorithm>

#include "sm103.cuh"

namespace mla {
namespace {

using namespace sm103;

constexpr int WROWS = 32;      // rows per window (one per lane)
constexpr int STAGES = 3;      // windows in shared memory
constexpr int MAX_ROW_BYTES = 2048;

struct RowSrc {
  int64_t src;  // source row of the cache (physical block * bs + slot); -1: bad block
  bool live;    // the row exists (row < total_rows)
};

__device__ __forceinline__ RowSrc resolve_row(const int32_t *__restrict__ block_table,
                                              int bt_stride, int num_blocks, int block_size,
                                              int num_seqs,
                                              const int32_t *__restrict__ seq_request,
                                              const int32_t *__restrict__ seq_start,
                                              const int32_t *__restrict__ cu_rows,
                                              int total_rows, int row) {
  RowSrc r{-1, row < total_rows};
  if (!r.live) return r;
  const int i = find_seq(cu_rows, num_seqs, row);
  const int j = __ldg(seq_start + i) + (row - __ldg(cu_rows + i));
  const int req = __ldg(seq_request + i);
  const int blk = __ldg(block_table + int64_t(req) * bt_stride + j / block_size);
  if (blk >= 0 && blk < num_blocks) r.src = int64_t(blk) * block_size + (j % block_size);
  return r;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}

// One warp per CTA; windows w = blockIdx.x, + gridDim.x, ...
__global__ void __launch_bounds__(32) gather_bulk_kernel(
    const uint8_t *__restrict__ cache, int num_blocks, int block_size, int row_bytes,
    const int32_t *__restrict__ block_table, int bt_stride, int num_seqs,
    const int32_t *__restrict__ seq_request, const int32_t *__restrict__ seq_start,
    const int32_t *__restrict__ cu_rows, int total_rows, uint8_t *__restrict__ ws,
    int32_t *status) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x;
  const uint32_t stage_bytes = uint32_t(WROWS) * row_bytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * stage_bytes);
  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(smem_u32(bars + s), 1);
    fence_mbar_init();
  }
  __syncwarp();
  const int nwin = (total_rows + WROWS - 1) / WROWS;
  auto resolve = [&](int w) {
    return resolve_row(block_table, bt_stride, num_blocks, block_size, num_seqs, seq_request,
                       seq_start, cu_rows, total_rows, w * WROWS + lane);
  };
  RowSrc cur = resolve(blockIdx.x);
  bool ok = true;
  int kk = 0;
  for (int w = blockIdx.x; w < nwin && ok; w += gridDim.x, ++kk) {
    const int s = kk % STAGES;
    uint8_t *stage = smem + s * stage_bytes;
    // the stage's previous window (kk - STAGES) has been read by its store:
    // stores 0 .. kk-2 are issued, at most STAGES-2 of them may still read
    if (lane == 0) bulk_wait_read<STAGES - 2>();
    __syncwarp();
    const bool valid = cur.live && cur.src >= 0;
    if (cur.live && cur.src < 0) {
      if (status) atomicOr(status, MLA_STATUS_BAD_BLOCK);
      uint4 *z = reinterpret_cast<uint4 *>(stage + lane * row_bytes);
      for (int c = 0; c < row_bytes / 16; ++c) z[c] = make_uint4(0, 0, 0, 0);
    }
    // runs of rows consecutive in the cache: a run starts where the previous
    // lane's row is not the cache row just before this one
    const int64_t prev = __shfl_up_sync(0xffffffffu, cur.src, 1);
    const bool prev_valid = __shfl_up_sync(0xffffffffu, valid ? 1 : 0, 1) != 0;
    const bool start = valid && (lane == 0 || !prev_valid || prev + 1 != cur.src);
    const uint32_t starts = __ballot_sync(0xffffffffu, start);
    const uint32_t stops = starts | __ballot_sync(0xffffffffu, !valid);
    const int n_valid = __popc(__ballot_sync(0xffffffffu, valid));
    const uint32_t bar = smem_u32(bars + s);
    if (lane == 0) mbar_expect_tx(bar, uint32_t(n_valid) * row_bytes);
    __syncwarp();
    if (start) {
      const uint32_t above = lane == 31 ? 0u : (stops & ~((2u << lane) - 1u));
      const int end = above ? __ffs(above) - 1 : WROWS;
      bulk_load(smem_u32(stage + lane * row_bytes), cache + cur.src * row_bytes,
                uint32_t(end - lane) * row_bytes, bar);
    }
    // the next window's sources, while this one's copies are in flight
    cur = resolve(w + gridDim.x);
    // store the previous window
    if (kk >= 1) {
      const int sp = (kk - 1) % STAGES;
      const bool landed = mbar_wait(smem_u32(bars + sp), uint32_t(((kk - 1) / STAGES) & 1));
      ok = __all_sync(0xffffffffu, landed) != 0;  // the warp leaves the loop together
      fence_async_smem();  // the zero rows written with plain stores
      __syncwarp();
      if (ok && lane == 0) {
        const int wp = w - int(gridDim.x);
        const int rows = min(WROWS, total_rows - wp * WROWS);
        bulk_store(ws + int64_t(wp) * WROWS * row_bytes, smem_u32(smem + sp * stage_bytes),
                   uint32_t(rows) * row_bytes);
        bulk_commit();
      }
    }
  }
  // the last window's store; then every store has finished before exit
  if (kk >= 1) {
    const int sp = (kk - 1) % STAGES;
    const bool landed =
        __all_sync(0xffffffffu, mbar_wait(smem_u32(bars + sp), uint32_t(((kk - 1) / STAGES) & 1)));
    fence_async_smem();
    __syncwarp();
    if (ok && landed && lane == 0) {
      const int wp = int(blockIdx.x) + (kk - 1) * int(gridDim.x);
      const int rows = min(WROWS, total_rows - wp * WROWS);
      bulk_store(ws + int64_t(wp) * WROWS * row_bytes, smem_u32(smem + sp * stage_bytes),
                 uint32_t(rows) * row_bytes);
      bulk_commit();
    }
  }
  if (lane == 0) bulk_wait_all();
  __syncwarp();
}

}  // namespace

int launch_gather(const void *cache, int num_blocks, int block_size, int row_bytes,
                  const int32_t *block_table, int bt_stride, int num_seqs,
                  const int32_t *seq_request, const int32_t *seq_start,
                  const int32_t *cu_rows, int total_rows, void *ws, int32_t *status,
                  cudaStream_t s) {
  if (total_rows == 0) return MLA_OK;
  if (row_bytes % 16 != 0 || row_bytes > MAX_ROW_BYTES) return MLA_ERR_UNSUPPORTED;
  const int smem = STAGES * WROWS * row_bytes + STAGES * 8;
  static int attr_bytes = 0;
  if (smem > attr_bytes) {
    if (cudaFuncSetAttribute(gather_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             STAGES * WROWS * MAX_ROW_BYTES + STAGES * 8) != cudaSuccess)
      return MLA_ERR_CUDA;
    attr_bytes = STAGES * WROWS * MAX_ROW_BYTES + STAGES * 8;
  }
  const int nwin = (total_rows + WROWS - 1) / WROWS;
  // persistent: as many one-warp CTAs as fit (two per SM at 1152-byte rows)
  const int per_sm = smem > 0 ? std::max(1, std::min(8, (220 * 1024) / smem)) : 1;
  const int grid = std::min(nwin, per_sm * num_sms());
  launch_begin(s);
  gather_bulk_kernel<<<grid, WROWS, smem, s>>>(
      static_cast<const uint8_t *>(cache), num_blocks, block_size, row_bytes, block_table,
      bt_stride, num_seqs, seq_request, seq_start, cu_rows, total_rows,
      static_cast<uint8_t *>(ws), status);
  return launch_status(s, "gather_bulk_kernel");
}

int gather_take_errors() { return sm103::take_error_flags_here(); }

}  // namespace mla
