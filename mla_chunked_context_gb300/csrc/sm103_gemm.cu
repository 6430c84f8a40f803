// W_kv_b up-projection on the 5th-generation tensor cores (sm_103a):
//   kv[h, m, c] = sum_k latent[m, k] w_kv_b[h*(Dn+Dv) + c, k]
//   (bf16 in, f32 accumulate, fp16/bf16 out; head-major output [H, M, Dn+Dv])
// M = context rows of a chunk (or new tokens), K = kv_lora_rank, N = H*(Dn+Dv).
// Head-major output makes each 128x256 output tile one contiguous 64 KB block
// (row-major [M, N] put its 128 rows 64 KB apart, and the TMA stores of that
// pattern ran at 2.7 TB/s and held the kernel to 70% of the tensor peak it
// reaches without them).
// The MLA up-projection is not on the pages; it is the standard MLA prefill
// step that turns the gathered latent rows into per-head K_nope and V.
//
// Design: persistent, warp-specialised, 2-SM MMA, A-stationary.  CTAs run
// in pairs (a cluster of two, one CTA per SM); a pair computes 256x256 output
// tiles with tcgen05.mma.cta_group::2 (M=256: 128 rows in each SM's tensor
// memory).  Each SM holds only its own 128 A rows and its half (128 rows) of
// the B tile.  A work unit is (256-row block of the latent, segment of the
// N tiles): the pair loads the block's A rows once (all of K, 128 KB per SM,
// resident for the unit) and streams only B through a 5-stage ring.  Per
// tile an SM then reads 128 KB of operands instead of 256 KB; with the
// output written at the same time, the SM's memory interface is what bounds
// this kernel (halving the operand loads alone took it from 1393 to 1724
// TFLOP/s on 32768 rows).
//   warp 0      (both CTAs) TMA producer: the unit's A rows, then its own B
//               half 128x64 per stage; the loads of both CTAs complete on the
//               even CTA's barriers.
//   warp 1      (both CTAs) allocates 512 TMEM columns in the pair; in the
//               even CTA lane 0 issues the MMAs (M=256, N=256, K=16; 4 per
//               stage) into one of two 256-column f32 accumulators, and
//               commits stage, accumulator and A barriers to both CTAs.
//   warps 2-5   (both CTAs) epilogue of the CTA's own 128 rows: tcgen05.ld
//               32 lanes x 32 columns, round to fp16 (or bf16), a 32x64
//               staging tile in the 128-byte swizzle, written back by one
//               tensor store (TMA) per tile piece; the accumulator is handed
//               back on the even CTA's barrier with a relaxed arrive.
// Units are numbered segment-major, row block fastest, and dealt to the
// pairs round-robin: the pairs that run at the same time sweep the same
// weight tiles in step (read once from L2 for all of them, and kept there
// with an evict-last hint while the output streams past); this ordering ran
// 8% faster than giving concurrent pairs different segments.
#include <cstdio>

#include "sm103.cuh"

namespace mla {
namespace sm103 {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 5;
constexpr int MAX_K = 512;                    // A rows are resident: K <= 512
constexpr int PAIR_M = 2 * BM;                // rows of a pair tile
constexpr int A_BLOCK = BM * BK * 2;          // 16 KB: this CTA's A rows, one K block
constexpr int A_BYTES = (MAX_K / BK) * A_BLOCK;  // 128 KB: all of K
constexpr int B_BYTES = (BN / 2) * BK * 2;    // 16 KB: this CTA's half of B, one K block
constexpr int EPI_WARPS = 4;
constexpr int STG_BYTES = 32 * 64 * 2;        // one warp's 32x64 16-bit staging tile
constexpr int SMEM_BYTES = 1024 /*align slack*/ + A_BYTES + STAGES * B_BYTES +
                           EPI_WARPS * STG_BYTES + 256 /*barriers*/;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;

struct GemmArgs {
  int M, N, K;
  int num_pm, num_n;  // pair tiles along M, tiles along N
  int nseg;           // N segments per 256-row block: a unit is (block, segment)
  int hd;             // output columns per head (Dn + Dv): the output is [N/hd, M, hd]
                      // (written through the output tensor map)
  int32_t *status;    // nullable: MLA_STATUS_FP16_RANGE when an fp16 output overflowed
};

// Unit u: N tiles [t0, t1) of segment u / num_pm, row block u % num_pm.
__device__ __forceinline__ void unit_range(const GemmArgs &g, int u, int &pm, int &t0, int &t1) {
  const int sgm = u / g.num_pm;
  pm = u - sgm * g.num_pm;
  t0 = sgm * g.num_n / g.nseg;
  t1 = (sgm + 1) * g.num_n / g.nseg;
}

template <bool kF16Out>
__global__ void __launch_bounds__(THREADS, 1)
    up_proj_tc_kernel(const __grid_constant__ CUtensorMap tm_a,
                      const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_o, GemmArgs g) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + A_BYTES;
  uint8_t *sStage = sB + STAGES * B_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sStage + EPI_WARPS * STG_BYTES);
  // bars: full[S], empty[S], acc_full[2], acc_empty[2], a_full, a_empty,
  // mma_done; then the TMEM base address slot.  full, acc_empty and a_full
  // are used in the even CTA only.
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  const uint32_t accf0 = smem_u32(bars + 2 * STAGES), acce0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t a_full = smem_u32(bars + 2 * STAGES + 4);
  const uint32_t a_empty = smem_u32(bars + 2 * STAGES + 5);
  const uint32_t done_bar = smem_u32(bars + 2 * STAGES + 6);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 7);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: the CTA that issues the MMAs
  const int num_units = g.num_pm * g.nseg;
  const int first = blockIdx.x >> 1, step = gridDim.x >> 1;
  const int kblocks = g.K / BK;
  // the even CTA's barriers, as seen from this CTA
  const uint32_t full0_lead = mapa_shared(full0, 0);
  const uint32_t acce0_lead = mapa_shared(acce0, 0);
  const uint32_t a_full_lead = mapa_shared(a_full, 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf0 + 8 * a, 1);
      mbar_init(acce0 + 8 * a, 2 * EPI_WARPS);  // epilogue warps of both CTAs
    }
    mbar_init(a_full, 1);
    mbar_init(a_empty, 1);
    mbar_init(done_bar, 1);
    fence_mbar_init();
    prefetch_map(&tm_a);
    prefetch_map(&tm_b);
    prefetch_map(&tm_o);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any load or arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs)
    int stage = 0;
    uint32_t phase = 0;
    int issued_parity[STAGES];
    for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
    int a_issued = -1;  // parity of the last A load, -1: none
    const uint64_t pol_w = policy_evict_last();
    bool ok = true;
    int k = 0;          // units of this pair so far
    for (int u = first; u < num_units && ok; u += step, ++k) {
      int pm, t0, t1;
      unit_range(g, u, pm, t0, t1);
      const int m0 = pm * PAIR_M + int(rank) * BM;
      // the previous unit's MMAs are done with the resident A rows
      if (!mbar_wait(a_empty, uint32_t((k & 1) ^ 1))) break;
      if (rank == 0) mbar_expect_tx(a_full, uint32_t(2 * kblocks * A_BLOCK));  // both CTAs
      for (int kb = 0; kb < kblocks; ++kb)
        tma_load_2d_pair(smem_u32(sA + kb * A_BLOCK), &tm_a, a_full_lead, kb * BK, m0);
      a_issued = k & 1;
      for (int t = t0; t < t1 && ok; ++t) {
        const int nb = t * BN + int(rank) * (BN / 2);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_expect_tx(full0 + 8 * stage, 2 * B_BYTES);  // both CTAs' bytes
          tma_load_2d_pair_hint(smem_u32(sB + stage * B_BYTES), &tm_b, full0_lead + 8 * stage,
                                kb * BK, nb, pol_w);
          issued_parity[stage] = int(phase);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    // every load this CTA issued has landed before the pair may exit: the
    // even CTA's barriers count both CTAs' bytes; the odd CTA knows its loads
    // landed once the MMAs that read them released the buffer
    for (int s = 0; s < STAGES; ++s) {
      if (issued_parity[s] < 0) continue;
      if (rank == 0)
        mbar_wait(full0 + 8 * s, uint32_t(issued_parity[s]));
      else
        mbar_wait(empty0 + 8 * s, uint32_t(issued_parity[s]));
    }
    if (a_issued >= 0) {
      if (rank == 0)
        mbar_wait(a_full, uint32_t(a_issued));
      else
        mbar_wait(a_empty, uint32_t(a_issued));
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer (even CTA)
    constexpr uint32_t idesc = idesc_f16kind(PAIR_M, BN, false, false, true);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    int k = 0;
    for (int u = first; u < num_units && ok; u += step, ++k) {
      int pm, t0, t1;
      unit_range(g, u, pm, t0, t1);
      if (!mbar_wait(a_full, uint32_t(k & 1))) break;
      for (int t = t0; t < t1 && ok; ++t) {
        if (!mbar_wait(acce0 + 8 * acc, acc_phase ^ 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + kb * A_BLOCK);
          const uint32_t b_addr = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16_pair(d_tmem, desc_kmajor_sw128(a_addr + kk * 32),
                          desc_kmajor_sw128(b_addr + kk * 32), idesc, (kb | kk) != 0);
          // the B stage is free in both CTAs once these MMAs finish
          mma_commit_pair_mc(empty0 + 8 * stage, uint16_t(0x3));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_pair_mc(accf0 + 8 * acc, uint16_t(0x3));  // accumulator complete
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // the resident A rows are free in both CTAs once this unit's MMAs finish
      mma_commit_pair_mc(a_empty, uint16_t(0x3));
    }
    // every MMA this thread issued has completed before TMEM is released
    mma_commit_pair_mc(done_bar, uint16_t(0x1));
    mbar_wait(done_bar, 0);
  } else if (warp >= 2) {
    // ---------------- epilogue: TMEM -> 16-bit -> swizzled smem -> tensor stores
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const uint32_t stg = smem_u32(sStage + (warp - 2) * STG_BYTES);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    float amax = 0.f;  // largest magnitude rounded to fp16 (range check)
    for (int u = first; u < num_units && ok; u += step) {
      int pm, t0, t1;
      unit_range(g, u, pm, t0, t1);
      const int m0 = pm * PAIR_M + int(rank) * BM;
      for (int t = t0; t < t1; ++t) {
        const int n0 = t * BN;
        if (!mbar_wait(accf0 + 8 * acc, acc_phase)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_row = tmem_base + (uint32_t(quarter * 32) << 16) + uint32_t(acc * BN);
#pragma unroll 1
        for (int j = 0; j < BN / 64; ++j) {
          uint32_t lo[32], hi[32];
          tmem_ld32(t_row + j * 64, lo);
          tmem_ld32(t_row + j * 64 + 32, hi);
          tmem_wait_ld();
          if (kF16Out) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(lo[e])), fabsf(__uint_as_float(hi[e]))));
          }
          // the previous piece's tensor store has read the staging tile
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
          // lane = row: its 64 values as 8 16-byte pieces, XOR-swizzled (the
          // tensor store's 128-byte swizzle)
          const uint32_t row = stg + uint32_t(lane * 128);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t *src = (c < 4) ? lo + 8 * c : hi + 8 * (c - 4);
            uint4 v;
            if (kF16Out) {
              v.x = pack_f16(__uint_as_float(src[0]), __uint_as_float(src[1]));
              v.y = pack_f16(__uint_as_float(src[2]), __uint_as_float(src[3]));
              v.z = pack_f16(__uint_as_float(src[4]), __uint_as_float(src[5]));
              v.w = pack_f16(__uint_as_float(src[6]), __uint_as_float(src[7]));
            } else {
              v.x = pack_bf16(__uint_as_float(src[0]), __uint_as_float(src[1]));
              v.y = pack_bf16(__uint_as_float(src[2]), __uint_as_float(src[3]));
              v.z = pack_bf16(__uint_as_float(src[4]), __uint_as_float(src[5]));
              v.w = pack_bf16(__uint_as_float(src[6]), __uint_as_float(src[7]));
            }
            st_shared_v4(row + uint32_t((c ^ (lane & 7)) << 4), v);
          }
          // the staging tile is the 128-byte-swizzled layout of a 64-column x
          // 32-row box: one tensor store writes it (rows past M are clipped).
          // With the stores on the TMA engine the epilogue issues no global
          // stores and no shared-memory loads of its own: 673 -> 636 us on
          // 32768 rows against coalesced LSU stores from the same tile.
          fence_async_smem();
          __syncwarp();
          const int n = n0 + j * 64, head = n / g.hd, col = n % g.hd;
          if (lane == 0) {
            tma_store_3d(&tm_o, stg, col, m0 + quarter * 32, head);
            bulk_commit();
          }
        }
        // the accumulator is read (every tcgen05.ld waited for): hand it
        // back without waiting for this tile's output stores to drain -- a
        // release arrive waited for them, and the MMAs of the tile after next
        // waited on it (0.79 of the bf16 peak on 32768 rows; 0.86 without)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(acce0_lead + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // every tensor store has completed
    __syncwarp();
    // a finite accumulator of magnitude >= 65520 became +-inf in fp16
    if (kF16Out && g.status && amax >= kF16Overflow) atomicOr(g.status, MLA_STATUS_FP16_RANGE);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs or loads may touch it
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace
}  // namespace sm103

bool make_tmap_3d_16(CUtensorMap *map, bool fp16, const void *base, uint64_t dim0, uint64_t dim1,
                     uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                     uint32_t box1, bool swizzle128) {
  auto fn = sm103::encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {dim0, dim1, dim2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        3, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_2d_16(CUtensorMap *map, bool fp16, const void *base, uint64_t dim0, uint64_t dim1,
                     uint64_t row_stride_bytes, uint32_t box0, uint32_t box1, bool swizzle128) {
  auto fn = sm103::encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        2, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool tc_available() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return major == 10 && minor == 3 && sm103::encode_fn() != nullptr;
}

bool tc_gemm_ok(const mla_dims_t &d, int kv_dtype, int64_t lda, const void *latent,
                const void *w, const void *kv) {
  const int hd = d.qk_nope_dim + d.v_dim;
  const int N = d.num_heads * hd;
  auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  return d.dtype == MLA_DTYPE_BF16 && (kv_dtype == MLA_DTYPE_F16 || kv_dtype == MLA_DTYPE_BF16) &&
         d.kv_lora_rank % sm103::BK == 0 && d.kv_lora_rank <= sm103::MAX_K &&
         N % sm103::BN == 0 && hd % 64 == 0 &&
         (lda * 2) % 16 == 0 && al16(latent) && al16(w) && al16(kv);
}

int launch_up_proj_tc(const mla_dims_t &d, int kv_dtype, const void *latent, int64_t lda,
                      int rows, const void *w, void *kv, int32_t *status, cudaStream_t s) {
  using namespace sm103;
  const int K = d.kv_lora_rank;
  const int hd = d.qk_nope_dim + d.v_dim;
  const int N = d.num_heads * hd;
  CUtensorMap ta, tb;
  const bool f16 = kv_dtype == MLA_DTYPE_F16;
  CUtensorMap to;
  if (!make_tmap_2d_16(&ta, false, latent, K, rows, uint64_t(lda) * 2, BK, BM, true) ||
      !make_tmap_2d_16(&tb, false, w, K, N, uint64_t(K) * 2, BK, BN / 2, true) ||
      !make_tmap_3d_16(&to, f16, kv, hd, rows, N / hd, uint64_t(hd) * 2,
                       uint64_t(rows) * hd * 2, 64, 32, true))
    return MLA_ERR_CUDA;
  GemmArgs g{rows, N, K, (rows + PAIR_M - 1) / PAIR_M, N / BN, 1, hd, status};
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(up_proj_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(up_proj_tc_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return MLA_ERR_CUDA;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_clusters = 0;
  if (max_clusters == 0) {
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, up_proj_tc_kernel<true>, &cfg) != cudaSuccess ||
        n < 1)
      n = num_sms() / 2;
    max_clusters = n;
  }
  const int pairs = max_clusters;
  // N segments per row block: the fewest tile-times for the busiest pair,
  // counting a unit's A load as about one tile of B traffic
  long best = -1;
  for (int ns = 1; ns <= g.num_n; ++ns) {
    const long rounds = (long(g.num_pm) * ns + pairs - 1) / pairs;
    const long cost = rounds * ((g.num_n + ns - 1) / ns + 1);
    if (best < 0 || cost < best) {
      best = cost;
      g.nseg = ns;
    }
  }
  const int units = g.num_pm * g.nseg;
  const int clusters = units < pairs ? units : pairs;
  cfg.gridDim = dim3(2 * clusters);
  launch_begin(s);
  const cudaError_t e = f16 ? cudaLaunchKernelEx(&cfg, up_proj_tc_kernel<true>, ta, tb, to, g)
                            : cudaLaunchKernelEx(&cfg, up_proj_tc_kernel<false>, ta, tb, to, g);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  return launch_status(s, "up_proj_tc_kernel");
}

}  // namespace mla

namespace mla {
namespace {
// Waits on an mbarrier that nothing arrives on, with a short limit: the wait
// gives up, records the timeout bit and the kernel returns normally.
__global__ void bounded_wait_selftest_kernel(long long limit, int32_t *gave_up) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = sm103::smem_u32(&bar);
  sm103::mbar_init(b, 1);
  sm103::fence_mbar_init();
  *gave_up = sm103::mbar_wait_limit(b, 0, limit) ? 0 : 1;
}
}  // namespace

int gemm_take_errors() { return sm103::take_error_flags_here(); }

int launch_bounded_wait_selftest(long long limit_cycles, int32_t *gave_up, cudaStream_t s) {
  launch_begin(s);
  bounded_wait_selftest_kernel<<<1, 1, 0, s>>>(limit_cycles, gave_up);
  return launch_status(s, "bounded_wait_selftest_kernel");
}
}  // namespace mla
