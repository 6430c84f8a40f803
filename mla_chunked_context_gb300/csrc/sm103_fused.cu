// Context-chunk attention with the W_kv_b up-projection fused in (sm_103a):
// K_nope and V of every key tile are computed on chip from the gathered
// latent rows and consumed there, never written to HBM.
//
// What it computes is the context attention of a chunk (PR #50613 report,
// item 4: (O, LSE) per query row and head over the chunk's keys; item 3: a
// continued request's result LSE-merged into its stored partial), with the
// keys and values of the up-projection (DeepSeek-V3 MLA: W_kv_b [H*(Dn+Dv),
// L], K_nope = c_kv W_k^T, V = c_kv W_v^T per head):
//   s_j = scale * (q_nope . K_nope[j, h] + q_pe . k_pe[j]),
//   O = sum_j softmax(s)_j V[j, h],  LSE = ln sum_j exp(s_j).
// K_nope and V are rounded to fp16 once from the fp32 accumulator, as the
// unfused path stores them, so both paths compute the same numbers.
//
// A cluster of two CTAs (one per SM) works on one head at a time, each CTA
// holding half of the head's W_kv_b rows resident in tensor memory as the A
// operand of its up-projection (128 rows x 512 bf16 = 256 TMEM columns):
//   rank 0 (keys):   K^T tile = W_k (TMEM) x latent^T (the latent tile is the
//                    B operand, loaded by each CTA's own TMA producer),
//                    converted to fp16 in shared memory; S = Q K^T (M=128
//                    queries, N=128 keys, K=192) and the online softmax; P
//                    (fp16) and the rescale factor go to rank 1's shared
//                    memory with st.async.
//   rank 1 (values): V^T tile = W_v (TMEM) x latent^T, converted the same way;
//                    each tile's P V (M=128, N=128, K=128) into TMEM, summed
//                    into O in registers with rank 0's rescale factor; the
//                    epilogue.
// Per 128-key tile each SM does 40-44 MMAs of 128x128x16 and moves about
// 400 KB through shared memory, where the unfused path writes and re-reads
// 64 KB of K/V per key and head through HBM.
//
// Units: a sequence of at most 128 queries (one query tile), a head, and a
// range of its 128-key tiles.  The (head, sequence, key tile) space is cut
// into one contiguous range per cluster; a (head, sequence) cut between
// clusters writes each piece to a key-split scratch slot, merged afterwards
// by the attention's split-combine kernel.
//
// Warps of each CTA (512 threads):
//   0  TMA producer: the latent ring (both ranks), k_pe and Q (rank 0).
//      Each CTA loads the latent itself into its own ring; the second
//      read of a tile comes from L2 (27% busy with it).  A ring shared by
//      the two SMs would make each refill wait for both SMs' MMAs and hold
//      them in lock step.
//   1  TMEM owner; issues each key tile's up-projection MMAs
//   2  issues the tile's second MMA group (S on rank 0, P.V on rank 1);
//      rank 1's P.V commit also arrives on rank 0's barrier (a P buffer
//      free again)
//   4-7  W rows into TMEM at each head change; accumulator -> fp16 staging
//   8-15 rank 0: softmax (a thread per query row and half tile); rank 1: O
//        in registers (a thread per query row and half of the columns),
//        rescaled and summed over the tiles' P.V results, and the epilogue
// TMEM: W half [0,256), buffers [256,384) [384,512).  Buffer b = J mod 2
// holds key tile J's up-projection accumulator until the convert warps
// have loaded it, then the tile's second result (rank 0: S, rank 1: its P.V),
// until the softmax / O warps have loaded that: the next tile's
// up-projection never waits for the previous one's conversion.
// Every wait is bounded (a timeout sets the error word and the roles wind
// down); both CTAs meet at a cluster barrier before either leaves.
#include <algorithm>
#include <vector>

#include "sm103.cuh"

namespace mla {

struct FusedPlan {
  int tph = 0, P = 0;          // key tiles per head, clusters
  std::vector<int4> items;     // (sequence, key tiles, first tile, (slot base + 1) | pieces << 16)
  std::vector<int> bounds;     // P + 1 range ends
  std::vector<int4> groups;    // split-combine groups (sequence, 0, first slot, slots)
};

int launch_split_combine(int n_groups, const int4 *groups, int H, int T, const int32_t *q_loc,
                         const int32_t *acc, const SplitScratch &split, float *o, float *lse,
                         cudaStream_t s);

namespace {

using namespace sm103;

constexpr int BQ = 128, BKV = 128;
constexpr int LR = 512, DN = 128, DR = 64, DV = 128, DQK = DN + DR, HD = DN + DV;
constexpr int KBLK = LR / 64;          // latent K-blocks of 64 per key tile
constexpr int RING = 5;                 // latent stages in flight
constexpr int NKPE = 1;                 // k_pe buffers
constexpr int STAGE = BKV * 64 * 2;     // 16 KB: 128 keys x 64 latent columns
constexpr int QBOX = BQ * 64 * 2;       // 16 KB
constexpr int HALF_OP = 128 * 64 * 2;   // one 64-wide block of a 128-row operand
constexpr int OPND = 2 * HALF_OP;       // 32 KB: a 128 x 128 16-bit operand
constexpr int P_BYTES = OPND + BQ * 4;  // a tile's P and alpha, sent by rank 0
// shared memory, offsets from the 1024-aligned base, the same in both CTAs
constexpr int OFF_RING = 0;                           // RING stages (both)
constexpr int OFF_A = OFF_RING + RING * STAGE;
constexpr int OFF_Q = OFF_A;                          // rank 0: Q, 3 boxes
constexpr int OFF_KPE = OFF_A + 3 * QBOX;             // rank 0: k_pe [NKPE]
constexpr int OFF_P = OFF_A;                          // rank 1: P [2]
constexpr int OFF_STG = OFF_A + (3 * QBOX + NKPE * STAGE > 2 * OPND ? 3 * QBOX + NKPE * STAGE
                                                                    : 2 * OPND);
                                                      // K^T (rank 0) / V^T (rank 1) [2]
constexpr int OFF_ALPHA = OFF_STG + 2 * OPND;         // rank 1: alpha [2][BQ]
constexpr int OFF_STATS = OFF_ALPHA + 2 * BQ * 4;     // rank 1: [2 units][m, l][BQ]
constexpr int OFF_BARS = OFF_STATS + 4 * BQ * 4;
constexpr int NBARS = 64;
constexpr int SMEM_BYTES = 1024 + OFF_BARS + NBARS * 8 + 16;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
constexpr int THREADS = 512;
constexpr uint32_t TMEM_COLS = 512, COL_W = 0, COL_BUF = 256;  // buffer b at COL_BUF + 128 b
constexpr int MAX_PAIRS = 128;
constexpr int MAX_ITEMS = 1024;
constexpr float kRescaleThreshold = 8.0f;  // log2 of the tolerated growth of the running max

// mbarrier indices.  TMEM buffer b (of 2) holds a key tile's up-projection
// accumulator, then that tile's second result (rank 0: S, rank 1: its P.V).
enum : int {
  B_FULL = 0,                // [RING] latent stage landed
  B_EMPTY = B_FULL + RING,   // [RING] latent stage used by this CTA's MMAs
  B_ACCF = B_EMPTY + RING,   // [2] the up-projection in buffer b is complete
  B_STGR = B_ACCF + 2,       // [2] accumulator loaded and fp16 staging written (4 warps)
  B_STGF = B_STGR + 2,       // [2] staging read by the tile's second MMA group
  B_RESF = B_STGF + 2,       // [2] the tile's second result (S / P.V) is complete
  B_RESR = B_RESF + 2,       // [2] ... and loaded (rank 0: softmax, rank 1: O warps; 8 warps)
  B_KPEF = B_RESR + 2,       // [NKPE] rank 0: k_pe landed
  B_KPEE = B_KPEF + NKPE,    // [NKPE] rank 0: k_pe used
  B_QF = B_KPEE + NKPE,      // rank 0: Q landed
  B_QE,                      // rank 0: Q used by the unit's last S
  B_W,                       // W rows in TMEM (4 warps)
  B_PFREE,                   // [2] rank 0: P buffer free: rank 1's P.V commit + its 8 O warps
  B_PFULL = B_PFREE + 2,     // [2] rank 1: P and alpha of a tile landed (rank 0's st.async bytes)
  B_STATS = B_PFULL + 2,     // [2] rank 1: a unit's (m, l) written by rank 0 (4 warps)
  B_DONE = B_STATS + 2,      // the up-projection issuer's MMAs are complete
  B_DONE2,                   // the second issuer's MMAs are complete
  B_COUNT
};
static_assert(B_COUNT <= NBARS, "barrier slots");

struct FusedParams {
  int n_items, H, T, npairs, tiles_per_head;
  float scale_log2;
  const int32_t *q_loc, *k_loc, *acc;
  const uint16_t *w;                 // W_kv_b [H*(Dn+Dv)][L] bf16
  float *o, *lse, *split_o, *split_lse;
  int32_t *status;                   // nullable: MLA_STATUS_FP16_RANGE on a K/V overflow
  int bounds[MAX_PAIRS + 1];         // cluster c: flattened key tiles [bounds[c], bounds[c+1])
  // (sequence, key tiles, first tile in a head's order, (slot base + 1) | max pieces << 16)
  int4 items[MAX_ITEMS];
};

// One unit of a cluster: head h, the sequence of item i, its key tiles
// [kt0, kt1); slot >= 0: a piece of a split (h, sequence), whose last piece
// also sets LSE = -inf in the slots [slot + 1, clear_to) no piece of this
// head uses.
struct Unit {
  int h, seq, kt0, kt1, slot, clear_to;
};

constexpr int MAX_SPLIT_GROUPS = 16;  // groups one split-combine launch takes

__host__ __device__ inline int pair_of(const int *bounds, int npairs, int x) {
  int lo = 0, hi = npairs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (bounds[mid] <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ bool next_unit(const FusedParams &p, int pair, int &f, Unit &u) {
  const int f1 = p.bounds[pair + 1];
  if (f >= f1) return false;
  const int h = f / p.tiles_per_head, r = f - h * p.tiles_per_head;
  int lo = 0, hi = p.n_items - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.items[mid].z <= r)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int4 it = p.items[lo];
  u.h = h;
  u.seq = it.x;
  u.kt0 = r - it.z;
  u.kt1 = min(it.y, u.kt0 + (f1 - f));
  const int sb = (it.w & 0xffff) - 1, maxp = it.w >> 16;
  if (sb < 0) {
    u.slot = -1;
    u.clear_to = 0;
  } else {
    u.slot = sb + pair - pair_of(p.bounds, p.npairs, h * p.tiles_per_head + it.z);
    u.clear_to = u.kt1 == it.y ? sb + maxp : 0;
  }
  f += u.kt1 - u.kt0;
  return true;
}

// D (+)= A (TMEM) x B (shared-memory descriptor)^T, kind::f16.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Wait with cluster-scope acquire: for phases completed by arrivals of the
// other CTA, whose shared-memory writes this thread then reads.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
  auto try_once = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
  };
  if (try_once()) return true;
  const long long t0 = clock64();
  while (!try_once()) {
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(&g_error_flags, kErrWaitTimeout);
      return false;
    }
  }
  return true;
}

// Asynchronous stores into a cluster peer's shared memory, each counting its
// bytes on the peer's mbarrier at `rbar` (complete_tx): no fence and no
// arrival by the writer.
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                            uint32_t d, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          addr),
      "r"(a), "r"(b), "r"(c), "r"(d), "r"(rbar)
      : "memory");
}
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
               "r"(__float_as_uint(v)), "r"(rbar)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Named barrier `id` over 8 warps (256 threads): AND of pred.
__device__ __forceinline__ bool named_bar_and(int id, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %1, 0;\n bar.red.and.pred q, %2, 256, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(pred ? 1 : 0), "r"(id)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of 16-byte chunk c (0..15: columns 8c..8c+7) of row r in a
// 128-row operand of two 64-column blocks, 128-byte swizzle.
__device__ __forceinline__ uint32_t opnd_off(int r, int c) {
  return uint32_t((c >> 3) * HALF_OP + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(THREADS, 1)
    attn_fused_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_lat,
                      const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + OFF_BARS;
  auto bar = [&](int k) { return bar0 + 8u * uint32_t(k); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_BARS + NBARS * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int f_begin = p.bounds[pair];

  // key tiles of this cluster (both CTAs walk the same units)
  int total_tiles = 0;
  {
    int f = f_begin;
    Unit u;
    while (next_unit(p, pair, f, u)) total_tiles += u.kt1 - u.kt0;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < RING; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_ACCF + b), 1);
      mbar_init(bar(B_STGR + b), 4);
      mbar_init(bar(B_STGF + b), 1);
      mbar_init(bar(B_RESF + b), 1);
      mbar_init(bar(B_RESR + b), 8);
      mbar_init(bar(B_PFREE + b), 9);
      mbar_init(bar(B_PFULL + b), 1);
      mbar_init(bar(B_STATS + b), 4);
    }
    for (int b = 0; b < NKPE; ++b) {
      mbar_init(bar(B_KPEF + b), 1);
      mbar_init(bar(B_KPEE + b), 1);
    }
    mbar_init(bar(B_QF), 1);
    mbar_init(bar(B_QE), 1);
    mbar_init(bar(B_W), 4);
    mbar_init(bar(B_DONE), 1);
    mbar_init(bar(B_DONE2), 1);
    fence_mbar_init();
    if (rank == 0) {
      prefetch_map(&tm_q);
      prefetch_map(&tm_lat);
    } else {
      // rank 1's P buffers expect their first tile's P and alpha
      for (int b = 0; b < 2 && b < total_tiles; ++b) mbar_expect_tx(bar(B_PFULL + b), P_BYTES);
    }
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any load or remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    {
      // ---------------- TMA producer
      int f = f_begin, J = 0, nu = 0;
      Unit u;
      bool ok = true;
      int last_use[RING], kpe_par[NKPE], q_par = -1;
      for (int b = 0; b < NKPE; ++b) kpe_par[b] = -1;
      for (int s = 0; s < RING; ++s) last_use[s] = -1;
      while (ok && next_unit(p, pair, f, u)) {
        const int k_beg = __ldg(p.k_loc + u.seq), q_beg = __ldg(p.q_loc + u.seq);
        for (int j = u.kt0; ok && j < u.kt1; ++j, ++J) {
          const int row = k_beg + j * BKV;
          for (int kb = 0; kb < KBLK; ++kb) {
            const int g = J * KBLK + kb, s = g % RING, n = g / RING;
            if (n > 0 && !mbar_wait(bar(B_EMPTY + s), uint32_t((n - 1) & 1))) {
              ok = false;
              break;
            }
            mbar_expect_tx(bar(B_FULL + s), STAGE);
            tma_load_2d(sbase + OFF_RING + s * STAGE, &tm_lat, bar(B_FULL + s), kb * 64, row);
            last_use[s] = n;
          }
          if (!ok) break;
          if (rank == 1) continue;
          const int b = J % NKPE;
          if (J >= NKPE && !mbar_wait(bar(B_KPEE + b), uint32_t((J / NKPE - 1) & 1))) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar(B_KPEF + b), STAGE);
          tma_load_2d(sbase + OFF_KPE + b * STAGE, &tm_lat, bar(B_KPEF + b), LR, row);
          kpe_par[b] = (J / NKPE) & 1;
          if (j == u.kt0) {
            // the unit's queries, once the previous unit's last S is done
            // with the buffer (after this tile's loads: the up-projection
            // needs no Q)
            if (nu > 0 && !mbar_wait(bar(B_QE), uint32_t((nu - 1) & 1))) {
              ok = false;
              break;
            }
            mbar_expect_tx(bar(B_QF), 3 * QBOX);
            const int qy = u.h * p.T + q_beg;
            for (int i = 0; i < 3; ++i)
              tma_load_2d(sbase + OFF_Q + i * QBOX, &tm_q, bar(B_QF), i * 64, qy);
            q_par = nu & 1;
            ++nu;
          }
        }
      }
      // every load has landed before the CTA may leave
      for (int s = 0; s < RING; ++s)
        if (last_use[s] >= 0) {
          mbar_wait(bar(B_FULL + s), uint32_t(last_use[s] & 1));
          mbar_wait(bar(B_EMPTY + s), uint32_t(last_use[s] & 1));
        }
      for (int b = 0; b < NKPE; ++b)
        if (kpe_par[b] >= 0) mbar_wait(bar(B_KPEF + b), uint32_t(kpe_par[b]));
      if (q_par >= 0) mbar_wait(bar(B_QF), uint32_t(q_par));
    }
  } else if ((warp == 1 || warp == 2) && lane == 0) {
    // ---------------- MMA issuers: warp 1 the up-projection of each key tile,
    // warp 2 the tile's second group (S on rank 0, P.V on rank 1) as soon as
    // its operands are staged, so that neither waits behind the other
    constexpr uint32_t ID_G = idesc_f16kind(128, BKV, false, false, true);   // W x latent, bf16
    constexpr uint32_t ID_SN = idesc_f16kind(BQ, BKV, false, true, false);   // q_nope x K^T, fp16
    constexpr uint32_t ID_SR = idesc_f16kind(BQ, BKV, false, false, true);   // q_pe x k_pe, bf16
    constexpr uint32_t ID_PV = idesc_f16kind(BQ, DV, false, false, false);   // P x V^T, fp16
    const uint32_t q_addr = sbase + OFF_Q;
    int f = f_begin, J = 0, nu = 0, prev_h = -1, wl = 0;
    Unit u;
    bool ok = true;
    if (warp == 1) {
      while (ok && next_unit(p, pair, f, u)) {
        if (u.h != prev_h) {
          if (!mbar_wait(bar(B_W), uint32_t(wl & 1))) {
            ok = false;
            break;
          }
          ++wl;
          prev_h = u.h;
        }
        for (int j = u.kt0; ok && j < u.kt1; ++j, ++J) {
          const int b = J & 1;
          // buffer b is free once tile J-2's second result has been loaded
          if (J >= 2 && !mbar_wait(bar(B_RESR + b), uint32_t(((J - 2) >> 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + COL_BUF + uint32_t(b * 128);
          for (int kb = 0; kb < KBLK; ++kb) {
            const int g = J * KBLK + kb, s = g % RING, n = g / RING;
            if (!mbar_wait(bar(B_FULL + s), uint32_t(n & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t st = sbase + OFF_RING + uint32_t(s * STAGE);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ts(d, tmem + COL_W + uint32_t(kb * 32 + k * 8),
                     desc_kmajor_sw128(st + uint32_t(k * 32)), ID_G, (kb | k) != 0);
            mma_commit(bar(B_EMPTY + s));
          }
          if (!ok) break;
          mma_commit(bar(B_ACCF + b));
        }
      }
    } else {
      while (ok && next_unit(p, pair, f, u)) {
        const int nt = u.kt1 - u.kt0;
        for (int j = 0; ok && j < nt; ++j, ++J) {
          const int b = J & 1;
          const uint32_t par = uint32_t((J >> 1) & 1);
          const uint32_t d = tmem + COL_BUF + uint32_t(b * 128);
          // the staging is written and the accumulator in buffer b loaded
          if (!mbar_wait(bar(B_STGR + b), par)) {
            ok = false;
            break;
          }
          if (rank == 0) {
            const int kb = J % NKPE;
            if (!mbar_wait(bar(B_KPEF + kb), uint32_t((J / NKPE) & 1)) ||
                (j == 0 && !mbar_wait(bar(B_QF), uint32_t(nu & 1)))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t kt = sbase + OFF_STG + uint32_t(b * OPND);
            const uint32_t kp = sbase + OFF_KPE + uint32_t(kb * STAGE);
#pragma unroll
            for (int kk = 0; kk < DN / 16; ++kk)
              mma_bf16(d, desc_kmajor_sw128(q_addr + uint32_t((kk >> 2) * QBOX + (kk & 3) * 32)),
                       desc_mnmajor_sw128(kt + uint32_t(kk * 2048), HALF_OP), ID_SN, kk != 0);
#pragma unroll
            for (int kk = 0; kk < DR / 16; ++kk)
              mma_bf16(d, desc_kmajor_sw128(q_addr + uint32_t(2 * QBOX + kk * 32)),
                       desc_kmajor_sw128(kp + uint32_t(kk * 32)), ID_SR, 1u);
            mma_commit(bar(B_RESF + b));
            mma_commit(bar(B_STGF + b));
            mma_commit(bar(B_KPEE + kb));
            if (j == nt - 1) mma_commit(bar(B_QE));
          } else {
            // P and alpha of the tile, written by rank 0
            if (!mbar_wait_cluster(bar(B_PFULL + b), par)) {
              ok = false;
              break;
            }
            // the buffer's next phase expects tile J+2's bytes (rank 0 sends
            // them only after this tile's P.V and the O warps are done)
            if (J + 2 < total_tiles) mbar_expect_tx(bar(B_PFULL + b), P_BYTES);
            fence_async_smem();
            tc_fence_after();
            const uint32_t pa = sbase + OFF_P + uint32_t(b * OPND);
            const uint32_t vb = sbase + OFF_STG + uint32_t(b * OPND);
#pragma unroll
            for (int kk = 0; kk < BKV / 16; ++kk) {
              const uint32_t off = uint32_t((kk >> 2) * HALF_OP + (kk & 3) * 32);
              mma_bf16(d, desc_kmajor_sw128(pa + off), desc_kmajor_sw128(vb + off), ID_PV,
                       kk != 0);
            }
            mma_commit(bar(B_RESF + b));
            mma_commit(bar(B_STGF + b));
            mma_commit_mc(bar(B_PFREE + b), 0x1);  // rank 0's barrier
          }
        }
        ++nu;
      }
    }
    const uint32_t done = bar(warp == 1 ? B_DONE : B_DONE2);
    mma_commit(done);
    mbar_wait(done, 0);
  } else if (warp >= 4 && warp < 8) {
    // ---------------- W rows into TMEM; accumulator -> fp16 operand staging
    const int quarter = warp & 3, d = quarter * 32 + lane;  // W row / TMEM lane
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    int f = f_begin, J = 0, prev_h = -1;
    Unit u;
    bool ok = true;
    while (ok && next_unit(p, pair, f, u)) {
      if (u.h != prev_h) {
        // the previous head's up-projections are complete: this warp has
        // converted their last result
        const uint4 *wr = reinterpret_cast<const uint4 *>(
            p.w + (int64_t(u.h) * HD + int64_t(rank) * DN + d) * LR);
#pragma unroll 1
        for (int c = 0; c < LR / 64; ++c) {
          uint32_t r[32];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint4 v = __ldg(wr + c * 8 + e);
            r[4 * e] = v.x;
            r[4 * e + 1] = v.y;
            r[4 * e + 2] = v.z;
            r[4 * e + 3] = v.w;
          }
          tmem_st32(tmem + lane_off + COL_W + uint32_t(c * 32), r);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_W));
        prev_h = u.h;
      }
      for (int j = u.kt0; ok && j < u.kt1; ++j, ++J) {
        const int b = J & 1;
        if (!mbar_wait(bar(B_ACCF + b), uint32_t((J >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t src = tmem + lane_off + COL_BUF + uint32_t(b * 128);
        uint32_t pk[64];
        float amax = 0.f;  // fp16 range check of this row's K or V values
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(src + uint32_t(c * 32), r);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float x0 = __uint_as_float(r[2 * e]), x1 = __uint_as_float(r[2 * e + 1]);
            amax = fmaxf(amax, fmaxf(fabsf(x0), fabsf(x1)));
            pk[c * 16 + e] = pack_f16(x0, x1);
          }
        }
        if (p.status && amax >= kF16Overflow) atomicOr(p.status, MLA_STATUS_FP16_RANGE);
        if (J >= 2 && !mbar_wait(bar(B_STGF + b), uint32_t(((J - 2) >> 1) & 1))) {
          ok = false;
          break;
        }
        uint8_t *stg = smem + OFF_STG + b * OPND;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          *reinterpret_cast<uint4 *>(stg + opnd_off(d, c)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        fence_async_smem();
        tc_fence_before();  // the tile's second MMA group overwrites the accumulator after this
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_STGR + b));
      }
    }
  } else if (warp >= 8 && rank == 0) {
    // ---------------- softmax: two warps per TMEM sub-partition, a thread per
    // query row and half tile (keys hw*64 .. hw*64+63).  The halves of a row
    // agree on its running max through shared memory at a named barrier
    // (an AND of the warps' status, so that all leave together after a wait
    // gave up), then each writes its half of P and keeps its half of the sum.
    const int quarter = warp & 3, row = quarter * 32 + lane, hw = (warp - 8) >> 2;
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const uint32_t p_rem = mapa_shared(sbase + OFF_P, 1);
    const uint32_t alpha_rem = mapa_shared(sbase + OFF_ALPHA, 1);
    const uint32_t stats_rem = mapa_shared(sbase + OFF_STATS, 1);
    const uint32_t pfull_rem = mapa_shared(bar(B_PFULL), 1);
    const uint32_t statsb_rem = mapa_shared(bar(B_STATS), 1);
    // exchange buffers (this CTA's copy of the alpha/stats area is unused):
    // xmax [2 tiles][2 halves][BQ], xl [2 halves][BQ]
    float *xmax = reinterpret_cast<float *>(smem + OFF_ALPHA);
    float *xl = xmax + 4 * BQ;
    int f = f_begin, J = 0, ui = 0;
    Unit u;
    bool ok = true;
    while (next_unit(p, pair, f, u)) {
      const int nk = __ldg(p.k_loc + u.seq + 1) - __ldg(p.k_loc + u.seq);
      float m_used = neg_inf(), l = 0.f;
      bool all = true;
      for (int j = u.kt0; j < u.kt1; ++j, ++J) {
        const int b = J & 1;
        if (ok) ok = mbar_wait(bar(B_RESF + b), uint32_t((J >> 1) & 1));
        tc_fence_after();
        float sv[64];
        if (ok) {
          uint32_t r0[32], r1[32];
          const uint32_t s_col = tmem + lane_off + COL_BUF + uint32_t(b * 128 + hw * 64);
          tmem_ld32(s_col, r0);
          tmem_ld32(s_col + 32u, r1);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            sv[e] = __uint_as_float(r0[e]);
            sv[32 + e] = __uint_as_float(r1[e]);
          }
        }
        // S is loaded: the buffer may take the tile after next
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_RESR + b));
        const int valid = nk - j * BKV - hw * 64;  // keys of the sequence in this half
        float t[32];
#pragma unroll
        for (int e = 0; e < 32; ++e)
          t[e] = fmaxf(e < valid ? sv[e] : neg_inf(), e + 32 < valid ? sv[e + 32] : neg_inf());
#pragma unroll
        for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
          for (int e = 0; e < w; ++e) t[e] = fmaxf(t[e], t[e + w]);
        xmax[(b * 2 + hw) * BQ + row] = t[0];
        all = named_bar_and(1, ok);
        if (!all) break;
        const float mx = fmaxf(t[0], xmax[(b * 2 + (hw ^ 1)) * BQ + row]) * p.scale_log2;
        float alpha = 1.f;
        if (mx > m_used + kRescaleThreshold || m_used == neg_inf()) {
          const float m_new = fmaxf(mx, m_used);
          if (m_used != neg_inf() && m_new != neg_inf()) alpha = exp2f(m_used - m_new);
          m_used = m_new;
        }
        const float nbase = (m_used == neg_inf()) ? 0.f : -m_used;
        l *= alpha;
        if (J >= 2) ok = mbar_wait(bar(B_PFREE + b), uint32_t(((J - 2) >> 1) & 1));
        if (!ok) continue;  // the next barrier takes every warp out
        const uint32_t pb = p_rem + uint32_t(b * OPND);
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k0 = c * 8 + 2 * e;
            const float x0 = k0 < valid ? ex2_approx(fmaf(sv[k0], p.scale_log2, nbase)) : 0.f;
            const float x1 =
                k0 + 1 < valid ? ex2_approx(fmaf(sv[k0 + 1], p.scale_log2, nbase)) : 0.f;
            ls[e] += x0 + x1;
            pk[e] = pack_f16(x0, x1);
          }
          st_async_v4(pb + opnd_off(row, hw * 8 + c), pk[0], pk[1], pk[2], pk[3],
                      pfull_rem + 8u * uint32_t(b));
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        if (hw == 0)
          st_async_f32(alpha_rem + uint32_t((b * BQ + row) * 4), alpha, pfull_rem + 8u * uint32_t(b));
      }
      if (!all) break;
      // the unit's (m, l) per row: the halves' sums share the running max
      xl[hw * BQ + row] = l;
      if (!named_bar_and(1, ok)) break;
      if (hw == 0) {
        st_cluster_f32(stats_rem + uint32_t(((ui & 1) * 2 * BQ + row) * 4), m_used);
        st_cluster_f32(stats_rem + uint32_t(((ui & 1) * 2 * BQ + BQ + row) * 4),
                       l + xl[BQ + row]);
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(statsb_rem + 8u * uint32_t(ui & 1));
      }
      ++ui;
    }
    // rank 1's last arrivals on the P buffers land here: wait for them
    for (int Jx = (J >= 2 ? J - 2 : 0); ok && Jx < J; ++Jx)
      ok = mbar_wait(bar(B_PFREE + (Jx & 1)), uint32_t((Jx >> 1) & 1));
  } else if (warp >= 8) {
    // ---------------- rank 1: O accumulated in registers, a thread per query
    // row and half of the 128 output columns: O = alpha O + (this tile's
    // P.V), then the unit epilogue
    const int quarter = warp & 3, row = quarter * 32 + lane, hw = (warp - 8) >> 2;
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const uint32_t pfree_rem = mapa_shared(bar(B_PFREE), 0);
    const float *alpha_s = reinterpret_cast<const float *>(smem + OFF_ALPHA);
    const float *stats_s = reinterpret_cast<const float *>(smem + OFF_STATS);
    int f = f_begin, J = 0, ui = 0;
    Unit u;
    bool ok = true;
    // after a wait gave up, the remaining waits are skipped and the named
    // barrier of the epilogue (an AND of the warps' status) takes all out
    while (next_unit(p, pair, f, u)) {
      float o[64];
#pragma unroll
      for (int e = 0; e < 64; ++e) o[e] = 0.f;
      for (int j = u.kt0; j < u.kt1; ++j, ++J) {
        const int b = J & 1;
        const uint32_t par = uint32_t((J >> 1) & 1);
        if (ok) ok = mbar_wait_cluster(bar(B_PFULL + b), par);
        const float alpha = ok ? alpha_s[b * BQ + row] : 1.f;
        __syncwarp();  // the warp's rows have read alpha: the P buffer may be rewritten
        if (ok && lane == 0) mbar_arrive_cluster(pfree_rem + 8u * uint32_t(b));
        if (ok) ok = mbar_wait(bar(B_RESF + b), par);
        tc_fence_after();
        if (ok) {
          const uint32_t src = tmem + lane_off + COL_BUF + uint32_t(b * 128 + hw * 64);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t r[32];
            tmem_ld32(src + uint32_t(c * 32), r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e)
              o[c * 32 + e] = fmaf(o[c * 32 + e], alpha, __uint_as_float(r[e]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(bar(B_RESR + b));
      }
      // ---- epilogue of the unit
      if (ok) ok = mbar_wait_cluster(bar(B_STATS + (ui & 1)), uint32_t((ui >> 1) & 1));
      const float m = stats_s[(ui & 1) * 2 * BQ + row];
      const float lsum = stats_s[(ui & 1) * 2 * BQ + BQ + row];
      const int q_beg = __ldg(p.q_loc + u.seq), nq = __ldg(p.q_loc + u.seq + 1) - q_beg;
      const int t = q_beg + row;
      float lse = (lsum > 0.f) ? (m + __log2f(lsum)) * 0.69314718055994531f : neg_inf();
      float w_new = (lsum > 0.f) ? 1.f / lsum : 0.f, w_old = 0.f;
      bool write = row < nq;
      float *orow, *lse_dst;
      if (u.slot >= 0) {
        const int64_t r = (int64_t(u.slot) * p.H + u.h) * BQ + row;
        orow = p.split_o + r * DV;
        lse_dst = p.split_lse + r;
      } else {
        orow = p.o + (int64_t(t) * p.H + u.h) * DV;
        lse_dst = p.lse + int64_t(u.h) * p.T + t;
        if (write && p.acc != nullptr && __ldg(p.acc + u.seq) != 0) {
          const float old = *lse_dst;
          if (lsum == 0.f) {
            write = false;  // nothing new: keep the stored partial
          } else if (!is_neg_inf(old)) {
            const float m2 = fmaxf(old, lse);
            const float eo = expf(old - m2), en = expf(lse - m2);
            w_old = eo / (eo + en);
            w_new *= en / (eo + en);
            lse = m2 + logf(eo + en);
          }
        }
      }
      // both halves have read the stored LSE before the first writes it
      if (!named_bar_and(2, ok)) break;
      if (write) {
        float4 *dst = reinterpret_cast<float4 *>(orow + hw * 64);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float4 v = make_float4(o[4 * e] * w_new, o[4 * e + 1] * w_new, o[4 * e + 2] * w_new,
                                 o[4 * e + 3] * w_new);
          if (w_old != 0.f) {
            const float4 ov = dst[e];
            v.x += w_old * ov.x;
            v.y += w_old * ov.y;
            v.z += w_old * ov.z;
            v.w += w_old * ov.w;
          }
          dst[e] = v;
        }
        if (hw == 0) *lse_dst = lse;
      }
      if (hw == 0 && row < nq)
        for (int s2 = u.slot + 1; s2 < u.clear_to; ++s2)
          p.split_lse[(int64_t(s2) * p.H + u.h) * BQ + row] = neg_inf();
      ++ui;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the other may still write to it
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

bool fused_attn_ok(const mla_dims_t &d, int64_t latent_ld) {
  return d.dtype == MLA_DTYPE_BF16 && d.qk_nope_dim == DN && d.qk_rope_dim == DR &&
         d.v_dim == DV && d.kv_lora_rank == LR && (latent_ld * 2) % 16 == 0 && latent_ld >= 576;
}

// Whether the fused kernel takes these sequences: at most 128 queries each
// (one query tile: a second would repeat the up-projection), at most
// MAX_ITEMS with keys, and on average at least `min_tiles` key tiles each
// (each unit pays a queries load and a pipeline refill).
bool fused_attn_fits(int num_seqs, const int32_t *q_loc_host, const int32_t *k_loc_host,
                     int min_tiles) {
  int items = 0;
  int64_t tiles = 0;
  for (int i = 0; i < num_seqs; ++i) {
    const int nq = q_loc_host[i + 1] - q_loc_host[i], nk = k_loc_host[i + 1] - k_loc_host[i];
    if (nq <= 0 || nk <= 0) continue;
    if (nq > BQ) return false;
    ++items;
    tiles += (nk + BKV - 1) / BKV;
  }
  return items > 0 && items <= MAX_ITEMS && tiles >= int64_t(min_tiles) * items;
}

// The fused kernel's work split (host only): the sequences with queries
// and keys become items (sequence, key tiles, first tile in a head's order,
// slot info); cluster c takes the flattened (head, item, key tile) range
// [bounds[c], bounds[c+1]) of equal shares; a (head, item) unit cut between
// clusters writes each piece to a key-split scratch slot (the item gets as
// many slots as the most pieces of any head), merged by the split-combine
// groups.  When the cut items need more than `split_slots` slots or 16
// groups, the ranges end on unit boundaries instead (the unit start nearest
// each equal share) and nothing is cut.
int plan_fused(int H, int num_seqs, const int32_t *q_loc_host, const int32_t *k_loc_host,
               int clusters, int split_slots, FusedPlan &plan) {
  plan = FusedPlan{};
  struct It { int seq, tiles, tbase; };
  std::vector<It> items;
  int tph = 0;
  for (int i = 0; i < num_seqs; ++i) {
    const int nq = q_loc_host[i + 1] - q_loc_host[i], nk = k_loc_host[i + 1] - k_loc_host[i];
    if (nq <= 0 || nk <= 0) continue;  // no queries, or rows that keep O=0, LSE=-inf
    if (nq > BQ) return MLA_ERR_UNSUPPORTED;
    const int tiles = (nk + BKV - 1) / BKV;
    items.push_back({i, tiles, tph});
    tph += tiles;
  }
  if (items.empty()) return MLA_OK;
  if (int(items.size()) > MAX_ITEMS || clusters < 1) return MLA_ERR_UNSUPPORTED;
  const int64_t N = int64_t(H) * tph;
  if (N > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  const int P = int(std::min<int64_t>(std::min(clusters, MAX_PAIRS), N));
  plan.tph = tph;
  plan.P = P;
  plan.bounds.resize(P + 1);
  for (int c = 0; c <= P; ++c) plan.bounds[c] = int(int64_t(c) * N / P);
  auto pieces = [&](std::vector<int> &maxp) {
    maxp.assign(items.size(), 1);
    for (int h = 0; h < H; ++h)
      for (size_t i = 0; i < items.size(); ++i) {
        const int x0 = h * tph + items[i].tbase, x1 = x0 + items[i].tiles - 1;
        const int k =
            pair_of(plan.bounds.data(), P, x1) - pair_of(plan.bounds.data(), P, x0) + 1;
        maxp[i] = std::max(maxp[i], k);
      }
  };
  std::vector<int> maxp;
  pieces(maxp);
  int slots = 0, groups = 0;
  for (int k : maxp)
    if (k > 1) {
      slots += k;
      ++groups;
    }
  if (groups > 0 && (slots > split_slots || groups > MAX_SPLIT_GROUPS)) {
    for (int c = 1; c < P; ++c) {
      const int x = plan.bounds[c], h = x / tph, r = x - h * tph;
      size_t i = 0;
      while (i + 1 < items.size() && items[i + 1].tbase <= r) ++i;
      const int s0 = h * tph + items[i].tbase, s1 = s0 + items[i].tiles;
      plan.bounds[c] = std::max(plan.bounds[c - 1], (x - s0 <= s1 - x) ? s0 : s1);
    }
    pieces(maxp);
  }
  int used = 0;
  for (size_t i = 0; i < items.size(); ++i) {
    int info = 0;
    if (maxp[i] > 1) {
      info = (used + 1) | (maxp[i] << 16);
      plan.groups.push_back(make_int4(items[i].seq, 0, used, maxp[i]));
      used += maxp[i];
    }
    plan.items.push_back(make_int4(items[i].seq, items[i].tiles, items[i].tbase, info));
  }
  return MLA_OK;
}

int launch_attn_fused(const mla_dims_t &d, int num_seqs, const int32_t *q_loc,
                      const int32_t *k_loc, const int32_t *q_loc_host, const int32_t *k_loc_host,
                      int T, const void *q_prep, const void *latent, int64_t latent_ld, int rows,
                      const void *w, const int32_t *acc, float *o, float *lse,
                      const SplitScratch *split, int32_t *status, cudaStream_t s) {
  auto al16 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
  if (!fused_attn_ok(d, latent_ld) || !al16(q_prep) || !al16(latent) || !al16(w))
    return MLA_ERR_UNSUPPORTED;
  const int H = d.num_heads;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    if (cudaOccupancyMaxActiveClusters(&n, attn_fused_kernel, &cfg) != cudaSuccess || n < 1)
      n = num_sms() / 2;
    max_clusters = std::min(n, MAX_PAIRS);
  }
  FusedPlan plan;
  int rc = plan_fused(H, num_seqs, q_loc_host, k_loc_host, max_clusters,
                      (split && split->o) ? split->slots : 0, plan);
  if (rc || plan.items.empty()) return rc;
  const int P = plan.P;
  thread_local FusedParams prm;
  prm.n_items = int(plan.items.size());
  prm.H = H;
  prm.T = T;
  prm.npairs = P;
  prm.tiles_per_head = plan.tph;
  prm.scale_log2 = d.softmax_scale * 1.4426950408889634f;
  prm.q_loc = q_loc;
  prm.k_loc = k_loc;
  prm.acc = acc;
  prm.w = static_cast<const uint16_t *>(w);
  prm.o = o;
  prm.lse = lse;
  prm.split_o = split ? split->o : nullptr;
  prm.split_lse = split ? split->lse : nullptr;
  prm.status = status;
  for (int c = 0; c <= P; ++c) prm.bounds[c] = plan.bounds[c];
  for (size_t i = 0; i < plan.items.size(); ++i) prm.items[i] = plan.items[i];

  CUtensorMap tq, tlat;
  if (!make_tmap_2d_16(&tq, false, q_prep, DQK, uint64_t(H) * T, uint64_t(DQK) * 2, 64, BQ,
                       true) ||
      !make_tmap_2d_16(&tlat, false, latent, 576, uint64_t(rows > 0 ? rows : 1),
                       uint64_t(latent_ld) * 2, 64, BKV, true))
    return MLA_ERR_CUDA;
  cfg.gridDim = dim3(2 * P);
  launch_begin(s);
  if (cudaLaunchKernelEx(&cfg, attn_fused_kernel, tq, tlat, prm) != cudaSuccess)
    return MLA_ERR_CUDA;
  rc = launch_status(s, "attn_fused_kernel");
  if (rc) return rc;
  if (!plan.groups.empty())
    rc = launch_split_combine(int(plan.groups.size()), plan.groups.data(), H, T, q_loc, acc,
                              *split, o, lse, s);
  return rc;
}

int fused_take_errors() { return sm103::take_error_flags_here(); }

}  // namespace mla

// Host-only view of the fused kernel's work split (what launch_attn_fused
// would hand each cluster), for checks without a GPU.
extern "C" int mla_fused_attn_plan(int32_t num_heads, int32_t num_seqs, const int32_t *q_loc_host,
                                   const int32_t *k_loc_host, int32_t clusters,
                                   int32_t split_slots, int32_t *bounds, int32_t bounds_cap,
                                   int32_t *items, int32_t items_cap, int32_t *num_clusters,
                                   int32_t *num_items, int32_t *num_groups) {
  if (num_heads < 1 || num_seqs < 0 || clusters < 1 || split_slots < 0 || !num_clusters ||
      !num_items || !num_groups || (num_seqs > 0 && (!q_loc_host || !k_loc_host)))
    return MLA_ERR_INVALID;
  for (int i = 0; i < num_seqs; ++i)
    if (q_loc_host[i + 1] < q_loc_host[i] || k_loc_host[i + 1] < k_loc_host[i])
      return MLA_ERR_INVALID;
  mla::FusedPlan plan;
  const int rc = mla::plan_fused(num_heads, num_seqs, q_loc_host, k_loc_host, clusters,
                                 split_slots, plan);
  if (rc) return rc;
  *num_clusters = plan.P;
  *num_items = int32_t(plan.items.size());
  *num_groups = int32_t(plan.groups.size());
  if (bounds == nullptr && items == nullptr) return MLA_OK;  // sizes only
  if (!bounds || !items || bounds_cap < plan.P + 1 || items_cap < int(plan.items.size()))
    return MLA_ERR_TOO_SMALL;
  for (int c = 0; c <= plan.P; ++c) bounds[c] = plan.bounds[c];
  for (size_t i = 0; i < plan.items.size(); ++i) {
    items[4 * i] = plan.items[i].x;
    items[4 * i + 1] = plan.items[i].y;
    items[4 * i + 2] = plan.items[i].z;
    items[4 * i + 3] = plan.items[i].w;
  }
  return MLA_OK;
}
