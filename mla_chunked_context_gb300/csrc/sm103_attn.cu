// Varlen MLA attention on the 5th-generation tensor cores (sm_103a), for the
// DeepSeek-V3 head shape: q/k = [nope 128 | rope 64] (192), v = 128.  q and
// the latent (k_pe) are bf16; the up-projected K_nope and V are fp16.
//
// What it computes (PR #50613 report, item 4: a backend's
// run_prefill_context_chunk over a ContextChunk returns (O, LSE) per query row
// and head; item 3: the chunk result is accumulated into the context
// partial): for each sequence i, query token t in [q_loc[i], q_loc[i+1]) and
// head h, with keys j in [k_loc[i], k_loc[i+1]):
//   s_j = scale * (q_nope . K_nope[j, h] + q_pe . k_pe[j])
//   O   = sum_j softmax(s)_j V[j, h];   LSE = ln sum_j exp(s_j)
// Context chunks see every key of their sequence; the causal (new-token)
// mode lets query p see keys 0..p.  K_nope and V come from the up-projected
// head-major workspace kv [H, rows, 256] (columns [0,128) / [128,256));
// k_pe is the latent row's tail, latent[row][512:576], shared by all heads.
//
// One CTA = one (sequence, 128-query tile, head) and a range of its 128-key
// tiles: all of them, or -- when a launch has too few (sequence, tile, head)
// units to fill the GPU -- one of several key splits, whose partial (O, LSE)
// go to a scratch slot and are LSE-merged by split_combine_kernel (the same
// merge as the chunk accumulation, over a split of the key set).  The same
// unit also runs in two kernels where one CTA per SM walks many units: the
// persistent one-unit kernel (prepared queries, units of a few dozen key
// tiles) and the looping kernel (many short units, a warpgroup per unit).
// Two softmax warpgroups share every S tile: A takes its keys 0-63, B keys
// 64-127, each thread half a query row; the two exchange their half-row
// maxima through shared memory every tile, so both apply the same running
// max and accumulate into one O.
//   warp 0     TMA producers: lane 0 the 128x192 Q tile once and per key
//              tile K = [K_nope (2 boxes) | k_pe (1 box)], lane 1 V (2
//              boxes), each double-buffered, 128-byte swizzle; a stage is
//              reloaded once the MMA that read it has completed (the S-full
//              / P.V-done commits).
//   warp 1     TMEM owner + S issuer: S = Q K^T (M=128, N=128, K=192: 8 fp16
//              tcgen05.mma for the nope part, 4 bf16 for the rope part) into
//              one of three S buffers.  Three S buffers let S of tiles j+1
//              and j+2 run on the tensor pipe while tile j is exponentiated,
//              so the pipe does not wait for the softmax (with two, the S of
//              tile j+2 had to follow the P.V of tile j, and the pipe idled
//              half the time).
//   warp 10    P.V issuer: O += P V (M=128, N=128, K=128: 8 fp16
//              tcgen05.mma, P read from TMEM, V an MN-major shared-memory
//              operand).  A tcgen05.mma holds its issuing thread for about
//              50 cycles, so one thread issuing both kinds was the bound.
//              Operand descriptors are built once; a K step adds its offset.
//   warps 2-5  softmax warpgroup A, warps 6-9 warpgroup B: one thread per
//              query row and half row; tcgen05.ld the half row of S, mask,
//              half-row max, exchange, online softmax in base 2 with a
//              lazily raised running max (O is rescaled in TMEM only when
//              the max grows by more than 2^8; exact, since O/l and LSE use
//              the same max), P as fp16 written over the warpgroup's own S
//              columns with tcgen05.st.  Epilogue: A writes columns 0-63 of
//              O, B columns 64-127; the result is written or LSE-merged into
//              the stored partial (accumulate).
// TMEM: S0 [0,128) S1 [128,256) S2 [256,384) (P_A over S cols [0,32), P_B
//       over [64,96)), O [384,512).
#include <algorithm>
#include <vector>

#include "sm103.cuh"

namespace mla {
namespace {

using namespace sm103;

constexpr int BQ = 128, BKV = 128, RING = 2, HALF = BKV / 2;
constexpr int DN = 128, DR = 64, DV = 128, DQK = DN + DR, HD = DN + DV;
constexpr int QBOX = 128 * 64 * 2;           // 16 KB: 128 rows x 64 16-bit
constexpr int KBOX = BKV * 64 * 2;           // 16 KB: 128 rows x 64 16-bit
constexpr int Q_BYTES = 3 * QBOX;            // 48 KB
constexpr int K_BYTES = 3 * KBOX;            // 48 KB: K_nope (2 boxes) + k_pe
constexpr int V_BYTES = 2 * KBOX;            // 32 KB
// one-CTA kernel: half-row maxima [2 warpgroups][2 tile parities][128],
// row sums [2][128], per-warp ok flags [2 parities][8]
constexpr int XCHG1_BYTES = (2 * 2 * 128 + 2 * 128) * 4 + 2 * 8 * 4;
constexpr int SMEM_BYTES1 = 1024 + Q_BYTES + RING * (K_BYTES + V_BYTES) + XCHG1_BYTES + 256;
constexpr int NSBUF = 3;                      // S buffers of the one-CTA kernel
constexpr uint32_t COL_O1 = NSBUF * BKV;      // its O accumulator
constexpr int THREADS = 320;
constexpr int THREADS1 = THREADS + 32;        // the one-CTA kernel: + a P.V issuer warp
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_O = 256;
constexpr int MAX_ITEMS = 1536;
constexpr int MAX_SPLIT_GROUPS = 16;   // split (sequence, tile)s per launch
constexpr int MAX_GROUP_SPLITS = 16;   // key splits of one (sequence, tile)
constexpr float kRescaleThreshold = 8.0f;    // log2 of the tolerated growth

struct AttnParams {
  int n_items, H, T, causal;
  float scale_log2;
  const int32_t *q_loc, *k_loc, *acc;
  float *o, *lse;
  // final-merge mode (fout != nullptr): (o, lse) hold the context partial,
  // read only; tokens below pnt are LSE-merged with it, the result goes to
  // fout (bf16 if fout_bf16, else f32) and flse (nullable)
  void *fout;
  float *flse;
  int pnt, fout_bf16;
  // q layout: 0 = the caller's [T, H, 192] bf16 (q_nope converted to fp16 in
  // shared memory); 1 = prepared head-major [H, T, 192] with q_nope already
  // fp16 (prepare_q_kernel), so a Q tile is one contiguous 48 KB block
  int q_prepared;
  // key-split scratch: slot k holds O [H][BQ][DV] (normalised) and LSE
  // [H][BQ] of one split
  float *split_o, *split_lse;
  // nullable: MLA_STATUS_FP16_RANGE when a q_nope value overflowed fp16
  int32_t *status;
  // looping and persistent kernels: after its context keys, each sequence
  // attends its own new tokens (rows q_loc[i] .. q_loc[i+1] of the second
  // K/V and latent maps), causally; context keys are then neither causal
  // nor split
  int new_keys;
  // (sequence, query tile | (split slot + 1) << 16, first key tile, end key
  // tile), the most key tiles first
  int4 items[MAX_ITEMS];
};

__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2^x with the SFU's approximate exponent (relative error below 2^-21; P is
// then rounded to fp16, 2^-11).  Arguments here are at most 8 (the lazily
// raised running max), results below 2^-126 flush to zero.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-input max (NaN inputs ignored, as fmaxf), and packed pairs of
// floats in one 64-bit register for the paired fp32 FMA / add of sm_100+:
// one instruction per two elements where the softmax has one per element.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t x, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// 16 consecutive 32-bit TMEM columns of the warp's 32 lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Four packed bf16 pairs to fp16 pairs (exact for bf16 values of magnitude
// 2^-14 .. 65504); amax collects the largest magnitude converted.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 x, float &amax) {
  uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xffff0000u);
    amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
    w4[e] = pack_f16(lo, hi);
  }
  return make_uint4(w4[0], w4[1], w4[2], w4[3]);
}

// q_nope (Q boxes 0 and 1) to fp16 in place, to meet the fp16 K_nope in the
// S MMA.  Thread tid of nthr; a value beyond fp16's range sets
// MLA_STATUS_FP16_RANGE in *status (nullable).
__device__ __forceinline__ void convert_q_nope(uint8_t *sQ, int tid, int nthr, int32_t *status) {
  uint4 *qv = reinterpret_cast<uint4 *>(sQ);
  float amax = 0.f;
#pragma unroll 4
  for (int v = tid; v < 2 * QBOX / 16; v += nthr) qv[v] = bf16x8_to_f16x8(qv[v], amax);
  fence_async_smem();
  if (status && amax >= kF16Overflow) atomicOr(status, MLA_STATUS_FP16_RANGE);
}

// Final-merge mode: whether token t (of sequence seq) is LSE-merged with
// the stored context partial -- a token below pnt, unless the launch's
// per-sequence flags (acc, when given) say that the partial holds no earlier
// result for the sequence.
__device__ __forceinline__ bool fin_merges(const AttnParams &p, int seq, int t) {
  return t < p.pnt && (p.acc == nullptr || __ldg(p.acc + seq) != 0);
}

// Brings the half row of the stored partial that the epilogue will merge
// with (a continued request, or the context partial in final-merge mode)
// into L2 while the unit computes, instead of leaving the epilogue to wait
// on it from HBM.
__device__ __forceinline__ void prefetch_partial(const AttnParams &p, int h, int seq, int slot,
                                                 int q_beg, int nq, int qpos, int wg) {
  if (qpos >= nq || slot >= 0) return;
  const int t = q_beg + qpos;
  const bool fin = p.fout != nullptr;
  const bool acc = !fin && p.acc != nullptr && __ldg(p.acc + seq) != 0;
  if (!acc && !(fin && fin_merges(p, seq, t))) return;
  const float *row = p.o + (int64_t(t) * p.H + h) * DV + wg * (DV / 2);
  asm volatile("prefetch.global.L2 [%0];" ::"l"(row));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(row + 32));
}

// The 256 softmax threads of the one-CTA kernel meet at named barrier 1;
// the result is the AND of `ok` over them (every warp passes the same
// value for all its lanes).
__device__ __forceinline__ bool softmax_bar_and(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred a, b;\n setp.ne.u32 a, %1, 0;\n bar.red.and.pred b, 1, 256, a;\n"
      " selp.u32 %0, 1, 0, b;\n}\n"
      : "=r"(r)
      : "r"(ok ? 1u : 0u)
      : "memory");
  return r != 0;
}

// One 128-key tile (tile J of the CTA, S buffer J % 3) of the online
// softmax, for one warpgroup's half (64 keys, the first being key k0 of the
// sequence) of query row qpos: S from TMEM (s_col), masked past the
// sequence (and, causal, past the query); the half-row maxima of both
// warpgroups meet in xm (parity J % 2) at named barrier 1, so both raise the
// shared running max alike; P as fp16 over the warpgroup's S columns; the
// warpgroup's 64 columns of O (o_col) rescaled when the max grew -- after
// the P.V of tile J-1 -- then an arrival on pfull_bar.  A warp whose wait
// gives up still reaches the barrier with ok_w false, and every warp leaves
// at that tile (returns false), so the barrier counts always match.
__device__ __forceinline__ bool softmax_tile1(const AttnParams &p, uint32_t s_col, uint32_t o_col,
                                              uint32_t sfull_bar, uint32_t sfull_parity,
                                              uint32_t b_odone, uint32_t pfull_bar, int J,
                                              int k0, int kend, float *xm, int wg,
                                              int row, bool &ok_w, float &m_used, float &l,
                                              int lane) {
  float sv[HALF];  // raw scores (scale applied below)
  float mh = neg_inf();
  if (ok_w) ok_w = __all_sync(0xffffffffu, mbar_wait(sfull_bar, sfull_parity)) != 0;
  if (ok_w) {
    tc_fence_after();
    uint32_t r0[32], r1[32];
    tmem_ld32(s_col, r0);  // both halves in flight before the wait
    tmem_ld32(s_col + 32u, r1);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      sv[e] = __uint_as_float(r0[e]);
      sv[32 + e] = __uint_as_float(r1[e]);
    }
    // mask keys from kend on (past the sequence, and with a causal mask past
    // the query)
    const int valid = kend - k0;
    if (valid < HALF) {
#pragma unroll
      for (int e = 0; e < HALF; ++e)
        if (e >= valid) sv[e] = neg_inf();
    }
    // half-row max as a tree of three-input maxima (32 instructions for the
    // 64 values, no serial dependency chain)
    float t[22], u[8];
#pragma unroll
    for (int i = 0; i < 21; ++i) t[i] = fmax3(sv[3 * i], sv[3 * i + 1], sv[3 * i + 2]);
    t[21] = sv[63];
#pragma unroll
    for (int i = 0; i < 7; ++i) u[i] = fmax3(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
    u[7] = t[21];
    mh = fmaxf(fmax3(u[0], u[1], u[2]), fmax3(fmax3(u[3], u[4], u[5]), u[6], u[7]));
  }
  const int par = J & 1;
  xm[(wg * 2 + par) * BQ + row] = mh;
  if (!softmax_bar_and(ok_w)) {
    ok_w = false;
    return false;
  }
  // the row max (scale > 0: the max of the scaled scores is the scaled
  // max); fmaxf of the two halves gives both warpgroups the same value
  const float mx = fmaxf(mh, xm[((1 - wg) * 2 + par) * BQ + row]) * p.scale_log2;
  float alpha = 1.f;
  bool rescale = false;
  if (mx > m_used + kRescaleThreshold || m_used == neg_inf()) {
    const float m_new = fmaxf(mx, m_used);
    if (m_used != neg_inf() && m_new != neg_inf()) {
      alpha = exp2f(m_used - m_new);
      rescale = true;
    }
    m_used = m_new;
  }
  const float nbase = (m_used == neg_inf()) ? 0.f : -m_used;
  l *= alpha;
  uint32_t pk[HALF / 2];
  // exponent arguments two at a time (paired FMA), sums in two paired
  // accumulators (four independent partial sums)
  const uint64_t sc2 = f2pack(p.scale_log2, p.scale_log2), nb2 = f2pack(nbase, nbase);
  uint64_t acc[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
  for (int e = 0; e < HALF / 2; ++e) {
    float xa, xb;
    f2unpack(f2fma(f2pack(sv[2 * e], sv[2 * e + 1]), sc2, nb2), xa, xb);
    const float a = ex2_approx(xa), b = ex2_approx(xb);
    acc[e & 1] = f2add(acc[e & 1], f2pack(a, b));
    pk[e] = pack_f16(a, b);
  }
  float s0, s1, s2, s3;
  f2unpack(acc[0], s0, s1);
  f2unpack(acc[1], s2, s3);
  l += (s0 + s1) + (s2 + s3);
  // P over this warpgroup's own S columns (already read).  O is rescaled
  // once the previous tile's P.V is done (done barrier (J-1) % 3: the P.V of
  // tile J+2 cannot run before this warp arrives, and that of tile J-4
  // finished before S of tile J-1 was issued, so the wait is one phase from
  // its barrier's state); otherwise this tile's P.V may follow the previous
  // one directly.
  tmem_st32(s_col, pk);
  if (__any_sync(0xffffffffu, rescale)) {
    const bool done = J == 0 || mbar_wait(b_odone + 8u * uint32_t((J - 1) % NSBUF),
                                          uint32_t(((J - 1) / NSBUF) & 1));
    if (!__all_sync(0xffffffffu, done)) {
      ok_w = false;  // reported at the next tile's barrier or in the epilogue
    } else {
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < DV / 2 / 32; ++c) {
        uint32_t r[32];
        const uint32_t oc = o_col + uint32_t(c * 32);
        tmem_ld32(oc, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
        tmem_st32(oc, r);
      }
    }
  }
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(pfull_bar);
  return true;
}

// Epilogue of one (query tile, head) unit of the one-CTA kernel, run by both
// softmax warpgroups: after the unit's last P.V (odone at odone_parity), the
// row sum is the sum of the two warpgroups' (same running max); each writes
// its 64 columns of O / l -- or LSE-merges them into the stored partial (a
// continued request), into the key-split scratch slot, or with the context
// partial into the final output -- as the launch asks.  All threads of the
// CTA meet at one barrier.  Returns the AND over the threads of `ok`.
__device__ __forceinline__ bool unit_epilogue1(const AttnParams &p, uint32_t o_col, float *xl,
                                               uint8_t *stage, uint32_t b_odone,
                                               uint32_t odone_parity, int wg,
                                               int row, int lane, int h, int seq, int slot,
                                               int q_beg, int nq, int qpos, int n_tiles,
                                               float m_used, float l, bool ok) {
  if (ok && n_tiles > 0 && !__all_sync(0xffffffffu, mbar_wait(b_odone, odone_parity))) ok = false;
  xl[wg * BQ + row] = l;
  const int t = q_beg + qpos;
  const int64_t li = int64_t(h) * p.T + t;
  const bool fin = p.fout != nullptr;
  const bool split = slot >= 0;  // a key split: its own partial goes to the scratch slot
  const bool accumulate = !fin && !split && p.acc != nullptr && __ldg(p.acc + seq) != 0;
  const bool merge_old = accumulate || (fin && fin_merges(p, seq, t));
  // the stored LSE is read by both warpgroups before either writes it
  const float old = (merge_old && qpos < nq) ? p.lse[li] : neg_inf();
  // this warpgroup's half of the output row, and the row's LSE
  float *orow = split ? p.split_o + ((int64_t(slot) * p.H + h) * BQ + row) * DV + wg * (DV / 2)
                      : p.o + (int64_t(t) * p.H + h) * DV + wg * (DV / 2);
  // the stored half row, when it holds a result (finite LSE), read now with
  // all 16 loads in flight
  float4 ov[DV / 2 / 4];
  const bool have_old = merge_old && qpos < nq && !is_neg_inf(old);
  if (have_old) {
#pragma unroll
    for (int i = 0; i < DV / 2 / 4; ++i) ov[i] = reinterpret_cast<const float4 *>(orow)[i];
  }
  tc_fence_before();
  // both warpgroups' sums are in xl after this barrier; all threads take
  // part, the MMA warps too
  const int okv = __syncthreads_and(ok ? 1 : 0);
  tc_fence_after();
  const float lsum = xl[row] + xl[BQ + row];
  const bool store = okv && qpos < nq;
  float lse = (lsum > 0.f) ? (m_used + __log2f(lsum)) * 0.69314718055994531f : neg_inf();
  float w_new = (lsum > 0.f) ? 1.f / lsum : 0.f, w_old = 0.f;
  float *lse_dst = split ? p.split_lse + (int64_t(slot) * p.H + h) * BQ + row : p.lse + li;
  bool write = store;
  if (store && merge_old) {
    if (lsum == 0.f) {
      if (!fin) {
        write = false;  // nothing new: keep the stored partial
      } else if (!is_neg_inf(old)) {
        w_old = 1.f;  // the result is the context partial alone
        lse = old;
      }
    } else if (!is_neg_inf(old)) {
      const float m2 = fmaxf(old, lse);
      const float eo = expf(old - m2), en = expf(lse - m2);
      w_old = eo / (eo + en);
      w_new *= en / (eo + en);
      lse = m2 + logf(eo + en);
    }
  }
  // the result rows go through shared memory (`stage`: 128 rows x 512 B of
  // float32, 16-byte chunk k of row r at chunk k ^ (r % 32), conflict-free
  // both ways; then a write flag per row), so that each warp store below
  // writes one whole row: a thread per row storing its own row made each
  // warp instruction touch 32 rows H x 512 B apart
  float4 *st4 = reinterpret_cast<float4 *>(stage);
  int *row_write = reinterpret_cast<int *>(stage + BQ * DV * 4);
  if (okv && n_tiles > 0) {
#pragma unroll
    for (int c = 0; c < DV / 2 / 16; ++c) {
      uint32_t ra[16];
      __syncwarp();  // converged after the per-lane stores of the previous piece
      tmem_ld16(o_col + uint32_t(c * 16), ra);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          v[k] = (w_new != 0.f) ? __uint_as_float(ra[4 * e + k]) * w_new : 0.f;
        float4 o4 = make_float4(v[0], v[1], v[2], v[3]);
        if (w_old != 0.f) {  // only when the stored LSE is finite (have_old)
          const float4 ovv = ov[c * 4 + e];
          o4.x += w_old * ovv.x;
          o4.y += w_old * ovv.y;
          o4.z += w_old * ovv.z;
          o4.w += w_old * ovv.w;
        }
        const int k = wg * (DV / 8) + c * 4 + e;  // 16-byte chunk of the row
        st4[row * (DV / 4) + (k ^ (row & 31))] = o4;
      }
    }
  } else {
    // no key tiles: zeros (stored only where the row is written)
#pragma unroll 1
    for (int c = 0; c < DV / 8; ++c)
      st4[row * (DV / 4) + ((wg * (DV / 8) + c) ^ (row & 31))] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (wg == 0) row_write[row] = write ? 1 : 0;
  if (write && wg == 0) {
    if (!fin)
      *lse_dst = lse;
    else if (p.flse)
      p.flse[li] = lse;
  }
  asm volatile("bar.sync 1, 256;" ::: "memory");  // the 256 softmax threads
  // warp w of the softmax warpgroups writes rows 16w .. 16w+15, 16 bytes a lane
  const int wi = wg * 4 + (row >> 5);
  const int t0 = t - row;  // the tile's first token
#pragma unroll 1
  for (int i = 0; i < BQ / 8; ++i) {
    const int rr = wi * (BQ / 8) + i;
    if (!row_write[rr]) continue;
    const float4 v = st4[rr * (DV / 4) + (lane ^ (rr & 31))];
    const int64_t rowbase = split ? ((int64_t(slot) * p.H + h) * BQ + rr) * DV
                                   : (int64_t(t0 + rr) * p.H + h) * DV;
    if (split) {
      reinterpret_cast<float4 *>(p.split_o + rowbase)[lane] = v;
    } else if (!fin) {
      reinterpret_cast<float4 *>(p.o + rowbase)[lane] = v;
    } else if (p.fout_bf16) {
      uint2 b2;
      b2.x = pack_bf16(v.x, v.y);
      b2.y = pack_bf16(v.z, v.w);
      reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.fout) + rowbase)[lane] = b2;
    } else {
      reinterpret_cast<float4 *>(static_cast<float *>(p.fout) + rowbase)[lane] = v;
    }
  }
  return okv != 0;
}

__global__ void __launch_bounds__(THREADS1, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_kv,
                   const __grid_constant__ CUtensorMap tm_lat,
                   const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sQ = smem;
  uint8_t *sK = sQ + Q_BYTES;
  uint8_t *sV = sK + RING * K_BYTES;
  float *xm = reinterpret_cast<float *>(sV + RING * V_BYTES);  // [2 wg][2 parities][128]
  float *xl = xm + 2 * 2 * BQ;                                 // [2 wg][128]
  uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(xm) + XCHG1_BYTES);
  // q, qready, K full [2 stages], V full [2 stages], S full [3 buffers], P
  // full [3 buffers] (8 softmax warps), P.V done [3 buffers], each issuer's
  // MMAs done
  const uint32_t b_q = smem_u32(bars + 0), b_qready = smem_u32(bars + 1);
  const uint32_t b_kfull = smem_u32(bars + 2), b_vfull = smem_u32(bars + 4);
  const uint32_t b_sfull = smem_u32(bars + 6), b_pfull = smem_u32(bars + 9);
  const uint32_t b_odone = smem_u32(bars + 12), b_done = smem_u32(bars + 15);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 17);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x / p.n_items;
  const int4 it = p.items[blockIdx.x - h * p.n_items];
  const int seq = it.x, qt = it.y & 0xffff, slot = (it.y >> 16) - 1;
  const int q_beg = __ldg(p.q_loc + seq), nq = __ldg(p.q_loc + seq + 1) - q_beg;
  const int k_beg = __ldg(p.k_loc + seq), nk = __ldg(p.k_loc + seq + 1) - k_beg;
  const int q0 = qt * BQ;  // first query of the tile, within the sequence
  // key tiles [kt0, kt0 + n_tiles) of the sequence (the host applied the
  // causal limit)
  const int kt0 = it.z, n_tiles = it.w - it.z;

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    mbar_init(b_qready, 4);
    for (int s = 0; s < RING; ++s) {
      mbar_init(b_kfull + 8 * s, 1);
      mbar_init(b_vfull + 8 * s, 1);
    }
    for (int b = 0; b < NSBUF; ++b) {
      mbar_init(b_sfull + 8 * b, 1);
      mbar_init(b_pfull + 8 * b, 8);
      mbar_init(b_odone + 8 * b, 1);
    }
    mbar_init(b_done, 1);
    mbar_init(b_done + 8, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane < 2 && n_tiles > 0) {
      // ---------------- TMA producers: lane 0 Q and K, lane 1 V, so that a
      // K stage is refilled as soon as its S is done and a V stage as soon
      // as its P.V is, each in its own order
      const bool kl = lane == 0;
      if (kl) {
        prefetch_map(&tm_q);
        prefetch_map(&tm_kv);
        prefetch_map(&tm_lat);
        const int qx = p.q_prepared ? 0 : h * DQK;
        const int qy = (p.q_prepared ? h * p.T : 0) + q_beg + q0;
        mbar_expect_tx(b_q, Q_BYTES);
        tma_load_2d(smem_u32(sQ), &tm_q, b_q, qx, qy);
        tma_load_2d(smem_u32(sQ + QBOX), &tm_q, b_q, qx + 64, qy);
        tma_load_2d(smem_u32(sQ + 2 * QBOX), &tm_q, b_q, qx + 128, qy);
      }
      int issued[RING];
      for (int s = 0; s < RING; ++s) issued[s] = -1;
      const uint32_t full = kl ? b_kfull : b_vfull;
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % RING;
        const uint32_t use = uint32_t(j / RING);  // use count of stage s
        const int krow = k_beg + (kt0 + j) * BKV;
        // stage s held tile j-2: its K is free once S of tile j-2 is done,
        // its V once the P.V of tile j-2 is
        if (j >= RING &&
            !mbar_wait((kl ? b_sfull : b_odone) + 8 * ((j - 2) % NSBUF),
                       uint32_t(((j - 2) / NSBUF) & 1)))
          break;
        if (kl) {
          uint8_t *k = sK + s * K_BYTES;
          mbar_expect_tx(full + 8 * s, K_BYTES);
          tma_load_3d(smem_u32(k), &tm_kv, full + 8 * s, 0, krow, h);
          tma_load_3d(smem_u32(k + KBOX), &tm_kv, full + 8 * s, 64, krow, h);
          tma_load_2d(smem_u32(k + 2 * KBOX), &tm_lat, full + 8 * s, 512, krow);
        } else {
          uint8_t *v = sV + s * V_BYTES;
          mbar_expect_tx(full + 8 * s, V_BYTES);
          tma_load_3d(smem_u32(v), &tm_kv, full + 8 * s, DN, krow, h);
          tma_load_3d(smem_u32(v + KBOX), &tm_kv, full + 8 * s, DN + 64, krow, h);
        }
        issued[s] = int(use & 1);
      }
      // every issued load has landed before the CTA may exit
      if (kl) mbar_wait(b_q, 0);
      for (int s = 0; s < RING; ++s)
        if (issued[s] >= 0) mbar_wait(full + 8 * s, uint32_t(issued[s]));
    }
  } else if (warp == 1 || warp == THREADS1 / 32 - 1) {
    if (lane == 0 && n_tiles > 0) {
      // ---------------- MMA issuers: warp 1 the S products, the last warp
      // the P.V products, each committing its own.  A tcgen05.mma holds its
      // issuing thread for about 50 cycles (more beside busy softmax warps),
      // so one issuer for both kinds left the tensor pipe idle while it
      // issued the other kind; split, S of tiles j+1 and j+2 and P.V of tile
      // j are issued side by side.  S of tile j reuses S buffer j % 3 once
      // the P.V of tile j-3 is done (they are issued by different threads,
      // so issue order alone would not order them).
      constexpr uint32_t idesc_nope = idesc_f16kind(BQ, BKV, false, false, false);  // fp16
      constexpr uint32_t idesc_rope = idesc_f16kind(BQ, BKV, false, false, true);   // bf16
      constexpr uint32_t idesc_o = idesc_f16kind(BQ, DV, false, true, false);       // fp16
      // descriptors built once; a K step or a stage adds its byte offset / 16
      // to the start-address field (shared addresses stay below 2^18, so the
      // 14-bit field never carries)
      bool ok = true;
      if (warp == 1) {
        const uint64_t dq = desc_kmajor_sw128(smem_u32(sQ));
        const uint64_t dk0 = desc_kmajor_sw128(smem_u32(sK));
        ok = mbar_wait(b_qready, 0);
        for (int j = 0; ok && j < n_tiles; ++j) {
          const int s = j % RING, b = j % NSBUF;
          if ((j >= NSBUF && !mbar_wait(b_odone + 8 * b, uint32_t(((j - NSBUF) / NSBUF) & 1))) ||
              !mbar_wait(b_kfull + 8 * s, uint32_t((j / RING) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dk = dk0 + uint64_t((s * K_BYTES) >> 4);
          const uint32_t d = tmem + COL_S + uint32_t(b * BKV);
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk) {
            const uint64_t off = uint64_t(((kk >> 2) * QBOX + (kk & 3) * 32) >> 4);
            mma_bf16(d, dq + off, dk + off, kk < DN / 16 ? idesc_nope : idesc_rope, kk != 0);
          }
          mma_commit(b_sfull + 8 * b);  // S ready; K stage s free
        }
      } else {
        const uint64_t dv0 = desc_mnmajor_sw128(smem_u32(sV), KBOX);
        for (int j = 0; ok && j < n_tiles; ++j) {
          const int s = j % RING, b = j % NSBUF;
          if (!mbar_wait(b_vfull + 8 * s, uint32_t((j / RING) & 1)) ||
              !mbar_wait(b_pfull + 8 * b, uint32_t((j / NSBUF) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // P_A (keys 0-63) over S columns [0, 32), P_B (keys 64-127) over [64, 96)
          const uint32_t pa = tmem + COL_S + uint32_t(b * BKV);
          const uint64_t dv = dv0 + uint64_t((s * V_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)
            mma_f16_ts(tmem + COL_O1, pa + uint32_t((kk >> 2) * HALF + (kk & 3) * 8),
                       dv + uint64_t((kk * 2048) >> 4), idesc_o, (j | kk) != 0);
          mma_commit(b_odone + 8 * b);  // P.V done; V stage s and S buffer b free
        }
      }
      // every MMA this thread issued has completed before TMEM is released
      const uint32_t dbar = b_done + (warp == 1 ? 0u : 8u);
      mma_commit(dbar);
      mbar_wait(dbar, 0);
    }
  } else {
    // ---------------- softmax warpgroups
    const int wg = (warp - 2) >> 2;        // 0: A (keys 0-63 of a tile), 1: B (64-127)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // query row of the tile = TMEM lane
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const int qpos = q0 + row;             // position within the sequence
    float m_used = neg_inf(), l = 0.f;
    bool ok = true;
    if (n_tiles > 0 && wg == 0) {
      if (!mbar_wait(b_q, 0))
        ok = false;
      else if (!p.q_prepared)
        convert_q_nope(sQ, threadIdx.x - 64, 128, p.status);
      __syncwarp();
      if (lane == 0) mbar_arrive(b_qready);
    }
    ok = __all_sync(0xffffffffu, ok) != 0;
    prefetch_partial(p, h, seq, slot, q_beg, nq, qpos, wg);
    // this warpgroup's 64 columns of O
    const uint32_t o_col = tmem + lane_off + COL_O1 + uint32_t(wg * (DV / 2));
    // the row's key bound, counted from the unit's first key
    const int kend = (p.causal ? min(nk, qpos + 1) : nk) - kt0 * BKV;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j % NSBUF;
      const uint32_t s_col = tmem + lane_off + COL_S + uint32_t(b * BKV + wg * HALF);
      if (!softmax_tile1(p, s_col, o_col, b_sfull + 8 * b, uint32_t((j / NSBUF) & 1), b_odone,
                         b_pfull + 8 * b, j, j * BKV + wg * HALF, kend, xm, wg, row, ok, m_used,
                         l, lane))
        break;
    }
    // the unit's last P.V: done barrier (n_tiles-1) % 3, its ((n_tiles-1)/3)-th phase
    // the K ring is free once the unit's last P.V is done: the epilogue
    // stages its rows there
    unit_epilogue1(p, o_col, xl, sK, b_odone + 8u * uint32_t((n_tiles + NSBUF - 1) % NSBUF),
                   uint32_t(((n_tiles - 1) / NSBUF) & 1), wg, row, lane, h, seq, slot, q_beg, nq,
                   qpos, n_tiles, m_used, l, ok);
  }
  if (warp < 2 || warp == THREADS1 / 32 - 1) __syncthreads_and(1);  // the softmax warps' vote
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Epilogue of one unit of the persistent one-CTA kernel: as
// unit_epilogue1, except that the two softmax warpgroups meet at named
// barrier 1 (the other warps have run ahead into the next unit), the row
// sums alternate between two buffers by unit (xl: this unit's), and each
// warp writes its own 32 half rows through its 1 KB staging tile (`stg`,
// 32 rows x 32 bytes, 16-byte chunks XOR-swizzled by row; the K ring holds
// the next unit's keys): each store instruction writes 32 contiguous bytes
// of 16 rows.  Returns the AND over the softmax threads of `ok`.
__device__ __forceinline__ bool unit_epilogue_p(const AttnParams &p, uint32_t o_col, float *xl,
                                                uint32_t stg, uint32_t b_odone,
                                                uint32_t odone_parity, int wg, int row, int lane,
                                                int h, int seq, int slot, int q_beg, int nq,
                                                int qpos, int n_tiles, float m_used, float l,
                                                bool ok) {
  if (ok && n_tiles > 0 && !__all_sync(0xffffffffu, mbar_wait(b_odone, odone_parity))) ok = false;
  xl[wg * BQ + row] = l;
  const int t = q_beg + qpos;
  const int64_t li = int64_t(h) * p.T + t;
  const bool fin = p.fout != nullptr;
  const bool split = slot >= 0;
  const bool accumulate = !fin && !split && p.acc != nullptr && __ldg(p.acc + seq) != 0;
  const bool merge_old = accumulate || (fin && fin_merges(p, seq, t));
  const float old = (merge_old && qpos < nq) ? p.lse[li] : neg_inf();
  const float *orow = p.o + (int64_t(t) * p.H + h) * DV + wg * (DV / 2);  // the stored partial
  tc_fence_before();
  const bool okv = softmax_bar_and(ok);  // both warpgroups' sums are in xl
  tc_fence_after();
  const float lsum = xl[row] + xl[BQ + row];
  const bool store = okv && qpos < nq;
  float lse = (lsum > 0.f) ? (m_used + __log2f(lsum)) * 0.69314718055994531f : neg_inf();
  float w_new = (lsum > 0.f) ? 1.f / lsum : 0.f, w_old = 0.f;
  bool write = store;
  if (store && merge_old) {
    if (lsum == 0.f) {
      if (!fin) {
        write = false;  // nothing new: keep the stored partial
      } else if (!is_neg_inf(old)) {
        w_old = 1.f;  // the result is the context partial alone
        lse = old;
      }
    } else if (!is_neg_inf(old)) {
      const float m2 = fmaxf(old, lse);
      const float eo = expf(old - m2), en = expf(lse - m2);
      w_old = eo / (eo + en);
      w_new *= en / (eo + en);
      lse = m2 + logf(eo + en);
    }
  }
  if (write && wg == 0) {
    if (split)
      p.split_lse[(int64_t(slot) * p.H + h) * BQ + row] = lse;
    else if (!fin)
      p.lse[li] = lse;
    else if (p.flse)
      p.flse[li] = lse;
  }
  // the warp's rows: row 16i + (lane >> 1) of the warp at dst + i * step,
  // this warpgroup's 64 columns; lane & 1 the 16-byte chunk of a round
  const uint32_t wmask = __ballot_sync(0xffffffffu, write);
  const int srow = lane >> 1, sk = lane & 1;
  const int r0 = row - lane + srow;  // tile row of this lane's first stored row
  const bool out16 = fin && p.fout_bf16;
  const int64_t es = out16 ? 2 : 4;
  const int64_t grow = split ? (int64_t(slot) * p.H + h) * BQ + r0
                             : int64_t(t - row + r0) * p.H + h;
  char *dst = reinterpret_cast<char *>(split ? p.split_o : (fin ? p.fout : p.o)) +
              (grow * DV + wg * (DV / 2)) * es;
  const int64_t step = (split ? 16 : int64_t(16) * p.H) * DV * es;
  const bool have = okv && n_tiles > 0;
#pragma unroll
  for (int c = 0; c < DV / 2 / 16; ++c) {
    // the stored row's piece first, then the TMEM read of the same piece
    float4 ov[4];
    if (w_old != 0.f) {  // only when the stored LSE is finite
#pragma unroll
      for (int i = 0; i < 4; ++i) ov[i] = reinterpret_cast<const float4 *>(orow)[c * 4 + i];
    }
    uint32_t ra[16];
    if (have) {
      __syncwarp();
      tmem_ld16(o_col + uint32_t(c * 16), ra);
      tmem_wait_ld();
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {  // 8 values (32 bytes) of the row a round
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int e = hh * 2 + k;     // float4 e of this piece of 16
        float4 o4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (have) {
          o4 = make_float4(__uint_as_float(ra[4 * e]) * w_new, __uint_as_float(ra[4 * e + 1]) * w_new,
                           __uint_as_float(ra[4 * e + 2]) * w_new,
                           __uint_as_float(ra[4 * e + 3]) * w_new);
          if (w_new == 0.f) o4 = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (w_old != 0.f) {
          const float4 ovv = ov[e];
          o4.x += w_old * ovv.x;
          o4.y += w_old * ovv.y;
          o4.z += w_old * ovv.z;
          o4.w += w_old * ovv.w;
        }
        st_shared_v4(stg + uint32_t(lane * 32 + ((k ^ ((lane >> 2) & 1)) << 4)),
                     make_uint4(__float_as_uint(o4.x), __float_as_uint(o4.y),
                                __float_as_uint(o4.z), __float_as_uint(o4.w)));
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int rr = 16 * i + srow;
        const uint4 v = ld_shared_v4(stg + uint32_t(rr * 32 + ((sk ^ ((rr >> 2) & 1)) << 4)));
        if ((wmask >> rr) & 1u) {
          const int64_t col = int64_t(c * 16 + hh * 8 + sk * 4);  // within the half row
          if (out16) {
            uint2 b2;
            b2.x = pack_bf16(__uint_as_float(v.x), __uint_as_float(v.y));
            b2.y = pack_bf16(__uint_as_float(v.z), __uint_as_float(v.w));
            *reinterpret_cast<uint2 *>(dst + i * step + col * 2) = b2;
          } else {
            *reinterpret_cast<uint4 *>(dst + i * step + col * 4) = v;
          }
        }
      }
      __syncwarp();  // the staging tile is rewritten next round
    }
  }
  return okv;
}

// The one-CTA attention as a persistent kernel, for launches of prepared
// queries with several units per SM: a CTA per SM walks the units
// u = blockIdx.x, + gridDim.x, ... (head-major, as the one-unit kernel's
// CTAs run) with its barriers and TMEM kept and the tiles of all its units
// numbered on (tile J of the CTA: S buffer, P-full and P.V-done J % 3, K/V
// stage J % 2).  The next unit's Q is loaded once the last S of the current
// unit is done, and its K/V tiles and first S products follow while the
// softmax warps still run the current unit's last tiles and epilogue (with
// a CTA per unit, the start and the end of each were exposed: about a
// quarter of a 32-key-tile unit).  The next unit's first P.V overwrites O
// only after the softmax warps have read it: they arrive on that tile's
// P-full after their epilogue.  The softmax warps re-read a unit's
// description from the launch parameters.
constexpr int XCHG2_BYTES = (2 * 2 * 128 + 2 * 2 * 128) * 4;  // xm; xl [2 unit parities]
constexpr int STG2_BYTES = 8 * 32 * 32;                         // 1 KB per softmax warp
constexpr int SMEM_BYTES2 =
    1024 + Q_BYTES + RING * (K_BYTES + V_BYTES) + XCHG2_BYTES + STG2_BYTES + 256;
static_assert(SMEM_BYTES2 <= 227 * 1024, "persistent kernel: shared memory");

__global__ void __launch_bounds__(THREADS1, 1)
    attn_tc_persist_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_kv,
                           const __grid_constant__ CUtensorMap tm_lat,
                           const __grid_constant__ CUtensorMap tm_kv2,
                           const __grid_constant__ CUtensorMap tm_lat2,
                           const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sQ = smem;
  uint8_t *sK = sQ + Q_BYTES;
  uint8_t *sV = sK + RING * K_BYTES;
  float *xm = reinterpret_cast<float *>(sV + RING * V_BYTES);  // [2 wg][2 tile parities][128]
  float *xl = xm + 2 * 2 * BQ;                                 // [2 unit parities][2 wg][128]
  uint8_t *sStg = reinterpret_cast<uint8_t *>(xl + 2 * 2 * BQ);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sStg + STG2_BYTES);
  // q, qfree, K full [2], V full [2], S full [3], P full [3] (8 softmax
  // warps), P.V done [3], each issuer's MMAs done
  const uint32_t b_q = smem_u32(bars + 0), b_qfree = smem_u32(bars + 1);
  const uint32_t b_kfull = smem_u32(bars + 2), b_vfull = smem_u32(bars + 4);
  const uint32_t b_sfull = smem_u32(bars + 6), b_pfull = smem_u32(bars + 9);
  const uint32_t b_odone = smem_u32(bars + 12), b_done = smem_u32(bars + 15);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 17);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_units = p.n_items * p.H;
  const int G = int(gridDim.x), b0 = int(blockIdx.x);
  // unit u: head u / n_items, item u % n_items
  auto item_of = [&](int u, int &h) {
    h = u / p.n_items;
    return p.items[u - h * p.n_items];
  };

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    mbar_init(b_qfree, 1);
    for (int s = 0; s < RING; ++s) {
      mbar_init(b_kfull + 8 * s, 1);
      mbar_init(b_vfull + 8 * s, 1);
    }
    for (int b = 0; b < NSBUF; ++b) {
      mbar_init(b_sfull + 8 * b, 1);
      mbar_init(b_pfull + 8 * b, 8);
      mbar_init(b_odone + 8 * b, 1);
    }
    mbar_init(b_done, 1);
    mbar_init(b_done + 8, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane < 2) {
      // ---------------- TMA producers: lane 0 Q and K, lane 1 V
      const bool kl = lane == 0;
      if (kl) {
        prefetch_map(&tm_q);
        prefetch_map(&tm_kv);
        prefetch_map(&tm_lat);
        if (p.new_keys) prefetch_map(&tm_lat2);
      }
      if (p.new_keys) prefetch_map(&tm_kv2);
      int issued[RING];
      for (int s = 0; s < RING; ++s) issued[s] = -1;
      int q_issued = -1;
      const uint32_t full = kl ? b_kfull : b_vfull;
      int J = 0, kq = 0;  // the CTA's key tiles; its units with tiles
      bool ok = true;
      for (int u = b0; ok && u < n_units; u += G) {
        int h;
        const int4 it = item_of(u, h);
        const int n_tiles = it.w - it.z;
        if (n_tiles <= 0) continue;
        const int seq = it.x, qt = it.y & 0xffff, kt0 = it.z;
        const int k_beg = __ldg(p.k_loc + seq), q_beg = __ldg(p.q_loc + seq);
        // with new keys: the unit's first ct tiles are context keys, the
        // rest the sequence's new tokens
        const int ct = p.new_keys ? (__ldg(p.k_loc + seq + 1) - k_beg + BKV - 1) / BKV : n_tiles;
        if (kl) {
          // the previous unit's S products are done with the Q tile
          if (kq > 0 && !mbar_wait(b_qfree, uint32_t((kq - 1) & 1))) break;
          const int qy = h * p.T + q_beg + qt * BQ;
          mbar_expect_tx(b_q, Q_BYTES);
          tma_load_2d(smem_u32(sQ), &tm_q, b_q, 0, qy);
          tma_load_2d(smem_u32(sQ + QBOX), &tm_q, b_q, 64, qy);
          tma_load_2d(smem_u32(sQ + 2 * QBOX), &tm_q, b_q, 128, qy);
          q_issued = kq & 1;
        }
        ++kq;
        for (int j = 0; j < n_tiles; ++j, ++J) {
          const int s = J % RING;
          const bool nk_tile = j >= ct;  // a new-token key tile
          const int krow = nk_tile ? q_beg + (j - ct) * BKV : k_beg + (kt0 + j) * BKV;
          const CUtensorMap *mkv = nk_tile ? &tm_kv2 : &tm_kv;
          // stage s held tile J-2: its K is free once S of tile J-2 is done,
          // its V once the P.V of tile J-2 is
          if (J >= RING && !mbar_wait((kl ? b_sfull : b_odone) + 8 * ((J - 2) % NSBUF),
                                      uint32_t(((J - 2) / NSBUF) & 1))) {
            ok = false;
            break;
          }
          if (kl) {
            uint8_t *k = sK + s * K_BYTES;
            mbar_expect_tx(full + 8 * s, K_BYTES);
            tma_load_3d(smem_u32(k), mkv, full + 8 * s, 0, krow, h);
            tma_load_3d(smem_u32(k + KBOX), mkv, full + 8 * s, 64, krow, h);
            tma_load_2d(smem_u32(k + 2 * KBOX), nk_tile ? &tm_lat2 : &tm_lat, full + 8 * s, 512,
                        krow);
          } else {
            uint8_t *v = sV + s * V_BYTES;
            mbar_expect_tx(full + 8 * s, V_BYTES);
            tma_load_3d(smem_u32(v), mkv, full + 8 * s, DN, krow, h);
            tma_load_3d(smem_u32(v + KBOX), mkv, full + 8 * s, DN + 64, krow, h);
          }
          issued[s] = int((J / RING) & 1);
        }
      }
      // every issued load has landed before the CTA may exit
      if (kl && q_issued >= 0) mbar_wait(b_q, uint32_t(q_issued));
      for (int s = 0; s < RING; ++s)
        if (issued[s] >= 0) mbar_wait(full + 8 * s, uint32_t(issued[s]));
    }
  } else if (warp == 1 || warp == THREADS1 / 32 - 1) {
    if (lane == 0) {
      // ---------------- MMA issuers: warp 1 the S products, the last warp
      // the P.V products, each committing its own (as in the one-unit kernel)
      constexpr uint32_t idesc_nope = idesc_f16kind(BQ, BKV, false, false, false);  // fp16
      constexpr uint32_t idesc_rope = idesc_f16kind(BQ, BKV, false, false, true);   // bf16
      constexpr uint32_t idesc_o = idesc_f16kind(BQ, DV, false, true, false);       // fp16
      bool ok = true;
      int J = 0, kq = 0;
      if (warp == 1) {
        const uint64_t dq = desc_kmajor_sw128(smem_u32(sQ));
        const uint64_t dk0 = desc_kmajor_sw128(smem_u32(sK));
        for (int u = b0; ok && u < n_units; u += G) {
          int h;
          const int4 it = item_of(u, h);
          const int n_tiles = it.w - it.z;
          if (n_tiles <= 0) continue;
          if (!mbar_wait(b_q, uint32_t(kq & 1))) break;
          ++kq;
          for (int j = 0; j < n_tiles; ++j, ++J) {
            const int s = J % RING, b = J % NSBUF;
            if ((J >= NSBUF &&
                 !mbar_wait(b_odone + 8 * b, uint32_t(((J - NSBUF) / NSBUF) & 1))) ||
                !mbar_wait(b_kfull + 8 * s, uint32_t((J / RING) & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t dk = dk0 + uint64_t((s * K_BYTES) >> 4);
            const uint32_t d = tmem + COL_S + uint32_t(b * BKV);
#pragma unroll
            for (int kk = 0; kk < DQK / 16; ++kk) {
              const uint64_t off = uint64_t(((kk >> 2) * QBOX + (kk & 3) * 32) >> 4);
              mma_bf16(d, dq + off, dk + off, kk < DN / 16 ? idesc_nope : idesc_rope, kk != 0);
            }
            mma_commit(b_sfull + 8 * b);  // S ready; K stage s free
            if (j == n_tiles - 1) mma_commit(b_qfree);  // the unit's last S: Q is free
          }
        }
      } else {
        const uint64_t dv0 = desc_mnmajor_sw128(smem_u32(sV), KBOX);
        for (int u = b0; ok && u < n_units; u += G) {
          int h;
          const int4 it = item_of(u, h);
          const int n_tiles = it.w - it.z;
          for (int j = 0; j < n_tiles; ++j, ++J) {
            const int s = J % RING, b = J % NSBUF;
            // P-full of the unit's first tile also means the softmax warps
            // have read the previous unit's O
            if (!mbar_wait(b_vfull + 8 * s, uint32_t((J / RING) & 1)) ||
                !mbar_wait(b_pfull + 8 * b, uint32_t((J / NSBUF) & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t pa = tmem + COL_S + uint32_t(b * BKV);
            const uint64_t dv = dv0 + uint64_t((s * V_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < BKV / 16; ++kk)
              mma_f16_ts(tmem + COL_O1, pa + uint32_t((kk >> 2) * HALF + (kk & 3) * 8),
                         dv + uint64_t((kk * 2048) >> 4), idesc_o, (j | kk) != 0);
            mma_commit(b_odone + 8 * b);  // P.V done; V stage s and S buffer b free
          }
        }
      }
      const uint32_t dbar = b_done + (warp == 1 ? 0u : 8u);
      mma_commit(dbar);
      mbar_wait(dbar, 0);
    }
  } else {
    // ---------------- softmax warpgroups
    const int wg = (warp - 2) >> 2;        // 0: A (keys 0-63 of a tile), 1: B (64-127)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // query row of the tile = TMEM lane
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const uint32_t o_col = tmem + lane_off + COL_O1 + uint32_t(wg * (DV / 2));
    const uint32_t stg = smem_u32(sStg) + uint32_t((warp - 2) * 1024);
    int J = 0, ku = 0;
    bool ok = true;
    for (int u = b0; u < n_units; u += G, ++ku) {
      int h;
      const int4 it = item_of(u, h);
      const int seq = it.x, qt = it.y & 0xffff, slot = (it.y >> 16) - 1;
      const int kt0 = it.z, n_tiles = it.w - it.z > 0 ? it.w - it.z : 0;
      const int q_beg = __ldg(p.q_loc + seq), nq = __ldg(p.q_loc + seq + 1) - q_beg;
      const int nk = __ldg(p.k_loc + seq + 1) - __ldg(p.k_loc + seq);
      const int qpos = qt * BQ + row;
      float m_used = neg_inf(), l = 0.f;
      prefetch_partial(p, h, seq, slot, q_beg, nq, qpos, wg);
      // the context key tiles, then with new keys the sequence's own new
      // tokens (keys 0 .. nq-1, causal): keys counted from the unit's
      // first, valid below kend.  With new keys the context keys are not
      // causal and not split, so their bound is nk on every row and the
      // first tile at or past it is the first new-token tile; until then
      // kend holds ~nk (negative: the context phase).
      int kend = (p.causal ? min(nk, qpos + 1) : nk) - kt0 * BKV;
      if (p.new_keys) kend = ~kend;
      for (int j = 0; j < n_tiles; ++j) {
        if (kend < 0 && j * BKV >= ~kend) kend = min(nq, qpos + 1) + j * BKV;
        const int JJ = J + j, b = JJ % NSBUF;
        const uint32_t s_col = tmem + lane_off + COL_S + uint32_t(b * BKV + wg * HALF);
        if (!softmax_tile1(p, s_col, o_col, b_sfull + 8 * b, uint32_t((JJ / NSBUF) & 1), b_odone,
                           b_pfull + 8 * b, JJ, j * BKV + wg * HALF, kend < 0 ? ~kend : kend, xm,
                           wg, row, ok, m_used, l, lane))
          break;
      }
      const int JL = J + n_tiles - 1;  // the unit's last tile
      ok = unit_epilogue_p(p, o_col, xl + (ku & 1) * 2 * BQ, stg,
                           b_odone + 8u * uint32_t((JL + NSBUF) % NSBUF),
                           uint32_t((JL / NSBUF) & 1), wg, row, lane, h, seq, slot, q_beg, nq,
                           qpos, n_tiles, m_used, l, ok);
      J += n_tiles;
      if (!ok) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// The same attention for launches of many short units (a few key tiles per
// (query tile, head)): a CTA per SM walks its units u = blockIdx.x,
// + gridDim.x, ... in turn, keeping its barriers and TMEM.  The two softmax
// warpgroups take alternate units (the CTA's k-th unit belongs to warpgroup
// k % 2), each with full 128-key rows and its own O accumulator, so one
// unit's epilogue (the read of O, the merge with the stored partial, the
// stores) runs while the other warpgroup's unit is scored and
// exponentiated.  The barriers count on across units (key tile J is the
// CTA's J-th over all its units; a warpgroup's pfull / odone / ofree count
// its own tiles and units), and a converter warp (warp 10) turns each
// unit's q_nope to fp16 as soon as it lands when the queries are not
// prepared, so the next unit's Q and K/V loads and its S MMAs overlap this
// unit's softmax and epilogue.
// TMEM: S0 [0,128) S1 [128,256) (P of a tile over the first 64 columns of
// its S buffer), O of warpgroup 0 [256,384), of warpgroup 1 [384,512).
constexpr int THREADS_LOOP = THREADS + 32;
constexpr int STG_LOOP_BYTES = 8 * 32 * 64;  // a 32 x 64-byte staging tile per softmax warp
constexpr int SMEM_BYTES_LOOP =
    1024 + Q_BYTES + RING * (K_BYTES + V_BYTES) + STG_LOOP_BYTES + 256;
static_assert(SMEM_BYTES_LOOP <= 227 * 1024, "looping kernel: shared memory");

// One 128-key tile of the online softmax for a full query row (qpos) of a
// warpgroup's unit: the row's scores come out of TMEM in two halves of 64
// keys, each masked (past the sequence, and causal past the query), its max
// raising the running max lazily (by more than 2^8 only), exponentiated and
// written back as fp16 P over the first 64 columns of the S buffer.  When the
// second half raises the max, the first half's P is rescaled in TMEM (rare).
// O is rescaled after the warpgroup's previous P.V (odone, its jw-th tile)
// has finished; then an arrival on pfull.  Returns false when a wait gave up.
__device__ __forceinline__ bool softmax_tile_full(const AttnParams &p, uint32_t s_col,
                                                  uint32_t o_col, uint32_t sfull_bar,
                                                  uint32_t sfull_parity, uint32_t b_odone,
                                                  uint32_t pfull_bar, int jw, int k0,
                                                  int kend, float &m_used, float &l, int lane) {
  // every exit is taken by the whole warp (its TMEM accesses are warp-wide)
  if (!__all_sync(0xffffffffu, mbar_wait(sfull_bar, sfull_parity))) return false;
  tc_fence_after();
  float alpha = 1.f;
  bool rescale = false;
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    float sv[HALF];
    __syncwarp();  // tcgen05.ld/st are warp-wide: the warp is converged here
    {
      uint32_t r0[32], r1[32];
      tmem_ld32(s_col + uint32_t(hh * HALF), r0);
      tmem_ld32(s_col + uint32_t(hh * HALF + 32), r1);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        sv[e] = __uint_as_float(r0[e]);
        sv[32 + e] = __uint_as_float(r1[e]);
      }
    }
    // keys k0 + hh * HALF + e, valid below kend (the row's key bound: the
    // source's key count, and with a causal mask its query position + 1)
    const int valid = kend - (k0 + hh * HALF);
    if (valid < HALF) {
#pragma unroll
      for (int e = 0; e < HALF; ++e)
        if (e >= valid) sv[e] = neg_inf();
    }
    // the half's max as a tree of three-input maxima
    float t[22], u[8];
#pragma unroll
    for (int i = 0; i < 21; ++i) t[i] = fmax3(sv[3 * i], sv[3 * i + 1], sv[3 * i + 2]);
    t[21] = sv[63];
#pragma unroll
    for (int i = 0; i < 7; ++i) u[i] = fmax3(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
    u[7] = t[21];
    const float mx =
        fmaxf(fmax3(u[0], u[1], u[2]), fmax3(fmax3(u[3], u[4], u[5]), u[6], u[7])) * p.scale_log2;
    float a_first = 1.f;  // this lane's rescale of the tile's first half of P
    if (mx > m_used + kRescaleThreshold || m_used == neg_inf()) {
      const float m_new = fmaxf(mx, m_used);
      if (m_used != neg_inf() && m_new != neg_inf()) {
        const float a = exp2f(m_used - m_new);
        alpha *= a;
        l *= a;
        rescale = true;
        if (hh == 1) a_first = a;
      }
      m_used = m_new;
    }
    if (hh == 1 && __any_sync(0xffffffffu, a_first != 1.f)) {
      // the first half's P was exponentiated against the old max (rows
      // whose max did not move multiply by 1, exactly); the whole warp
      // takes part in the TMEM read and write
      uint32_t r[32];
      tmem_wait_st();
      tmem_ld32(s_col, r);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const __half2 h2 = *reinterpret_cast<const __half2 *>(&r[e]);
        const float2 f = __half22float2(h2);
        r[e] = pack_f16(f.x * a_first, f.y * a_first);
      }
      tmem_st32(s_col, r);
    }
    const float nbase = (m_used == neg_inf()) ? 0.f : -m_used;
    uint32_t pk[HALF / 2];
    // exponent arguments two at a time (paired FMA), sums in two paired
    // accumulators
    const uint64_t sc2 = f2pack(p.scale_log2, p.scale_log2), nb2 = f2pack(nbase, nbase);
    uint64_t acc[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
    for (int e = 0; e < HALF / 2; ++e) {
      float xa, xb;
      f2unpack(f2fma(f2pack(sv[2 * e], sv[2 * e + 1]), sc2, nb2), xa, xb);
      const float a = ex2_approx(xa), b = ex2_approx(xb);
      acc[e & 1] = f2add(acc[e & 1], f2pack(a, b));
      pk[e] = pack_f16(a, b);
    }
    float s0, s1, s2, s3;
    f2unpack(acc[0], s0, s1);
    f2unpack(acc[1], s2, s3);
    l += (s0 + s1) + (s2 + s3);
    // P of keys [hh*64, hh*64+64) over columns [hh*32, hh*32+32): those S
    // columns are already read (the first half was read before it is
    // overwritten; the second half's own columns lie beyond 64)
    __syncwarp();
    tmem_st32(s_col + uint32_t(hh * 32), pk);
  }
  // the warpgroup's previous P.V into O has finished before O is rescaled
  if (!__all_sync(0xffffffffu, jw == 0 || mbar_wait(b_odone, uint32_t((jw - 1) & 1))))
    return false;
  tc_fence_after();
  if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
    for (int c = 0; c < DV / 32; ++c) {
      uint32_t r[32];
      const uint32_t oc = o_col + uint32_t(c * 32);
      tmem_ld32(oc, r);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
      tmem_st32(oc, r);
    }
  }
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(pfull_bar);
  return true;
}

// Epilogue of one unit for a full query row: after the unit's last P.V
// (odone at odone_parity), O / l and the LSE are written -- or LSE-merged
// into the stored partial (a continued request), into the key-split scratch
// slot, or with the context partial into the final output -- as the launch
// asks.  Each thread owns its row, so no barrier is needed; the warp
// arrives on b_ofree once it has read O from TMEM.
__device__ __forceinline__ bool unit_epilogue_full(const AttnParams &p, uint32_t o_col,
                                                   uint32_t b_odone, uint32_t odone_parity,
                                                   uint32_t b_ofree, uint32_t stg, int lane, int h,
                                                   int seq, int slot, int q_beg, int nq, int qpos,
                                                   int n_tiles, float m_used, float l, bool ok) {
  if (ok && n_tiles > 0 && !mbar_wait(b_odone, odone_parity)) ok = false;
  ok = __all_sync(0xffffffffu, ok) != 0;
  const int t = q_beg + qpos;
  const int64_t li = int64_t(h) * p.T + t;
  const bool fin = p.fout != nullptr;
  const bool split = slot >= 0;
  const bool accumulate = !fin && !split && p.acc != nullptr && __ldg(p.acc + seq) != 0;
  const bool merge_old = accumulate || (fin && fin_merges(p, seq, t));
  const bool live = qpos < nq;
  const float old = (merge_old && live) ? p.lse[li] : neg_inf();
  float *orow = split ? p.split_o + ((int64_t(slot) * p.H + h) * BQ + (qpos & (BQ - 1))) * DV
                      : p.o + (int64_t(t) * p.H + h) * DV;
  const bool have_old = merge_old && live && !is_neg_inf(old);
  tc_fence_after();
  const bool store = ok && live;
  float lse = (l > 0.f) ? (m_used + __log2f(l)) * 0.69314718055994531f : neg_inf();
  float w_new = (l > 0.f) ? 1.f / l : 0.f, w_old = 0.f;
  float *lse_dst = split ? p.split_lse + (int64_t(slot) * p.H + h) * BQ + (qpos & (BQ - 1))
                         : p.lse + li;
  bool write = store;
  if (store && merge_old) {
    if (l == 0.f) {
      if (!fin) {
        write = false;  // nothing new: keep the stored partial
      } else if (!is_neg_inf(old)) {
        w_old = 1.f;  // the result is the context partial alone
        lse = old;
      }
    } else if (!is_neg_inf(old)) {
      const float m2 = fmaxf(old, lse);
      const float eo = expf(old - m2), en = expf(lse - m2);
      w_old = eo / (eo + en);
      w_new *= en / (eo + en);
      lse = m2 + logf(eo + en);
    }
  }
  if (ok && n_tiles > 0) {
    // four pieces of 32 columns; the stored row's piece is loaded before
    // the TMEM read of the same piece.  The warp's 32 rows go out through
    // its 32 x 64-byte staging tile: each thread writes its row's 64 bytes
    // (four 16-byte chunks, XOR-swizzled by row), then each store
    // instruction writes 64 contiguous bytes of 8 rows (4 lanes per row)
    // instead of 16 bytes of 32 rows.
    const int srow = lane >> 2, sk = lane & 3;
    const int qpos0 = qpos - lane;  // the warp's first row
    const bool out16 = fin && p.fout_bf16;
    const uint32_t wmask = __ballot_sync(0xffffffffu, write);
    // row 8i + srow of the warp starts at dst + i * step (rows 8 apart: 8
    // query positions, in the same (slot, head) block when split)
    const int qr = qpos0 + srow;
    const int64_t row0 = split ? (int64_t(slot) * p.H + h) * BQ + (qr & (BQ - 1))
                               : int64_t(q_beg + qr) * p.H + h;
    const int64_t es = out16 ? 2 : 4;
    char *dst = reinterpret_cast<char *>(split ? p.split_o : (fin ? p.fout : p.o)) +
                row0 * DV * es;
    const int64_t step = (split ? 8 : int64_t(8) * p.H) * DV * es;
#pragma unroll 1
    for (int c = 0; c < DV / 32; ++c) {
      float4 ov[8];
      if (have_old && w_old != 0.f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) ov[i] = reinterpret_cast<const float4 *>(orow + c * 32)[i];
      }
      uint32_t r[32];
      __syncwarp();  // converged again after the per-lane loads above
      tmem_ld32(o_col + uint32_t(c * 32), r);
      tmem_wait_ld();
      if (c == DV / 32 - 1) {
        // O is read: the warpgroup's next unit may accumulate into it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_ofree);
      }
      // float32: two rounds of 16 values (64 bytes a row); bf16: the two
      // halves of the piece are packed into one 64-byte round
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float4 o4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int ee = hh * 4 + e;
          o4[e] = make_float4(__uint_as_float(r[4 * ee]) * w_new,
                              __uint_as_float(r[4 * ee + 1]) * w_new,
                              __uint_as_float(r[4 * ee + 2]) * w_new,
                              __uint_as_float(r[4 * ee + 3]) * w_new);
          if (w_old != 0.f) {  // only when the stored LSE is finite (have_old)
            o4[e].x += w_old * ov[ee].x;
            o4[e].y += w_old * ov[ee].y;
            o4[e].z += w_old * ov[ee].z;
            o4[e].w += w_old * ov[ee].w;
          }
        }
        if (out16) {
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const uint4 v = make_uint4(pack_bf16(o4[2 * k].x, o4[2 * k].y),
                                       pack_bf16(o4[2 * k].z, o4[2 * k].w),
                                       pack_bf16(o4[2 * k + 1].x, o4[2 * k + 1].y),
                                       pack_bf16(o4[2 * k + 1].z, o4[2 * k + 1].w));
            st_shared_v4(stg + uint32_t(lane * 64 + (((hh * 2 + k) ^ ((lane >> 1) & 3)) << 4)), v);
          }
          if (hh == 0) continue;  // the row's 64 bytes are complete after the second half
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            st_shared_v4(stg + uint32_t(lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)),
                         make_uint4(__float_as_uint(o4[k].x), __float_as_uint(o4[k].y),
                                    __float_as_uint(o4[k].z), __float_as_uint(o4[k].w)));
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = 8 * i + srow;
          const uint4 v = ld_shared_v4(stg + uint32_t(rr * 64 + ((sk ^ ((rr >> 1) & 3)) << 4)));
          if ((wmask >> rr) & 1u)
            reinterpret_cast<uint4 *>(dst + i * step + (out16 ? c * 64 : (c * 32 + hh * 16) * 4))[sk] =
                v;
        }
        __syncwarp();  // the staging tile is rewritten next round
      }
    }
  } else {
    if (n_tiles > 0) {  // O unread (a wait gave up): release it all the same
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_ofree);
    }
    if (write && n_tiles == 0) {
      if (!fin) {
        // no key (an accumulating row kept its partial: write is false)
        for (int c = 0; c < DV; c += 4)
          *reinterpret_cast<float4 *>(orow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        // no key: the context partial passes through (w_old = 1), or zeros
        for (int c = 0; c < DV; c += 4) {
          float4 o4 = make_float4(0.f, 0.f, 0.f, 0.f);
          if (w_old != 0.f) o4 = reinterpret_cast<const float4 *>(orow)[c / 4];
          const int64_t col = (int64_t(t) * p.H + h) * DV + c;
          if (p.fout_bf16) {
            uint2 b2;
            b2.x = pack_bf16(o4.x, o4.y);
            b2.y = pack_bf16(o4.z, o4.w);
            *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.fout) + col) = b2;
          } else {
            *reinterpret_cast<float4 *>(static_cast<float *>(p.fout) + col) = o4;
          }
        }
      }
    }
  }
  if (write) {
    if (!fin)
      *lse_dst = lse;
    else if (p.flse)
      p.flse[li] = lse;
  }
  return ok;
}

__global__ void __launch_bounds__(THREADS_LOOP, 1)
    attn_tc_loop_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_kv,
                        const __grid_constant__ CUtensorMap tm_lat,
                        const __grid_constant__ CUtensorMap tm_kv2,
                        const __grid_constant__ CUtensorMap tm_lat2,
                        const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sQ = smem;
  uint8_t *sK = sQ + Q_BYTES;
  uint8_t *sV = sK + RING * K_BYTES;
  uint8_t *sStg = sV + RING * V_BYTES;  // the softmax warps' epilogue staging tiles
  uint64_t *bars = reinterpret_cast<uint64_t *>(sStg + STG_LOOP_BYTES);
  const uint32_t b_q = smem_u32(bars + 0), b_qready = smem_u32(bars + 1);
  const uint32_t b_kfull = smem_u32(bars + 2), b_kempty = smem_u32(bars + 2 + RING);
  const uint32_t b_vfull = smem_u32(bars + 2 + 2 * RING), b_vempty = smem_u32(bars + 2 + 3 * RING);
  // sfull: [2 warpgroups][2 S buffers] -- the S MMA of a tile arrives on its
  // owner's barrier for that buffer, so each warpgroup sees every phase of
  // its barriers in order (a barrier shared by both would let a warpgroup
  // that skipped the other's phases take an old phase for the new one)
  const uint32_t b_sfull = smem_u32(bars + 2 + 4 * RING);
  const uint32_t b_pfull = b_sfull + 32;                    // [2]: per warpgroup
  const uint32_t b_odone = b_sfull + 48;                    // [2]: per warpgroup
  const uint32_t b_ofree = b_sfull + 64;                    // [2]: per warpgroup
  const uint32_t b_qfree = b_sfull + 80, b_done = b_sfull + 88;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 + 4 * RING + 12);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_units = p.n_items * p.H;

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    mbar_init(b_qready, 1);
    for (int s = 0; s < RING; ++s) {
      mbar_init(b_kfull + 8 * s, 1);
      mbar_init(b_kempty + 8 * s, 1);
      mbar_init(b_vfull + 8 * s, 1);
      mbar_init(b_vempty + 8 * s, 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(b_sfull + 16 * w, 1);
      mbar_init(b_sfull + 16 * w + 8, 1);
      mbar_init(b_pfull + 8 * w, 4);
      mbar_init(b_odone + 8 * w, 1);
      mbar_init(b_ofree + 8 * w, 4);
    }
    mbar_init(b_qfree, 1);
    mbar_init(b_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  struct Unit {
    int h, seq, qt, slot, kt0, n_tiles;
  };
  // units head-major (unit u: head u / n_items, item u % n_items; the items
  // come longest first), the CTA's k-th unit taken from the k-th block of
  // gridDim.x units in zigzag order: the units that run at the same time
  // are every query tile of a few heads, so each (sequence, head)'s keys are
  // read from DRAM once and shared in L2 by its query tiles, and the long
  // items spread over the CTAs
  const int G = int(gridDim.x), b = int(blockIdx.x);
  auto unit_at = [&](int k) { return k * G + ((k & 1) ? G - 1 - b : b); };
  auto unit_of = [&](int u) {
    Unit x;
    x.h = u / p.n_items;
    const int item = u - x.h * p.n_items;
    const int4 it = p.items[item];
    x.seq = it.x;
    x.qt = it.y & 0xffff;
    x.slot = (it.y >> 16) - 1;
    x.kt0 = it.z;
    x.n_tiles = it.w - it.z;
    return x;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      prefetch_map(&tm_q);
      prefetch_map(&tm_kv);
      prefetch_map(&tm_lat);
      if (p.new_keys) {
        prefetch_map(&tm_kv2);
        prefetch_map(&tm_lat2);
      }
      int k_issued[RING], v_issued[RING], q_issued = -1;
      for (int s = 0; s < RING; ++s) k_issued[s] = v_issued[s] = -1;
      int J = 0, kq = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int u = unit_at(k);
        if (u >= n_units) break;
        const Unit x = unit_of(u);
        if (x.n_tiles <= 0) continue;
        const int q_beg = __ldg(p.q_loc + x.seq), k_beg = __ldg(p.k_loc + x.seq);
        // with new keys: the unit's first ct tiles are context keys, the
        // rest the sequence's new tokens
        const int ct = p.new_keys ? (__ldg(p.k_loc + x.seq + 1) - k_beg + BKV - 1) / BKV : x.n_tiles;
        // the previous unit's S MMAs are done with the Q tile
        if (kq > 0 && !mbar_wait(b_qfree, uint32_t((kq - 1) & 1))) break;
        const int qx = p.q_prepared ? 0 : x.h * DQK;
        const int qy = (p.q_prepared ? x.h * p.T : 0) + q_beg + x.qt * BQ;
        mbar_expect_tx(b_q, Q_BYTES);
        tma_load_2d(smem_u32(sQ), &tm_q, b_q, qx, qy);
        tma_load_2d(smem_u32(sQ + QBOX), &tm_q, b_q, qx + 64, qy);
        tma_load_2d(smem_u32(sQ + 2 * QBOX), &tm_q, b_q, qx + 128, qy);
        q_issued = kq & 1;
        ++kq;
        for (int j = 0; j < x.n_tiles; ++j, ++J) {
          const int s = J % RING;
          const uint32_t use = uint32_t(J / RING);        // use count of slot s
          const bool nk_tile = j >= ct;                   // a new-token key tile
          const int krow = nk_tile ? q_beg + (j - ct) * BKV : k_beg + (x.kt0 + j) * BKV;
          const CUtensorMap *mkv = nk_tile ? &tm_kv2 : &tm_kv;
          const CUtensorMap *mlat = nk_tile ? &tm_lat2 : &tm_lat;
          if (J >= RING && !mbar_wait(b_kempty + 8 * s, (use - 1) & 1)) {
            ok = false;
            break;
          }
          uint8_t *kk = sK + s * K_BYTES;
          mbar_expect_tx(b_kfull + 8 * s, K_BYTES);
          tma_load_3d(smem_u32(kk), mkv, b_kfull + 8 * s, 0, krow, x.h);
          tma_load_3d(smem_u32(kk + KBOX), mkv, b_kfull + 8 * s, 64, krow, x.h);
          tma_load_2d(smem_u32(kk + 2 * KBOX), mlat, b_kfull + 8 * s, 512, krow);
          k_issued[s] = int(use & 1);
          if (J >= RING && !mbar_wait(b_vempty + 8 * s, (use - 1) & 1)) {
            ok = false;
            break;
          }
          uint8_t *v = sV + s * V_BYTES;
          mbar_expect_tx(b_vfull + 8 * s, V_BYTES);
          tma_load_3d(smem_u32(v), mkv, b_vfull + 8 * s, DN, krow, x.h);
          tma_load_3d(smem_u32(v + KBOX), mkv, b_vfull + 8 * s, DN + 64, krow, x.h);
          v_issued[s] = int(use & 1);
        }
      }
      // every issued load has landed before the CTA may exit
      if (q_issued >= 0) mbar_wait(b_q, uint32_t(q_issued));
      for (int s = 0; s < RING; ++s) {
        if (k_issued[s] >= 0) mbar_wait(b_kfull + 8 * s, uint32_t(k_issued[s]));
        if (v_issued[s] >= 0) mbar_wait(b_vfull + 8 * s, uint32_t(v_issued[s]));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc_nope = idesc_f16kind(BQ, BKV, false, false, false);  // fp16
      constexpr uint32_t idesc_rope = idesc_f16kind(BQ, BKV, false, false, true);   // bf16
      constexpr uint32_t idesc_o = idesc_f16kind(BQ, DV, false, true, false);       // fp16
      const uint32_t q_addr = smem_u32(sQ);
      int J0 = 0, kq = 0, ku = 0;
      int jw[2] = {0, 0}, uw[2] = {0, 0};   // per warpgroup: P.V tiles, units with tiles
      bool ok = true;
      for (int k = 0; ok; ++k, ++ku) {
        const int u = unit_at(k);
        if (u >= n_units) break;
        const Unit x = unit_of(u);
        const int n_tiles = x.n_tiles;
        if (n_tiles <= 0) continue;
        const int w = ku & 1;              // the warpgroup that owns this unit
        if (!mbar_wait(b_qready, uint32_t(kq & 1))) break;
        // S for key tile J into S buffer J & 1 (which held P of tile J-2,
        // whose P.V MMAs were issued before); after the unit's last S the
        // Q tile is released
        auto issue_s = [&](int j) -> bool {
          const int J = J0 + j, s = J % RING;
          if (!mbar_wait(b_kfull + 8 * s, uint32_t((J / RING) & 1))) return false;
          tc_fence_after();
          const uint32_t k_addr = smem_u32(sK + s * K_BYTES);
          const uint32_t d = tmem + COL_S + uint32_t((J & 1) * BKV);
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk) {
            const uint32_t off = uint32_t((kk >> 2) * QBOX + (kk & 3) * 32);
            mma_bf16(d, desc_kmajor_sw128(q_addr + off), desc_kmajor_sw128(k_addr + off),
                     kk < DN / 16 ? idesc_nope : idesc_rope, kk != 0);
          }
          mma_commit(b_sfull + 16 * w + 8 * (J & 1));
          mma_commit(b_kempty + 8 * s);
          if (j == n_tiles - 1) mma_commit(b_qfree);
          return true;
        };
        ok = issue_s(0);
        if (ok && n_tiles > 1) ok = issue_s(1);
        // the warpgroup's previous unit's epilogue has read its O
        if (ok && uw[w] > 0 && !mbar_wait(b_ofree + 8 * w, uint32_t((uw[w] - 1) & 1))) ok = false;
        const uint32_t od = tmem + COL_O + uint32_t(w * DV);
        for (int j = 0; ok && j < n_tiles; ++j) {
          const int J = J0 + j, s = J % RING;
          if (!mbar_wait(b_vfull + 8 * s, uint32_t((J / RING) & 1)) ||
              !mbar_wait(b_pfull + 8 * w, uint32_t(jw[w] & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t pa = tmem + COL_S + uint32_t((J & 1) * BKV);
          const uint32_t vb = smem_u32(sV + s * V_BYTES);
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)
            mma_f16_ts(od, pa + uint32_t(kk * 8), desc_mnmajor_sw128(vb + uint32_t(kk * 2048), KBOX),
                       idesc_o, (j | kk) != 0);
          mma_commit(b_odone + 8 * w);
          mma_commit(b_vempty + 8 * s);
          ++jw[w];
          if (j + 2 < n_tiles) ok = issue_s(j + 2);
        }
        ++uw[w];
        J0 += n_tiles;
        ++kq;
      }
      mma_commit(b_done);
      mbar_wait(b_done, 0);
    }
  } else if (warp == THREADS / 32) {
    // ---------------- Q converter (warp 10)
    int kq = 0;
    for (int k = 0;; ++k) {
      const int u = unit_at(k);
      if (u >= n_units) break;
      const Unit x = unit_of(u);
      if (x.n_tiles <= 0) continue;
      const bool ok = mbar_wait(b_q, uint32_t(kq & 1));
      if (ok && !p.q_prepared) convert_q_nope(sQ, lane, 32, p.status);
      __syncwarp();
      if (lane == 0) mbar_arrive(b_qready);
      ++kq;
      if (!ok) break;
    }
  } else {
    // ---------------- softmax warpgroups, on alternate units
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // query row of the tile = TMEM lane
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const uint32_t o_col = tmem + lane_off + COL_O + uint32_t(wg * DV);
    int J0 = 0, jw = 0;                    // the CTA's key tiles; this warpgroup's
    int sc0 = 0, sc1 = 0;                  // this warpgroup's tiles in S buffer 0 / 1
    bool ok = true;
    for (int k = 0, ku = 0;; ++k, ++ku) {
      const int u = unit_at(k);
      if (u >= n_units) break;
      const Unit x = unit_of(u);
      const int n_tiles = x.n_tiles > 0 ? x.n_tiles : 0;
      if ((ku & 1) != wg) {
        J0 += n_tiles;
        continue;
      }
      const int q_beg = __ldg(p.q_loc + x.seq), nq = __ldg(p.q_loc + x.seq + 1) - q_beg;
      const int nk = __ldg(p.k_loc + x.seq + 1) - __ldg(p.k_loc + x.seq);
      const int qpos = x.qt * BQ + row;    // position within the sequence
      float m_used = neg_inf(), l = 0.f;
      if (qpos < nq && x.slot < 0) {
        // the stored row the epilogue may merge with, into L2 meanwhile
        const int t = q_beg + qpos;
        const bool fin = p.fout != nullptr;
        const bool acc = !fin && p.acc != nullptr && __ldg(p.acc + x.seq) != 0;
        if (acc || (fin && fin_merges(p, x.seq, t))) {
          const float *r = p.o + (int64_t(t) * p.H + x.h) * DV;
#pragma unroll
          for (int c = 0; c < DV; c += 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(r + c));
        }
      }
      // the context key tiles (keys x.kt0 * BKV + ...), then with new keys
      // the sequence's own new tokens (keys 0 .. nq-1, causal): tile j's
      // keys counted from the unit's first, valid below kend
      const int ct = p.new_keys ? (nk + BKV - 1) / BKV : n_tiles;
      int kend = (p.causal ? min(nk, qpos + 1) : nk) - x.kt0 * BKV;
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j == ct) kend = min(nq, qpos + 1) + ct * BKV;
        const int J = J0 + j;
        const uint32_t s_col = tmem + lane_off + COL_S + uint32_t((J & 1) * BKV);
        const int sc = (J & 1) ? sc1++ : sc0++;
        ok = softmax_tile_full(p, s_col, o_col, b_sfull + 16 * wg + 8 * (J & 1),
                               uint32_t(sc & 1), b_odone + 8 * wg, b_pfull + 8 * wg, jw,
                               j * BKV, kend, m_used, l, lane);
        ok = __all_sync(0xffffffffu, ok) != 0;
        ++jw;
      }
      ok = unit_epilogue_full(p, o_col, b_odone + 8 * wg, uint32_t((jw - 1) & 1),
                              b_ofree + 8 * wg, smem_u32(sStg) + uint32_t((warp - 2) * 2048),
                              lane, x.h, x.seq, x.slot, q_beg, nq, qpos, n_tiles, m_used, l, ok);
      J0 += n_tiles;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// q [T, H, 192] bf16 -> head-major [H, T, 192] with q_nope (columns 0-127)
// rounded to fp16 (exact for bf16 values within fp16's range) and q_pe
// copied: one warp per (token, head) row, 24 lanes x 16 bytes, reads and
// writes both 384 contiguous bytes.
__global__ void __launch_bounds__(256) prepare_q_kernel(const uint4 *__restrict__ q,
                                                        uint4 *__restrict__ qh, int T, int H,
                                                        int32_t *status) {
  const int64_t rows = int64_t(T) * H;
  const int lane = threadIdx.x & 31;
  float amax = 0.f;  // largest q_nope magnitude converted (fp16 range check)
  for (int64_t r = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < rows;
       r += (int64_t(gridDim.x) * blockDim.x) >> 5) {
    if (lane >= DQK / 8) continue;
    const int64_t t = r / H, h = r - t * H;
    uint4 x = __ldg(q + r * (DQK / 8) + lane);
    if (lane < DN / 8) x = bf16x8_to_f16x8(x, amax);
    qh[(h * T + t) * (DQK / 8) + lane] = x;
  }
  if (status && amax >= kF16Overflow) atomicOr(status, MLA_STATUS_FP16_RANGE);
}

// LSE merge of the key splits of one (sequence, query tile, head) -- the
// merge the epilogue applies between its two warpgroups, over n partials --
// then written, or merged into the stored partial of a continued request,
// exactly as an unsplit CTA's epilogue does.  One warp per query row, a
// lane per 4 of the 128 output columns.
struct SplitGroups {
  int n, H, T;
  const int32_t *q_loc, *acc;
  const float *split_o, *split_lse;
  float *o, *lse;
  int4 g[MAX_SPLIT_GROUPS];  // (sequence, query tile, first slot, number of slots)
};

__global__ void __launch_bounds__(256) split_combine_kernel(const __grid_constant__ SplitGroups a) {
  const int gw = int((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  const int row = gw % BQ, gh = gw / BQ;
  if (gh >= a.n * a.H) return;
  const int h = gh % a.H;
  const int4 g = a.g[gh / a.H];
  const int q_beg = __ldg(a.q_loc + g.x), nq = __ldg(a.q_loc + g.x + 1) - q_beg;
  const int qpos = g.y * BQ + row;
  if (qpos >= nq) return;
  const int t = q_beg + qpos;
  // every split's LSE, then the splits' O rows four at a time: the loads of
  // a round are independent (indices past the last split repeat it), so
  // they are in flight together instead of one slot's after the other's
  auto slot_row = [&](int k) {
    return (int64_t(g.z + min(k, g.w - 1)) * a.H + h) * BQ + row;
  };
  float ls[MAX_GROUP_SPLITS];
  float m = neg_inf();
#pragma unroll
  for (int k = 0; k < MAX_GROUP_SPLITS; ++k) {
    ls[k] = k < g.w ? __ldg(a.split_lse + slot_row(k)) : neg_inf();
    m = fmaxf(m, ls[k]);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
  if (!is_neg_inf(m)) {
#pragma unroll
    for (int k0 = 0; k0 < MAX_GROUP_SPLITS; k0 += 4) {
      if (k0 >= g.w) break;
      float4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        v[i] = __ldg(reinterpret_cast<const float4 *>(a.split_o + slot_row(k0 + i) * DV) + lane);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // an empty split (and a repeated index) is never used
        if (is_neg_inf(ls[k0 + i])) continue;
        const float w = expf(ls[k0 + i] - m);
        l += w;
        acc.x += w * v[i].x;
        acc.y += w * v[i].y;
        acc.z += w * v[i].z;
        acc.w += w * v[i].w;
      }
    }
  }
  float lse = (l > 0.f) ? m + logf(l) : neg_inf();
  float w_new = (l > 0.f) ? 1.f / l : 0.f, w_old = 0.f;
  const int64_t li = int64_t(h) * a.T + t;
  float *orow = a.o + (int64_t(t) * a.H + h) * DV;
  const bool accumulate = a.acc != nullptr && __ldg(a.acc + g.x) != 0;
  if (accumulate) {
    const float old = a.lse[li];
    if (l == 0.f) return;  // nothing new: keep the stored partial
    if (!is_neg_inf(old)) {
      const float m2 = fmaxf(old, lse);
      const float eo = expf(old - m2), en = expf(lse - m2);
      w_old = eo / (eo + en);
      w_new *= en / (eo + en);
      lse = m2 + logf(eo + en);
    }
  }
  float4 o4 = make_float4(acc.x * w_new, acc.y * w_new, acc.z * w_new, acc.w * w_new);
  if (w_old != 0.f) {
    const float4 old = reinterpret_cast<const float4 *>(orow)[lane];
    o4.x += w_old * old.x;
    o4.y += w_old * old.y;
    o4.z += w_old * old.z;
    o4.w += w_old * old.w;
  }
  __syncwarp();  // every lane has read the stored LSE before lane 0 rewrites it
  reinterpret_cast<float4 *>(orow)[lane] = o4;
  if (lane == 0) a.lse[li] = lse;
}

// Work items of one launch: (sequence, query tile, key tiles [kt0, kt1),
// split slot or -1), the most key tiles first.  When the units (items x
// heads) are too few to fill the GPU (a long request with few queries), the
// longest items are split over their keys, at least kMinSplitTiles key
// tiles a split, into scratch slots that split_combine_kernel merges.
struct Item {
  int seq, qt, kt0, kt1, slot;
};
constexpr int kMinSplitTiles = 16;
// launches whose items average at most this many key tiles run on the
// looping kernel (one CTA per SM walking its units); with prepared queries
// (no conversion on the unit's path) up to kLoopTilesPrepared: there the
// overlap of one unit's epilogue with the next unit's work is worth more
// than the one-unit kernel's split rows (4 x 2048 causal new tokens with the
// final merge: 0.96 against 1.10 ms)
constexpr int kLoopTiles = 4;
constexpr int kLoopTilesPrepared = 16;
// the persistent one-unit kernel: launches of prepared queries with at
// least this many units per SM, and at most this many key tiles per unit on
// average (longer units hide a CTA's start and end themselves, and a CTA
// per unit lets the hardware even out the last wave: 4 x 2048 x 65536 took
// 28.96-29.16 ms persistent against 28.56-28.58 ms)
constexpr int kPersistUnits = 2;
constexpr int kPersistTiles = 64;

// A unit's cost beyond its key tiles (its Q tile and its partial's store,
// about two key tiles of traffic), for the balance estimate below.
constexpr int kUnitCostTiles = 2;

// The load of the busiest of G CTAs, in key tiles, when a launch's units
// (unit u: item u % n of head u / n) are dealt to them round robin -- as
// the persistent kernels walk them, and about as the hardware deals a CTA
// per unit to SMs that each hold one.
int64_t busiest_cta(const std::vector<Item> &items, int H, int G) {
  const size_t n = items.size();
  const int64_t units = int64_t(n) * H;
  std::vector<int64_t> load(size_t(G), 0);
  size_t i = 0, c = 0;
  for (int64_t u = 0; u < units; ++u) {
    load[c] += items[i].kt1 - items[i].kt0 + kUnitCostTiles;
    if (++i == n) i = 0;
    if (++c == size_t(G)) c = 0;
  }
  return *std::max_element(load.begin(), load.end());
}

int plan_items(int causal, int num_seqs, const int32_t *q_loc_host, const int32_t *k_loc_host,
               int H, const SplitScratch *split, bool skip_keyless, bool new_keys,
               std::vector<Item> &items, SplitGroups &sg) {
  auto by_cost = [](const Item &a, const Item &b) { return a.kt1 - a.kt0 > b.kt1 - b.kt0; };
  items.clear();
  sg.n = 0;
  for (int i = 0; i < num_seqs; ++i) {
    const int nq = q_loc_host[i + 1] - q_loc_host[i];
    const int nk = k_loc_host[i + 1] - k_loc_host[i];
    if ((nq + BQ - 1) / BQ > 0xffff) return MLA_ERR_UNSUPPORTED;  // 16-bit tile index
    if (skip_keyless && !new_keys && nk == 0) continue;  // its rows already hold O=0, LSE=-inf
    for (int qt = 0; qt * BQ < nq; ++qt) {
      int tiles = (nk + BKV - 1) / BKV;
      if (causal) tiles = std::min(tiles, qt + 1);
      // then the new tokens' keys up to the tile's last query
      if (new_keys) tiles += std::min((nq + BKV - 1) / BKV, qt + 1);
      items.push_back({i, qt, 0, tiles, -1});
    }
  }
  std::stable_sort(items.begin(), items.end(), by_cost);
  if (new_keys) return MLA_OK;  // never split
  const int64_t units = int64_t(items.size()) * H;
  if (split && split->o && !causal && units > 0 && units < split->target_ctas) {
    // at least `want` splits an item, so that the units reach the target;
    // beyond it, the split count whose units spread most evenly over the
    // SMs (the long request's 99 x 32768 chunk over 128 heads: 5 splits put
    // 5 units on 32 SMs and 4 on the rest, 7 splits 6 and 5)
    const int want0 = int((split->target_ctas + units - 1) / units);
    const int G = num_sms();
    std::vector<Item> best;
    SplitGroups best_sg = sg;
    int64_t best_load = -1;
    for (int want = want0; want <= std::max(want0, split->slots); ++want) {
      std::vector<Item> out;
      SplitGroups g = sg;
      int used = 0;
      for (const Item &it : items) {
        const int nt = it.kt1 - it.kt0;
        const int f = std::min({want, nt / kMinSplitTiles, MAX_GROUP_SPLITS});
        if (f < 2 || used + f > split->slots || g.n == MAX_SPLIT_GROUPS) {
          out.push_back(it);
          continue;
        }
        g.g[g.n++] = make_int4(it.seq, it.qt, used, f);
        for (int k = 0; k < f; ++k)
          out.push_back({it.seq, it.qt, it.kt0 + nt * k / f, it.kt0 + nt * (k + 1) / f, used + k});
        used += f;
      }
      std::stable_sort(out.begin(), out.end(), by_cost);
      const int64_t load = busiest_cta(out, H, G);
      if (best_load < 0 || load < best_load) {
        best.swap(out);
        best_sg = g;
        best_load = load;
      }
    }
    items.swap(best);
    sg = best_sg;
  }
  return MLA_OK;
}

}  // namespace

bool tc_attn_ok(const mla_dims_t &d, int kv_dtype, int64_t latent_ld) {
  return d.dtype == MLA_DTYPE_BF16 && kv_dtype == MLA_DTYPE_F16 && d.qk_nope_dim == DN &&
         d.qk_rope_dim == DR &&
         d.v_dim == DV && d.kv_lora_rank == 512 && (latent_ld * 2) % 16 == 0 &&
         latent_ld >= 576;
}

namespace {
// Many short units: one CTA per SM walks them (the next unit's loads and S
// MMAs overlapping this one's softmax and epilogue); otherwise a CTA per
// unit, so that a kernel running beside this one gets SMs as they retire.
bool takes_loop(int n_items, int64_t tiles, int H, bool q_prepared) {
  const int loop_tiles = q_prepared ? kLoopTilesPrepared : kLoopTiles;
  return int64_t(n_items) * H > num_sms() && tiles <= int64_t(loop_tiles) * n_items;
}
// Otherwise, with prepared queries, at least kPersistUnits units per SM and
// at most kPersistTiles key tiles per unit on average: one CTA per SM walks
// them, the next unit's loads and first S products overlapping this one's
// last tiles and epilogue.
bool takes_persist(int n_items, int64_t tiles, int H, bool q_prepared) {
  return q_prepared && int64_t(n_items) * H >= int64_t(kPersistUnits) * num_sms() &&
         tiles <= int64_t(kPersistTiles) * n_items;
}
}  // namespace

bool attn_tc_new_keys_ok(int num_seqs, const int32_t *q_loc_host, const int32_t *k_loc_host,
                         int H) {
  std::vector<Item> items;
  SplitGroups sg{};
  if (plan_items(0, num_seqs, q_loc_host, k_loc_host, H, nullptr, false, true, items, sg) ||
      items.empty() || items.size() > size_t(MAX_ITEMS))
    return false;
  int64_t tiles = 0;
  for (const Item &it : items) tiles += it.kt1 - it.kt0;
  return takes_loop(int(items.size()), tiles, H, true) ||
         takes_persist(int(items.size()), tiles, H, true);
}

int launch_attn_tc(const mla_dims_t &d, int causal, int num_seqs, const int32_t *q_loc,
                   const int32_t *k_loc, const int32_t *q_loc_host, const int32_t *k_loc_host,
                   int T, int kv_rows, const void *q, const void *kv, const void *latent,
                   int64_t latent_ld, const int32_t *accumulate, float *o, float *lse,
                   void *final_out, float *final_lse, int final_dtype, int pnt,
                   const SplitScratch *split, bool skip_keyless, bool q_prepared,
                   int32_t *status, cudaStream_t s, const NewKeySource *new_keys) {
  auto al16 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
  if (!al16(q) || !al16(kv) || !al16(latent)) return MLA_ERR_UNSUPPORTED;
  // new keys: the looping or the persistent kernel, non-causal context keys,
  // prepared queries (checked by attn_tc_new_keys_ok before the caller
  // commits to it)
  if (new_keys && (causal || !q_prepared || !al16(new_keys->kv) || !al16(new_keys->latent) ||
                   (new_keys->latent_ld * 2) % 16 != 0 || new_keys->latent_ld < 576))
    return MLA_ERR_UNSUPPORTED;
  const int H = d.num_heads;
  const int rows = k_loc_host[num_seqs];
  CUtensorMap tq, tkv, tlat;
  const bool tq_ok =
      q_prepared
          ? make_tmap_2d_16(&tq, false, q, DQK, uint64_t(H) * T, uint64_t(DQK) * 2, 64, 128, true)
          : make_tmap_2d_16(&tq, false, q, uint64_t(H) * DQK, uint64_t(T), uint64_t(H) * DQK * 2,
                            64, 128, true);
  if (!tq_ok ||
      !make_tmap_3d_16(&tkv, true, kv, HD, uint64_t(kv_rows > 0 ? kv_rows : 1), uint64_t(H),
                       uint64_t(HD) * 2, uint64_t(kv_rows > 0 ? kv_rows : 1) * HD * 2, 64, BKV,
                       true) ||
      !make_tmap_2d_16(&tlat, false, latent, 576, uint64_t(rows > 0 ? rows : 1),
                       uint64_t(latent_ld) * 2, 64, BKV, true))
    return MLA_ERR_CUDA;
  // the new tokens' K/V and latent rows (T of them), else copies of the
  // context maps that no tile reads
  CUtensorMap tkv2 = tkv, tlat2 = tlat;
  if (new_keys &&
      (!make_tmap_3d_16(&tkv2, true, new_keys->kv, HD, uint64_t(T), uint64_t(H),
                        uint64_t(HD) * 2, uint64_t(T) * HD * 2, 64, BKV, true) ||
       !make_tmap_2d_16(&tlat2, false, new_keys->latent, 576, uint64_t(T),
                        uint64_t(new_keys->latent_ld) * 2, 64, BKV, true)))
    return MLA_ERR_CUDA;
  std::vector<Item> items;
  SplitGroups sg{};
  const int rc = plan_items(causal, num_seqs, q_loc_host, k_loc_host, H,
                            final_out == nullptr && !new_keys ? split : nullptr,
                            skip_keyless && !causal && final_out == nullptr, new_keys != nullptr,
                            items, sg);
  if (rc) return rc;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES1) != cudaSuccess ||
        cudaFuncSetAttribute(attn_tc_loop_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES_LOOP) != cudaSuccess ||
        cudaFuncSetAttribute(attn_tc_persist_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES2) != cudaSuccess)
      return MLA_ERR_CUDA;
    attr_set = true;
  }
  thread_local AttnParams prm;  // large (24 KB); filled per launch batch
  for (size_t b = 0; b < items.size(); b += MAX_ITEMS) {
    const int n = int(std::min<size_t>(MAX_ITEMS, items.size() - b));
    prm.n_items = n;
    prm.H = H;
    prm.T = T;
    prm.causal = causal;
    prm.scale_log2 = d.softmax_scale * 1.4426950408889634f;
    prm.q_loc = q_loc;
    prm.k_loc = k_loc;
    prm.acc = accumulate;
    prm.o = o;
    prm.lse = lse;
    prm.fout = final_out;
    prm.flse = final_lse;
    prm.pnt = pnt;
    prm.fout_bf16 = final_dtype == MLA_DTYPE_BF16 ? 1 : 0;
    prm.split_o = split ? split->o : nullptr;
    prm.split_lse = split ? split->lse : nullptr;
    prm.q_prepared = q_prepared ? 1 : 0;
    prm.status = status;
    prm.new_keys = new_keys ? 1 : 0;
    for (int k = 0; k < n; ++k) {
      const Item &it = items[b + k];
      prm.items[k] = make_int4(it.seq, it.qt | ((it.slot + 1) << 16), it.kt0, it.kt1);
    }
    int64_t tiles = 0;
    for (int k = 0; k < n; ++k) tiles += items[b + k].kt1 - items[b + k].kt0;
    const bool loop = takes_loop(n, tiles, H, q_prepared);
    const bool persist = !loop && takes_persist(n, tiles, H, q_prepared);
    // only the looping and the persistent kernel take new keys
    if (new_keys && !loop && !persist) return MLA_ERR_UNSUPPORTED;
    launch_begin(s);
    if (loop)
      attn_tc_loop_kernel<<<num_sms(), THREADS_LOOP, SMEM_BYTES_LOOP, s>>>(tq, tkv, tlat, tkv2,
                                                                           tlat2, prm);
    else if (persist)
      attn_tc_persist_kernel<<<num_sms(), THREADS1, SMEM_BYTES2, s>>>(tq, tkv, tlat, tkv2, tlat2,
                                                                      prm);
    else
      attn_tc_kernel<<<n * H, THREADS1, SMEM_BYTES1, s>>>(tq, tkv, tlat, prm);
    const int rc = launch_status(
        s, loop ? "attn_tc_loop_kernel" : (persist ? "attn_tc_persist_kernel" : "attn_tc_kernel"));
    if (rc) return rc;
  }
  if (sg.n > 0) {
    sg.H = H;
    sg.T = T;
    sg.q_loc = q_loc;
    sg.acc = accumulate;
    sg.split_o = split->o;
    sg.split_lse = split->lse;
    sg.o = o;
    sg.lse = lse;
    const int64_t warps = int64_t(sg.n) * H * BQ;
    launch_begin(s);
    split_combine_kernel<<<int((warps * 32 + 255) / 256), 256, 0, s>>>(sg);
    return launch_status(s, "split_combine_kernel");
  }
  return MLA_OK;
}

int launch_prepare_q(const void *q, void *qh, int T, int H, int32_t *status, cudaStream_t s) {
  if (T == 0) return MLA_OK;
  const int64_t warps = int64_t(T) * H;
  int64_t blocks = (warps * 32 + 255) / 256;
  const int64_t cap = int64_t(num_sms()) * 16;
  if (blocks > cap) blocks = cap;
  launch_begin(s);
  prepare_q_kernel<<<int(blocks), 256, 0, s>>>(static_cast<const uint4 *>(q),
                                               static_cast<uint4 *>(qh), T, H, status);
  return launch_status(s, "prepare_q_kernel");
}

// The key-split merge on its own, for launches that cut (sequence, query
// tile, head) units elsewhere (the fused kernel): groups are (sequence, query
// tile, first slot, number of slots).
int launch_split_combine(int n_groups, const int4 *groups, int H, int T, const int32_t *q_loc,
                         const int32_t *acc, const SplitScratch &split, float *o, float *lse,
                         cudaStream_t s) {
  if (n_groups <= 0) return MLA_OK;
  if (n_groups > MAX_SPLIT_GROUPS) return MLA_ERR_UNSUPPORTED;
  SplitGroups sg{};
  sg.n = n_groups;
  sg.H = H;
  sg.T = T;
  sg.q_loc = q_loc;
  sg.acc = acc;
  sg.split_o = split.o;
  sg.split_lse = split.lse;
  sg.o = o;
  sg.lse = lse;
  for (int k = 0; k < n_groups; ++k) {
    if (groups[k].w < 0 || groups[k].w > MAX_GROUP_SPLITS) return MLA_ERR_UNSUPPORTED;
    sg.g[k] = groups[k];
  }
  const int64_t warps = int64_t(n_groups) * H * BQ;
  launch_begin(s);
  split_combine_kernel<<<int((warps * 32 + 255) / 256), 256, 0, s>>>(sg);
  return launch_status(s, "split_combine_kernel");
}

int attn_take_errors() { return sm103::take_error_flags_here(); }

}  // namespace mla
