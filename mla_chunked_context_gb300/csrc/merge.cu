// LSE-weighted merge of two partial attention results, with the
// prefix_num_tokens pass-through (PR #36540 report, "implementation
// breakdown", CUDA kernel layer), the empty-side rules of the PR #49294
// report (an empty side carries LSE=-inf and O=0; both empty gives O=0
// without NaN), and the two fills of context-free rows (PR #50613 report,
// item 3 init_mla_context_partial; PR #49294 report, mask_empty_context).
//
// HBM-bound.  One thread moves 8 elements (16 B of bf16 / 32 B of fp32) of a
// (token, head) row; consecutive threads cover consecutive 16-byte pieces of
// O [T, H, D], so every O access is a coalesced 16-byte vector.  A side's O
// is loaded only when that side is needed (its LSE finite and the token below
// prefix_num_tokens), so garbage or NaN in an unused side is never read into
// arithmetic and its bytes never move.
#include <algorithm>

#include "common.cuh"

namespace mla {
namespace {

struct Vec8 {
  float v[8];
};

__device__ __forceinline__ Vec8 load8(const float *p) {
  const float4 a = __ldcs(reinterpret_cast<const float4 *>(p));
  const float4 b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
  return Vec8{{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w}};
}

__device__ __forceinline__ Vec8 load8(const __nv_bfloat16 *p) {
  const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(p));
  Vec8 r;
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    r.v[2 * i] = __uint_as_float(w[i] << 16);
    r.v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
  return r;
}

__device__ __forceinline__ void store8(float *p, const Vec8 &x) {
  __stcs(reinterpret_cast<float4 *>(p), make_float4(x.v[0], x.v[1], x.v[2], x.v[3]));
  __stcs(reinterpret_cast<float4 *>(p) + 1, make_float4(x.v[4], x.v[5], x.v[6], x.v[7]));
}

__device__ __forceinline__ void store8(__nv_bfloat16 *p, const Vec8 &x) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x.v[2 * i], x.v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t *>(&h);
  }
  __stcs(reinterpret_cast<uint4 *>(p), make_uint4(w[0], w[1], w[2], w[3]));
}

// Piece index math in 32 bits (Idx = uint32_t) when T*H*(D/8) fits, else 64
// bits, and with shifts when D/8 and H are powers of two (kPow2): integer
// division is a long instruction sequence, 64-bit division several times
// longer, and this kernel issues it once per 16-byte piece (32-bit indices
// took the 8192 x 128 x 128 case from 131.7 to 127.6 us).
template <typename TI, typename TO, typename Idx, bool kPow2>
__global__ void __launch_bounds__(256) merge_kernel(
    TO *out, float *__restrict__ out_lse, const TI *prefix_o,
    const float *__restrict__ prefix_lse, const TI *suffix_o,
    const float *__restrict__ suffix_lse, int T, int H, int D, int pnt, int vpr_log2,
    int h_log2) {
  const Idx vpr = Idx(D >> 3);  // 8-element pieces per (token, head) row
  const Idx total = Idx(T) * Idx(H) * vpr;
  const Idx stride = Idx(gridDim.x) * blockDim.x;
  for (Idx i = Idx(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const Idx row = kPow2 ? (i >> vpr_log2) : i / vpr;
    const int piece = int(i - row * vpr);
    const Idx tt = kPow2 ? (row >> h_log2) : row / Idx(H);
    const int t = int(tt), h = int(row - tt * Idx(H));
    const int64_t off = int64_t(row) * D + int64_t(piece) * 8;
    const int64_t li = int64_t(h) * T + t;
    Vec8 r;
    float lse;
    const float sl = suffix_lse[li];
    if (t >= pnt) {
      r = load8(suffix_o + off);
      lse = sl;
    } else {
      const float pl = prefix_lse[li];
      const bool pe = is_neg_inf(pl), se = is_neg_inf(sl);
      if (pe && se) {
#pragma unroll
        for (int k = 0; k < 8; ++k) r.v[k] = 0.f;
        lse = neg_inf();
      } else if (pe) {
        r = load8(suffix_o + off);
        lse = sl;
      } else if (se) {
        r = load8(prefix_o + off);
        lse = pl;
      } else {
        const float m = fmaxf(pl, sl);
        const float a = expf(pl - m), b = expf(sl - m);
        const float inv = 1.f / (a + b);
        const float wa = a * inv, wb = b * inv;
        const Vec8 x = load8(prefix_o + off), y = load8(suffix_o + off);
#pragma unroll
        for (int k = 0; k < 8; ++k) r.v[k] = wa * x.v[k] + wb * y.v[k];
        lse = m + logf(a + b);
      }
    }
    store8(out + off, r);
    if (out_lse != nullptr && piece == 0) out_lse[li] = lse;
  }
}

__global__ void fill_empty_rows_kernel(float *__restrict__ o, float *__restrict__ lse,
                                       int T, int H, int Dv,
                                       const int32_t *__restrict__ slices) {
  const int lo = slices[2 * blockIdx.y], hi = slices[2 * blockIdx.y + 1];
  const int64_t n_o = int64_t(hi - lo) * H * Dv;
  const int64_t base = int64_t(lo) * H * Dv;
  if ((Dv & 3) == 0 && (reinterpret_cast<uintptr_t>(o) & 15) == 0) {
    // 16-byte stores: the slice's rows are one contiguous block
    float4 *o4 = reinterpret_cast<float4 *>(o + base);
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_o / 4;
         i += int64_t(gridDim.x) * blockDim.x)
      o4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_o;
         i += int64_t(gridDim.x) * blockDim.x)
      o[base + i] = 0.f;
  }
  const int64_t n_l = int64_t(hi - lo) * H;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_l;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int h = int(i / (hi - lo)), t = lo + int(i - int64_t(h) * (hi - lo));
    lse[int64_t(h) * T + t] = neg_inf();
  }
}

template <typename TO>
__global__ void mask_empty_context_kernel(float *__restrict__ lse, TO *__restrict__ o,
                                          int T, int H, int D, int R,
                                          const int32_t *__restrict__ qsl,
                                          const int32_t *__restrict__ csl) {
  // one warp per token: find the owning request, then clear its rows
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const int r = find_seq(qsl, R, warp);
  if (csl[r + 1] - csl[r] != 0) return;
  const int64_t n = int64_t(H) * D;
  for (int64_t i = lane; i < n; i += 32) o[int64_t(warp) * n + i] = from_f32<TO>(0.f);
  for (int h = lane; h < H; h += 32) lse[int64_t(h) * T + warp] = neg_inf();
}

int grid_for(int64_t work, int threads) {
  const int64_t need = (work + threads - 1) / threads;
  const int64_t cap = int64_t(num_sms()) * 8;
  return int(need < cap ? (need > 0 ? need : 1) : cap);
}

}  // namespace

int launch_merge(void *out, float *out_lse, const void *prefix_o, const float *prefix_lse,
                 const void *suffix_o, const float *suffix_lse, int T, int H, int D,
                 int pnt, int in_dtype, int out_dtype, cudaStream_t s) {
  const int64_t work = int64_t(T) * H * (D / 8);
  const int grid = grid_for(work, 256);
  // 32-bit piece indices while they and the grid stride fit; shifts when
  // D/8 and H are powers of two
  const bool small = work + int64_t(grid) * 256 < (int64_t(1) << 32);
  const int vpr = D / 8;
  const bool pow2 = (vpr & (vpr - 1)) == 0 && (H & (H - 1)) == 0;
  const int vl = __builtin_ctz(unsigned(vpr)), hl = __builtin_ctz(unsigned(H));
  launch_begin(s);
#define MLA_MERGE_K(TI, TO, IDX, P2)                                                   \
  merge_kernel<TI, TO, IDX, P2><<<grid, 256, 0, s>>>(                                  \
      static_cast<TO *>(out), out_lse, static_cast<const TI *>(prefix_o), prefix_lse,  \
      static_cast<const TI *>(suffix_o), suffix_lse, T, H, D, pnt, vl, hl)
#define MLA_MERGE(TI, TO)                                                              \
  do {                                                                                 \
    if (small && pow2)                                                                 \
      MLA_MERGE_K(TI, TO, uint32_t, true);                                             \
    else if (small)                                                                    \
      MLA_MERGE_K(TI, TO, uint32_t, false);                                            \
    else                                                                               \
      MLA_MERGE_K(TI, TO, uint64_t, false);                                            \
  } while (0)
  if (in_dtype == MLA_DTYPE_BF16 && out_dtype == MLA_DTYPE_BF16)
    MLA_MERGE(__nv_bfloat16, __nv_bfloat16);
  else if (in_dtype == MLA_DTYPE_BF16)
    MLA_MERGE(__nv_bfloat16, float);
  else if (out_dtype == MLA_DTYPE_BF16)
    MLA_MERGE(float, __nv_bfloat16);
  else
    MLA_MERGE(float, float);
#undef MLA_MERGE
#undef MLA_MERGE_K
  return launch_status(s, "merge_kernel");
}

int launch_fill_empty_rows(float *o, float *lse, int T, int H, int Dv, int num_slices,
                           const int32_t *slices, cudaStream_t s) {
  if (num_slices == 0) return MLA_OK;
  // about four blocks per SM over all slices
  const int per_slice = std::max(4, std::min(256, 4 * num_sms() / num_slices));
  dim3 grid(per_slice, num_slices);
  launch_begin(s);
  fill_empty_rows_kernel<<<grid, 256, 0, s>>>(o, lse, T, H, Dv, slices);
  return launch_status(s, "fill_empty_rows_kernel");
}

int launch_mask_empty_context(float *lse, void *o, int dtype, int T, int H, int D, int R,
                              const int32_t *qsl, const int32_t *csl, cudaStream_t s) {
  const int blocks = (T * 32 + 255) / 256;
  launch_begin(s);
  if (dtype == MLA_DTYPE_BF16)
    mask_empty_context_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
        lse, static_cast<__nv_bfloat16 *>(o), T, H, D, R, qsl, csl);
  else
    mask_empty_context_kernel<float><<<blocks, 256, 0, s>>>(
        lse, static_cast<float *>(o), T, H, D, R, qsl, csl);
  return launch_status(s, "mask_empty_context_kernel");
}

}  // namespace mla
