// CUDA-core kernels for MLA shapes the tensor-core kernels are not built for
// (any head dims, float32 or bf16 storage; e.g. a 64-rank latent with 32-wide
// heads).  Arithmetic is float32 throughout.
//
//  * kv_up_proj_simt: kv[h, row, c] = latent[row, 0:L] . w_kv_b[h*hd + c, :],
//    head-major [H, rows, hd]; a 64x64-tile shared-memory GEMM (each thread
//    4x4 outputs).
//  * attn_simt: one warp per (query token, head); online softmax over the
//    sequence's keys in the base-2 domain, O accumulated in registers spread
//    over the lanes; result (O, LSE) written or LSE-merged into the partial.
#include "common.cuh"

namespace mla {
namespace {

constexpr int GT = 64, GK = 16;

template <typename T, typename TO>
__global__ void __launch_bounds__(256) kv_up_proj_simt(const T *__restrict__ A, int64_t lda,
                                                       const T *__restrict__ B, TO *__restrict__ C,
                                                       int M, int N, int K, int hd,
                                                       int32_t *status) {
  __shared__ float As[GK][GT + 1];
  __shared__ float Bs[GK][GT + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * GT, n0 = blockIdx.x * GT;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += GK) {
    for (int e = threadIdx.x; e < GT * GK; e += 256) {
      const int r = e / GK, k = e % GK;
      const int gm = m0 + r, gn = n0 + r, gk = k0 + k;
      As[k][r] = (gm < M && gk < K) ? to_f32(A[int64_t(gm) * lda + gk]) : 0.f;
      Bs[k][r] = (gn < N && gk < K) ? to_f32(B[int64_t(gn) * K + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < GK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[k][ty + 16 * i];
        b[i] = Bs[k][tx + 16 * i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float amax = 0.f;  // largest magnitude written (fp16 output: range check)
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gm = m0 + ty + 16 * i, gn = n0 + tx + 16 * j;
      // head-major output [N / hd, M, hd]
      if (gm < M && gn < N) {
        C[(int64_t(gn / hd) * M + gm) * hd + gn % hd] = from_f32<TO>(acc[i][j]);
        amax = fmaxf(amax, fabsf(acc[i][j]));
      }
    }
  if (sizeof(TO) == 2 && !is_bf16<TO>() && amax >= kF16Overflow && status)
    atomicOr(status, MLA_STATUS_FP16_RANGE);
}

constexpr int QK_PER_LANE = 8;  // qk dim up to 256
constexpr int V_PER_LANE = 8;   // v dim up to 256

struct AttnArgs {
  const void *q;
  const void *kv;
  const void *latent;
  int64_t latent_ld;
  float *o;
  float *lse;
  const int32_t *q_loc;
  const int32_t *k_loc;
  const int32_t *accumulate;
  int num_seqs, T, H, L, P, Dn, Dv, causal;
  int kv_rows;       // rows of the head-major kv [H, kv_rows, Dn+Dv]
  float scale_log2;  // softmax_scale * log2(e)
};

template <typename T, typename TK>
__global__ void __launch_bounds__(128) attn_simt(AttnArgs a) {
  const int lane = threadIdx.x & 31;
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int first = a.q_loc[0];
  const int ntok = a.q_loc[a.num_seqs] - first;
  if (w >= ntok * a.H) return;
  const int t = first + w / a.H, h = w % a.H;
  const int i = find_seq(a.q_loc, a.num_seqs, t);
  const int kbeg = a.k_loc[i];
  int nk = a.k_loc[i + 1] - kbeg;
  if (a.causal) nk = min(nk, t - a.q_loc[i] + 1);
  const int QK = a.Dn + a.P, HDIM = a.Dn + a.Dv;
  const T *q = static_cast<const T *>(a.q) + (int64_t(t) * a.H + h) * QK;
  const TK *kv = static_cast<const TK *>(a.kv);
  const T *lat = static_cast<const T *>(a.latent);
  float qr[QK_PER_LANE], acc[V_PER_LANE];
#pragma unroll
  for (int e = 0; e < QK_PER_LANE; ++e) {
    const int d = lane + 32 * e;
    qr[e] = d < QK ? to_f32(q[d]) : 0.f;
  }
#pragma unroll
  for (int e = 0; e < V_PER_LANE; ++e) acc[e] = 0.f;
  float m = neg_inf(), l = 0.f;
  for (int j = 0; j < nk; ++j) {
    const int64_t row = kbeg + j;
    const TK *kn = kv + (int64_t(h) * a.kv_rows + row) * HDIM;
    const T *kp = lat + row * a.latent_ld + a.L;
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < QK_PER_LANE; ++e) {
      const int d = lane + 32 * e;
      if (d < a.Dn)
        s = fmaf(qr[e], to_f32(kn[d]), s);
      else if (d < QK)
        s = fmaf(qr[e], to_f32(kp[d - a.Dn]), s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    s *= a.scale_log2;
    const float mn = fmaxf(m, s);
    const float corr = exp2f(m - mn);  // m = -inf on the first key: 0
    const float p = exp2f(s - mn);
    l = l * corr + p;
#pragma unroll
    for (int e = 0; e < V_PER_LANE; ++e) {
      const int d = lane + 32 * e;
      const float v = d < a.Dv ? to_f32(kn[a.Dn + d]) : 0.f;
      acc[e] = fmaf(p, v, acc[e] * corr);
    }
    m = mn;
  }
  const float ln2 = 0.69314718055994531f;
  const int64_t li = int64_t(h) * a.T + t;
  float *o = a.o + (int64_t(t) * a.H + h) * a.Dv;
  float lse = l > 0.f ? (m + log2f(l)) * ln2 : neg_inf();
  float wn = l > 0.f ? 1.f / l : 0.f, wo = 0.f;
  if (a.accumulate && a.accumulate[i] && l > 0.f) {
    const float old = a.lse[li];
    if (!is_neg_inf(old)) {
      const float mx = fmaxf(old, lse);
      const float eo = expf(old - mx), en = expf(lse - mx);
      wo = eo / (eo + en);
      wn *= en / (eo + en);
      lse = mx + logf(eo + en);
    }
  } else if (a.accumulate && a.accumulate[i]) {
    return;  // nothing new for this row: keep the stored partial
  }
#pragma unroll
  for (int e = 0; e < V_PER_LANE; ++e) {
    const int d = lane + 32 * e;
    if (d < a.Dv) o[d] = (wo != 0.f ? wo * o[d] : 0.f) + wn * acc[e];
  }
  if (lane == 0) a.lse[li] = lse;
}

}  // namespace

bool generic_dims_ok(const mla_dims_t &d) {
  return d.qk_nope_dim + d.qk_rope_dim <= 32 * QK_PER_LANE && d.v_dim <= 32 * V_PER_LANE;
}

template <typename T>
int up_proj_simt_out(int kv_dtype, const T *latent, int64_t lda, int rows, const T *w, void *kv,
                     int N, int K, int hd, int32_t *status, dim3 grid, cudaStream_t s) {
  launch_begin(s);
  if (kv_dtype == MLA_DTYPE_F32)
    kv_up_proj_simt<T, float><<<grid, 256, 0, s>>>(latent, lda, w, static_cast<float *>(kv), rows,
                                                   N, K, hd, status);
  else if (kv_dtype == MLA_DTYPE_F16)
    kv_up_proj_simt<T, __half><<<grid, 256, 0, s>>>(latent, lda, w, static_cast<__half *>(kv),
                                                    rows, N, K, hd, status);
  else
    kv_up_proj_simt<T, __nv_bfloat16><<<grid, 256, 0, s>>>(
        latent, lda, w, static_cast<__nv_bfloat16 *>(kv), rows, N, K, hd, status);
  return launch_status(s, "kv_up_proj_simt");
}

int launch_up_proj_simt(int dtype, int kv_dtype, const void *latent, int64_t lda, int rows,
                        const void *w, void *kv, int N, int K, int hd, int32_t *status,
                        cudaStream_t s) {
  if (rows == 0) return MLA_OK;
  dim3 grid((N + GT - 1) / GT, (rows + GT - 1) / GT);
  if (dtype == MLA_DTYPE_BF16)
    return up_proj_simt_out(kv_dtype, static_cast<const __nv_bfloat16 *>(latent), lda, rows,
                            static_cast<const __nv_bfloat16 *>(w), kv, N, K, hd, status, grid, s);
  return up_proj_simt_out(kv_dtype, static_cast<const float *>(latent), lda, rows,
                          static_cast<const float *>(w), kv, N, K, hd, status, grid, s);
}

template <typename T>
void attn_simt_kv(int kv_dtype, int blocks, const AttnArgs &a, cudaStream_t s) {
  if (kv_dtype == MLA_DTYPE_F32)
    attn_simt<T, float><<<blocks, 128, 0, s>>>(a);
  else if (kv_dtype == MLA_DTYPE_F16)
    attn_simt<T, __half><<<blocks, 128, 0, s>>>(a);
  else
    attn_simt<T, __nv_bfloat16><<<blocks, 128, 0, s>>>(a);
}

int launch_attn_simt(const mla_dims_t &d, int causal, int num_seqs, const int32_t *q_loc,
                     const int32_t *k_loc, int num_q_rows, int T, int kv_rows, const void *q,
                     const void *kv, int kv_dtype, const void *latent, int64_t latent_ld,
                     const int32_t *accumulate, float *o, float *lse, cudaStream_t s) {
  if (num_q_rows == 0 || num_seqs == 0) return MLA_OK;
  AttnArgs a{q, kv, latent, latent_ld, o, lse, q_loc, k_loc, accumulate, num_seqs, T,
             d.num_heads, d.kv_lora_rank, d.qk_rope_dim, d.qk_nope_dim, d.v_dim, causal,
             kv_rows, d.softmax_scale * 1.4426950408889634f};
  const int64_t warps = int64_t(num_q_rows) * d.num_heads;
  const int blocks = int((warps * 32 + 127) / 128);
  launch_begin(s);
  if (d.dtype == MLA_DTYPE_BF16)
    attn_simt_kv<__nv_bfloat16>(kv_dtype, blocks, a, s);
  else
    attn_simt_kv<float>(kv_dtype, blocks, a, s);
  return launch_status(s, "attn_simt");
}

}  // namespace mla
