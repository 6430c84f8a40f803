// placeholder, replaced by the tcgen05 GEMM
#include "common.cuh"
namespace mla {
bool tc_available() { return false; }
bool tc_gemm_ok(const mla_dims_t &, int64_t, const void *, const void *, const void *) { return false; }
int launch_up_proj_tc(const mla_dims_t &, const void *, int64_t, int, const void *, void *, cudaStream_t) { return MLA_ERR_UNSUPPORTED; }
bool tc_attn_ok(const mla_dims_t &, int64_t) { return false; }
int launch_attn_tc(const mla_dims_t &, int, int, const int32_t *, const int32_t *, const int32_t *,
                   const int32_t *, int, const void *, const void *, const void *, int64_t,
                   const int32_t *, float *, float *, cudaStream_t) { return MLA_ERR_UNSUPPORTED; }
}
