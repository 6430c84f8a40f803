// Internal declaration of the host planner shared by the C-ABI entry points.
#pragma once
#include <cstdint>
#include <vector>

#include "../../include/mla_chunked_context.h"

namespace mla {

int plan_chunks(const int32_t *context_lens, int32_t num_requests,
                int32_t row_budget, int32_t max_context_chunk,
                int32_t split_alignment, int64_t (*padded_rows)(int64_t, void *),
                void *padded_rows_ctx, std::vector<mla_chunk_t> &chunks,
                std::vector<int32_t> &starts, std::vector<int32_t> &seq_lens);

}  // namespace mla
