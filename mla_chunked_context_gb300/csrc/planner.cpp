// Host planner: packs each request's cached context into workspace-sized
// chunks (PR #50613 report, "implementation breakdown" item 2 and the key
// source snippet plan_mla_context_chunks / aligned_split_len).
//
// Requests are visited in order.  A request without context is in no chunk.
// Requests with context are appended to the open chunk while their padded
// rows fit the row budget.  The first one that does not fit is cut at the
// largest aligned length that fits (binary search over multiples of the
// alignment; the padded-row count is non-decreasing in the length) and the
// chunk closes.  If no aligned length fits, the chunk closes without it and
// the request opens the next chunk; appending it whole would overflow the
// workspace, which the page's invariants forbid.
#include <cstdint>
#include <vector>

#include "../../include/mla_chunked_context.h"
#include "planner.h"

namespace mla {

namespace {

struct Rows {
  int64_t (*fn)(int64_t, void *);
  void *ctx;
  int64_t operator()(int64_t x) const { return fn ? fn(x, ctx) : x; }
};

// Largest k*align with k*align <= min(max_chunk, floor((remaining-1)/align)*align)
// whose padded rows rows(start + k*align) - rows(start) fit in `available`.
int64_t split_len(const Rows &rows, int64_t start, int64_t remaining,
                  int64_t available, int64_t max_chunk, int64_t align) {
  int64_t cap = (remaining - 1) / align * align;
  if (max_chunk < cap) cap = max_chunk;
  int64_t lo = 0, hi = cap / align;
  const int64_t base = rows(start);
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) / 2;
    if (rows(start + mid * align) - base <= available)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo * align;
}

}  // namespace

int plan_chunks(const int32_t *context_lens, int32_t num_requests,
                int32_t row_budget, int32_t max_context_chunk,
                int32_t split_alignment, int64_t (*padded_rows)(int64_t, void *),
                void *padded_rows_ctx, std::vector<mla_chunk_t> &chunks,
                std::vector<int32_t> &starts, std::vector<int32_t> &seq_lens) {
  chunks.clear();
  starts.clear();
  seq_lens.clear();
  if (num_requests < 0 || row_budget < 1 || split_alignment < 1 ||
      max_context_chunk < 1)
    return MLA_ERR_INVALID;
  if (num_requests > 0 && !context_lens) return MLA_ERR_INVALID;
  for (int32_t r = 0; r < num_requests; ++r)
    if (context_lens[r] < 0) return MLA_ERR_INVALID;

  const Rows rows{padded_rows, padded_rows_ctx};
  int32_t req = 0;
  int64_t offset = 0;  // rows of the current request placed in earlier chunks
  while (req < num_requests) {
    if (context_lens[req] == 0) {
      if (offset != 0) return MLA_ERR_PLANNER_STUCK;
      ++req;
      continue;
    }
    mla_chunk_t c{};
    c.request_start = req;
    c.entry_offset = static_cast<int32_t>(starts.size());
    int64_t used = 0;
    while (req < num_requests && context_lens[req] > 0) {
      const int64_t left = context_lens[req] - offset;
      const int64_t need = rows(offset + left) - rows(offset);
      if (used + need <= row_budget) {
        starts.push_back(static_cast<int32_t>(offset));
        seq_lens.push_back(static_cast<int32_t>(left));
        used += need;
        ++req;
        offset = 0;
        continue;
      }
      const int64_t cut = split_len(rows, offset, left, row_budget - used,
                                    max_context_chunk, split_alignment);
      if (cut > 0) {
        starts.push_back(static_cast<int32_t>(offset));
        seq_lens.push_back(static_cast<int32_t>(cut));
        used += rows(offset + cut) - rows(offset);
        offset += cut;
      }
      break;
    }
    const int32_t n = static_cast<int32_t>(starts.size()) - c.entry_offset;
    if (n == 0) return MLA_ERR_PLANNER_STUCK;
    c.request_end = c.request_start + n;
    c.rows = static_cast<int32_t>(used);
    c.is_continuation = starts[c.entry_offset] > 0 ? 1 : 0;
    chunks.push_back(c);
  }
  return MLA_OK;
}

}  // namespace mla

extern "C" int mla_plan_context_chunks(
    const int32_t *context_lens, int32_t num_requests, int32_t row_budget,
    int32_t max_context_chunk, int32_t split_alignment,
    int64_t (*padded_rows)(int64_t, void *), void *padded_rows_ctx,
    mla_chunk_t *chunks, int32_t chunks_cap, int32_t *starts,
    int32_t *seq_lens, int32_t entries_cap, int32_t *num_chunks,
    int32_t *num_entries) {
  std::vector<mla_chunk_t> c;
  std::vector<int32_t> s, l;
  const int rc = mla::plan_chunks(context_lens, num_requests, row_budget,
                                  max_context_chunk, split_alignment,
                                  padded_rows, padded_rows_ctx, c, s, l);
  if (rc != MLA_OK) return rc;
  if (num_chunks) *num_chunks = static_cast<int32_t>(c.size());
  if (num_entries) *num_entries = static_cast<int32_t>(s.size());
  if (!chunks && !starts && !seq_lens) return MLA_OK;
  if (!chunks || !starts || !seq_lens) return MLA_ERR_INVALID;
  if (chunks_cap < static_cast<int32_t>(c.size()) ||
      entries_cap < static_cast<int32_t>(s.size()))
    return MLA_ERR_TOO_SMALL;
  for (size_t i = 0; i < c.size(); ++i) chunks[i] = c[i];
  for (size_t i = 0; i < s.size(); ++i) {
    starts[i] = s[i];
    seq_lens[i] = l[i];
  }
  return MLA_OK;
}
