// routing.cpp -- host-side batch routing: sort + group into the triple
// (lora_ids, grouped_offsets, end) of the "max.pipelines.lora.LoRAManagerV3"
// API page (sort_lora_batch, get_lora_graph_inputs).
//
// The sort is a counting sort over slot ids (stable by construction: each
// bucket is filled in arrival order), with the base bucket placed after every
// adapter bucket.  Grouping walks the sorted order and stops at the first
// base request.
#include <climits>
#include <cstdint>
#include <vector>

#include "../../include/lora_sgmv.h"

extern "C" lora_status_t lora_build_routing(int32_t num_requests, const int32_t* req_slot,
                                            const int32_t* req_num_tokens, int32_t max_num_loras,
                                            int32_t* perm, int32_t* lora_ids,
                                            int32_t* grouped_offsets, int32_t* num_groups,
                                            int32_t* end, int32_t* total_tokens) {
  if (num_requests < 0 || max_num_loras < 1) return LORA_ERR_SHAPE;
  if (!lora_ids || !grouped_offsets || !num_groups || !end || !total_tokens) return LORA_ERR_NULL;
  if (num_requests > 0 && (!req_slot || !req_num_tokens || !perm)) return LORA_ERR_NULL;

  int64_t total = 0;
  for (int32_t i = 0; i < num_requests; ++i) {
    const int32_t s = req_slot[i];
    if (s < -1 || s >= max_num_loras) return LORA_ERR_SLOT_RANGE;
    if (req_num_tokens[i] < 0) return LORA_ERR_SHAPE;
    total += req_num_tokens[i];
  }
  if (total > INT32_MAX) return LORA_ERR_SHAPE;

  // Bucket b = slot for adapters, b = max_num_loras for base requests.  The
  // table is only as large as the slots actually used by this batch would
  // need, so a huge max_num_loras with few requests does not allocate much.
  int32_t hi = -1;
  for (int32_t i = 0; i < num_requests; ++i)
    if (req_slot[i] > hi) hi = req_slot[i];
  const int32_t nb = hi + 2;  // adapter buckets 0..hi, base bucket hi+1
  std::vector<int32_t> start(static_cast<size_t>(nb) + 1, 0);
  for (int32_t i = 0; i < num_requests; ++i) {
    const int32_t b = req_slot[i] < 0 ? hi + 1 : req_slot[i];
    ++start[b + 1];
  }
  for (int32_t b = 0; b < nb; ++b) start[b + 1] += start[b];
  for (int32_t i = 0; i < num_requests; ++i) {
    const int32_t b = req_slot[i] < 0 ? hi + 1 : req_slot[i];
    perm[start[b]++] = i;
  }

  int32_t g = 0, row = 0;
  grouped_offsets[0] = 0;
  for (int32_t i = 0; i < num_requests; ++i) {
    const int32_t s = req_slot[perm[i]];
    if (s < 0) break;  // first base request: the triple stops here
    if (g == 0 || lora_ids[g - 1] != s) {
      lora_ids[g] = s;
      grouped_offsets[g] = row;
      ++g;
    }
    row += req_num_tokens[perm[i]];
    grouped_offsets[g] = row;
  }
  *num_groups = g;
  *end = row;
  *total_tokens = static_cast<int32_t>(total);
  return LORA_OK;
}

extern "C" lora_status_t lora_build_token_rows(int32_t num_requests, const int32_t* req_num_tokens,
                                               const int32_t* perm, int32_t end, int32_t* token_rows) {
  if (num_requests < 0 || end < 0) return LORA_ERR_SHAPE;
  if (end > 0 && !token_rows) return LORA_ERR_NULL;
  if (num_requests > 0 && (!req_num_tokens || !perm)) return LORA_ERR_NULL;
  // Row where each request starts, in arrival order.
  std::vector<int64_t> start(static_cast<size_t>(num_requests) + 1, 0);
  for (int32_t i = 0; i < num_requests; ++i) {
    if (req_num_tokens[i] < 0) return LORA_ERR_SHAPE;
    start[i + 1] = start[i] + req_num_tokens[i];
  }
  int32_t k = 0;
  for (int32_t i = 0; i < num_requests && k < end; ++i) {
    const int32_t r = perm[i];
    if (r < 0 || r >= num_requests) return LORA_ERR_SHAPE;
    for (int32_t t = 0; t < req_num_tokens[r] && k < end; ++t) token_rows[k++] = (int32_t)(start[r] + t);
  }
  return k == end ? LORA_OK : LORA_ERR_SHAPE;
}
