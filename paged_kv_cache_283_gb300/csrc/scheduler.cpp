// Step planning for chunked prefill ("How LLM Inference Serving Works",
// section "Chunked prefill"): each step has a token budget; all pending
// decodes (one token each) are taken first, the remaining budget goes to the
// pending prefills in queue order, and a prefill that does not fit is cut to
// what is left.  With more decodes than the budget, the first `budget` decodes
// run and no prefill does.

#include <stdint.h>

#include "../../include/pa.h"

extern "C" pa_status pa_plan_step(int budget, int num_decodes, const int32_t* prefill_remaining,
                                  int num_prefills, int32_t* chunk_out, int* decodes_out) {
  if (budget < 0 || num_decodes < 0 || num_prefills < 0 || !decodes_out ||
      (num_prefills > 0 && (!prefill_remaining || !chunk_out)))
    return PA_ERR_INVALID_ARG;
  for (int i = 0; i < num_prefills; ++i)
    if (prefill_remaining[i] < 0) return PA_ERR_INVALID_ARG;
  const int decodes = num_decodes < budget ? num_decodes : budget;
  int64_t left = static_cast<int64_t>(budget) - decodes;
  for (int i = 0; i < num_prefills; ++i) {
    const int64_t take = prefill_remaining[i] < left ? prefill_remaining[i] : left;
    chunk_out[i] = static_cast<int32_t>(take);
    left -= take;
  }
  *decodes_out = decodes;
  return PA_OK;
}
