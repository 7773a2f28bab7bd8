// Internal host-side declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include "pa.h"

// Records a one-line description of the failure for pa_last_error().
void pa_set_error(const char* msg);
// pa_set_error(msg) and return `st`.
pa_status pa_fail(pa_status st, const char* msg);

// The kernel pa_decode_ex picks when pa_decode_opts.kernel is 0: 3
// head-packed tensor-core, 2 per-head tensor-core, 1 SIMT.
int pa_decode_auto_kernel(const pa_cache_desc& cache, int32_t num_heads, int32_t num_seqs,
                          int32_t tokens_per_seq);
