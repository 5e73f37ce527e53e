// Internal declarations shared by the translation units of libpagedattn.
#pragma once
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/pagedattn.h"

// Rows of every tile-routine MMA (M): (query token, head-in-group) pairs of one KV head.
#define PA_ROWS 128

namespace pa_detail {

// Records a failed CUDA call for pa_last_cuda_error(); returns PA_OK or PA_ERR_CUDA.
int32_t note_cuda(cudaError_t e);
// Shape support check (see pa_shape in pagedattn.h).
int32_t check_shape(const pa_shape* s);
// cu_seqlens_q / ctx_lens consistency: cu[0] == 0, non-decreasing, 0 <= n_q <= ctx.
int32_t check_step_meta(int32_t B, const int32_t* cu, const int32_t* ctx);

}  // namespace pa_detail
