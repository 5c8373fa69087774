// tcgen05 index-score kernel (bf16, index_dim 128, block 128, 64-query tiles, 4 heads).
#pragma once
#include "common.cuh"

namespace msa {
bool index_tc_supported(const Dims& p);
bool index_topk_fused_supported(const Dims& p);
// scores may be null when sel is given (fused top-k); sel null = scores only.
cudaError_t launch_index_scores_tc(const Dims& p, const void* idx_q, const void* idx_k,
                                   float* scores, int32_t* sel, cudaStream_t st, int* status);
}  // namespace msa
