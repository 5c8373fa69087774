// tcgen05 decode index scan (bf16, index_dim 128, block 128, 4 index heads).
#pragma once
#include "common.cuh"

namespace msa {
bool index_scan_tc_supported(const Dims& p);
cudaError_t launch_index_scan_tc(const Dims& p, const void* idx_q, const void* idx_k,
                                 float* scores, cudaStream_t st, int* status);
}  // namespace msa
