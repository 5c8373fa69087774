// tcgen05 sparse-prefill kernel (bf16, head_dim 128, block 128, 64-query tiles).
#pragma once
#include "common.cuh"

namespace msa {
bool sparse_prefill_tc_supported(const Dims& p);
cudaError_t launch_sparse_prefill_tc(const Dims& p, const void* q, const void* k, const void* v,
                                     const int32_t* sel, void* out, float* lse, cudaStream_t st,
                                     int* status);
}  // namespace msa
