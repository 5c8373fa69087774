// Tensor-core (mma.sync) split-KV decode partials (bf16, head_dim 128, block 128, G <= 16).
#pragma once
#include "common.cuh"

namespace msa {
bool sparse_decode_mma_supported(const Dims& p);
cudaError_t launch_sparse_decode_mma(const Dims& p, const void* q, const void* k, const void* v,
                                     const int32_t* sel, float* ws_o, float* ws_l, int n_split,
                                     int per, cudaStream_t st, int* status);
}  // namespace msa
