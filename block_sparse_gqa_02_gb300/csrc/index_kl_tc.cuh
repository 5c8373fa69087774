// tcgen05 KL loss of the index branch (bf16, head_dim = index_dim = 128, block 128, 64-query
// tiles, 2 <= G <= 32): a query-tile kernel (loss, d idx_q) and a key-block kernel (d idx_k).
#pragma once
#include "common.cuh"

namespace msa {
bool index_kl_tc_supported(const Dims& p);
// scratch: a 1 KiB record per 128-row group (main lse2 per row, index normaliser per token),
// then the bitmap of which tiles selected which blocks
size_t index_kl_tc_workspace_bytes(const Dims& p);
cudaError_t launch_index_kl_tc(const Dims& p, const void* q, const void* k, const float* lse,
                               const void* idx_q, const void* idx_k, const int32_t* sel,
                               float* loss, float* d_idx_q, float* d_idx_k, void* workspace,
                               cudaStream_t st, int* status);
}  // namespace msa
