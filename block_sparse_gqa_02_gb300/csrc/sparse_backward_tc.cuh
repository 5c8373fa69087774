// tcgen05 backward of the sparse prefill attention (bf16, head_dim 128, block 128, 64-query
// tiles): a dQ kernel over query tiles and a dK/dV kernel over key blocks.
#pragma once
#include "common.cuh"

namespace msa {
bool sparse_backward_tc_supported(const Dims& p);
// scratch: a 1 KiB record per 128-row group (lse2 and D = dout . out of its rows), then the
// tile-selects-block bitmap
size_t sparse_backward_tc_workspace_bytes(const Dims& p);
cudaError_t launch_sparse_backward_tc(const Dims& p, const void* q, const void* k,
                                      const void* v, const int32_t* sel, const void* out,
                                      const float* lse, const void* dout, float* dq, float* dk,
                                      float* dv, void* workspace, cudaStream_t st, int* status);
// bit (sequence * Hkv + KV head, block, tile) set when that query tile selected that block:
// [B * Hkv, nB, ceil(nR / 32)] uint32, cleared then filled on the stream
cudaError_t launch_selection_bitmap(const Dims& p, const int32_t* sel, uint32_t* bits,
                                   cudaStream_t st);
// query tiles covered by one key-block CTA (a multiple of 32, at most 2048)
int tiles_per_cta(const Dims& p);
}  // namespace msa
