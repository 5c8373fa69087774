// Device-side validation of a call's index inputs, compiled in debug builds (-DMSA_DEBUG)
// only: the selection rows (every entry -1 or a block of the sequence, no block twice), the
// block table of a paged cache (every entry a physical block) and the cache lengths (within
// the table's capacity).  A failed check records a DebugCode in the device status word,
// which msa_get_device_status() reports as MSA_ERR_BOUNDS; nothing traps, and the kernels
// that follow skip out-of-range entries as they always do.
#include "common.cuh"

namespace msa {

#ifdef MSA_DEBUG
namespace {

// One thread per selection row; rows are [B, Hkv, nR, k].
__global__ void validate_sel_kernel(const int32_t* __restrict__ sel, Dims p, int* status) {
  const long long rows = (long long)p.B * p.Hkv * p.nR;
  for (long long row = blockIdx.x * (long long)blockDim.x + threadIdx.x; row < rows;
       row += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(row / ((long long)p.Hkv * p.nR));
    const int n_blocks = p.seq_lens ? (seq_len_of(p, b) + p.Bk - 1) / p.Bk : p.nB;
    const int32_t* r = sel + row * p.k;
    for (int i = 0; i < p.k; ++i) {
      const int e = r[i];
      debug_check(e >= -1 && e < n_blocks, status, kDbgSelRange);
      if (e < 0) continue;
      for (int j = 0; j < i; ++j) debug_check(r[j] != e, status, kDbgSelDuplicate);
    }
  }
}

// One thread per (sequence, logical block) of a paged cache, plus the lengths.
__global__ void validate_table_kernel(Dims p, int* status) {
  const long long n = (long long)p.B * p.nB;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(i / p.nB), j = (int)(i % p.nB);
    const int L = p.seq_lens[b];
    if (j == 0) debug_check(L >= 0 && L <= p.Sk, status, kDbgSeqLen);
    if (p.block_table && j < (seq_len_of(p, b) + p.Bk - 1) / p.Bk) {
      const int phys = p.block_table[i];
      debug_check(phys >= 0 && phys < p.n_phys, status, kDbgTableRange);
    }
  }
}

}  // namespace

cudaError_t launch_debug_validate(const Dims& p, const int32_t* sel, cudaStream_t st,
                                  int* status) {
  if (sel) {
    const long long rows = (long long)p.B * p.Hkv * p.nR;
    const int grid = (int)((rows + 255) / 256 < 1024 ? (rows + 255) / 256 : 1024);
    validate_sel_kernel<<<grid, 256, 0, st>>>(sel, p, status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.seq_lens) {
    const long long n = (long long)p.B * p.nB;
    const int grid = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    validate_table_kernel<<<grid, 256, 0, st>>>(p, status);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

#else

cudaError_t launch_debug_validate(const Dims&, const int32_t*, cudaStream_t, int*) {
  return cudaSuccess;
}

#endif

}  // namespace msa
