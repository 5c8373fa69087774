// Internal declarations shared by the MSA kernels and the C-ABI layer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

namespace msa {

// Shape after validation, with the derived sizes every kernel needs.
struct Dims {
  int B, Sq, Sk, Hq, Hkv, G, d, dI, Bk, k, Qt;
  int nB;        // ceil(Sk / Bk): blocks per sequence
  int nR;        // ceil(Sq / Qt): selection rows per (sequence, KV head)
  int q_off;     // position of query 0 (0 for prefill, Sk - 1 for decode)
  int decode;    // 1 when Sq == 1 and Qt == 1
  int dtype;     // 0 f32, 1 bf16
  float sm_scale, index_scale;
  int inject;    // test hook: 1 = the tensor-core prefill producer issues no copies
  // paged decode (all null / 0 for contiguous caches): per-sequence cache lengths [B],
  // block table [B, nB] of physical block ids, and the number of physical blocks
  const int32_t* seq_lens;
  const int32_t* block_table;
  int n_phys;
};

// ------------------------------------------------------------ debug checks
// A build with -DMSA_DEBUG checks indices on the device: every selection entry, block-table
// entry and cache length a call receives (launch_debug_validate), and the coordinates the
// tensor-core kernels give their tensor copies.  A failed check records a code 0xBxx in the
// device status word (reported as MSA_ERR_BOUNDS; the kernels' timeout codes use other
// ranges) and never traps; release builds compile the checks away.
#ifdef MSA_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

constexpr int kDebugCodeBase = 0xB00;
enum DebugCode : int {
  kDbgSelRange = 0xB01,       // a selection entry outside [-1, blocks of the sequence)
  kDbgSelDuplicate = 0xB02,   // a block listed twice in one selection row
  kDbgTableRange = 0xB03,     // a block-table entry outside [0, n_phys)
  kDbgSeqLen = 0xB04,         // a cache length outside [0, seq_k]
  kDbgCoord = 0xB05,          // a tensor-copy coordinate outside its tensor
  kDbgStore = 0xB06,          // an output index outside its tensor
};

__device__ __forceinline__ void debug_check(bool ok, int* status, int code) {
  if (kDebugChecks && !ok && status) atomicCAS(status, 0, code);
}

// Debug builds: validates the selection rows (sel may be null), block table and cache
// lengths of a call on the device before its kernels run.  Release builds: does nothing.
cudaError_t launch_debug_validate(const Dims& p, const int32_t* sel, cudaStream_t st,
                                  int* status);

// Cache length of sequence b (the decode query sits at position len - 1).
__device__ __forceinline__ int seq_len_of(const Dims& p, int b) {
  if (!p.seq_lens) return p.Sk;
  const int L = p.seq_lens[b];
  return L < 0 ? 0 : (L > p.Sk ? p.Sk : L);
}

// Position of the last query of selection row m; its block is the row's current block.
__host__ __device__ inline int row_last_pos(const Dims& p, int m) {
  int last = m * p.Qt + p.Qt - 1;
  if (last > p.Sq - 1) last = p.Sq - 1;
  return p.q_off + last;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// 16-byte vector of T converted to fp32 (4 floats or 8 bf16 -> 8 floats).
template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const float* p, float* o) {
    float4 x = *reinterpret_cast<const float4*>(p);
    o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
  }
};
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* o) {
    uint4 x = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

// ----------------------------------------------------------------- launchers
// Each returns the launch error (cudaSuccess when the kernel was queued).
cudaError_t launch_index_scores(const Dims& p, const void* idx_q, const void* idx_k,
                                float* scores, cudaStream_t st, int* dev_status);
// shared = 1: one selection per (sequence, row) from the heads' summed scores, written to
// every head (the aggregated selection used as an ablation)
cudaError_t launch_block_topk(const Dims& p, const float* scores, int32_t* sel,
                              cudaStream_t st, int shared = 0);
cudaError_t launch_sparse_prefill(const Dims& p, const void* q, const void* k,
                                  const void* v, const int32_t* sel, void* out, float* lse,
                                  cudaStream_t st, int* dev_status);
cudaError_t launch_sparse_decode(const Dims& p, const void* q, const void* k, const void* v,
                                 const int32_t* sel, void* out, float* lse, float* ws,
                                 cudaStream_t st, int* dev_status);

// Gradients of the sparse prefill attention: dq [B,Sq,Hq,d], dk, dv [B,Hkv,Sk,d], fp32;
// dk and dv are cleared on the stream first, then accumulated.
cudaError_t launch_sparse_prefill_backward(const Dims& p, const void* q, const void* k,
                                           const void* v, const int32_t* sel, const void* out,
                                           const float* lse, const void* dout, float* dq,
                                           float* dk, float* dv, void* workspace,
                                           cudaStream_t st, int* status);
// Workspace bytes of the backward (0 on the CUDA-core path).
size_t backward_workspace_bytes(const Dims& p);

// KL loss of the index branch toward the main branch (see index_kl.cu): loss (device
// scalar, cleared then accumulated), d_idx_q [B,Sq,Hkv,dI] written, d_idx_k [B,Sk,dI]
// cleared then accumulated; fp32.
cudaError_t launch_index_kl(const Dims& p, const void* q, const void* k, const float* lse,
                            const void* idx_q, const void* idx_k, const int32_t* sel,
                            float* loss, float* d_idx_q, float* d_idx_k, void* workspace,
                            cudaStream_t st, int* status);
// Workspace bytes of the index KL (0 on the CUDA-core path).
size_t index_kl_workspace_bytes(const Dims& p);

// Decode split-KV: number of block groups each (sequence, KV head) is split into, and
// the scratch it needs (partial outputs and partial log-sum-exps, fp32).
int decode_num_splits(const Dims& p);
size_t decode_workspace_bytes(const Dims& p);

// Largest candidate count the top-k kernel keeps in shared memory.
constexpr int kMaxBlocks = 32768;

}  // namespace msa
