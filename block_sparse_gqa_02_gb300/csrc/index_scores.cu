// Index branch of MSA: causal index logits of NI index query heads against the one shared
// index key head, max-pooled into one score per (query tile, key block) for every head.
// ("Sparse Attention Cannot Be Directly Ported Across Architectures", paragraph
// introducing MSA: a lightweight full attention with four query heads and one key head;
// aietalks.com, "Block-level retrieval makes sparse attention easier to run on GPUs".)
//
// This file holds the CUDA-core kernels: the prefill kernel for fp32 inputs and shapes
// the tensor-core kernel does not cover, and the decode scan, which streams the index
// key cache once from HBM.
#include "common.cuh"
#include "index_scan_tc.cuh"
#include "index_tc.cuh"

namespace msa {

// ---------------------------------------------------------------------------------------
// Prefill, CUDA cores.  One CTA per (query tile m, sequence b); thread r owns the query
// row (head g = r / Qt, token m*Qt + r % Qt) and keeps it in registers.  Key blocks
// 0..cb are staged in shared memory as fp32; blocks after cb get -inf.
// ---------------------------------------------------------------------------------------
template <typename T, int DI>
__global__ void __launch_bounds__(256) index_scores_prefill_simt(
    const T* __restrict__ iq, const T* __restrict__ ik, float* __restrict__ scores, Dims p) {
  extern __shared__ float smem[];
  float* keys = smem;                          // [Bk][DI]
  float* rowmax = smem + p.Bk * DI;            // [NI * Qt]  (NI * Qt <= blockDim.x)
  const int m = blockIdx.x, b = blockIdx.y;
  const int NI = p.Hkv, Qt = p.Qt;
  const int rows = NI * Qt;
  const int cb = row_last_pos(p, m) / p.Bk;
  float* srow0 = scores + ((size_t)b * NI * p.nR + m) * p.nB;   // + g * nR * nB + blk

  // blocks after the current one hold no visible key
  const int n_after = p.nB - cb - 1;
  for (int i = threadIdx.x; i < NI * n_after; i += blockDim.x)
    srow0[(size_t)(i / n_after) * p.nR * p.nB + cb + 1 + i % n_after] = -INFINITY;

  const int r = threadIdx.x;
  const int g = r / Qt, tl = r % Qt;
  const int t = m * Qt + tl;
  const bool active = r < rows && t < p.Sq;
  const int pos = p.q_off + t;
  float qv[DI];
  if (active) {
    const T* qp = iq + (((size_t)b * p.Sq + t) * NI + g) * DI;
#pragma unroll
    for (int c = 0; c < DI; c += Vec16<T>::N) Vec16<T>::load(qp + c, qv + c);
  }
  for (int blk = 0; blk <= cb; ++blk) {
    const int j0 = blk * p.Bk;
    const int nk = min(p.Bk, p.Sk - j0);
    __syncthreads();
    const T* kp = ik + ((size_t)b * p.Sk + j0) * DI;
    for (int e = threadIdx.x * Vec16<T>::N; e < nk * DI; e += blockDim.x * Vec16<T>::N)
      Vec16<T>::load(kp + e, keys + e);
    __syncthreads();
    float mx = -INFINITY;
    if (active) {
      const int jmax = min(nk, pos - j0 + 1);    // causal: keys j <= pos
      for (int jj = 0; jj < jmax; ++jj) {
        const float4* kr = reinterpret_cast<const float4*>(keys + jj * DI);
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < DI / 4; ++c) {
          float4 kv = kr[c];
          acc = fmaf(qv[4 * c], kv.x, acc);
          acc = fmaf(qv[4 * c + 1], kv.y, acc);
          acc = fmaf(qv[4 * c + 2], kv.z, acc);
          acc = fmaf(qv[4 * c + 3], kv.w, acc);
        }
        mx = fmaxf(mx, acc);
      }
    }
    if (r < rows) rowmax[r] = mx;
    __syncthreads();
    if (threadIdx.x < NI) {                     // one thread per head reduces its Qt rows
      float best = -INFINITY;
      for (int i = threadIdx.x * Qt; i < (threadIdx.x + 1) * Qt; ++i) best = fmaxf(best, rowmax[i]);
      srow0[(size_t)threadIdx.x * p.nR * p.nB + blk] =
          best == -INFINITY ? -INFINITY : best * p.index_scale;
    }
  }
}

// ---------------------------------------------------------------------------------------
// Decode scan.  The new token's NI index queries (fp32 in shared memory) against every key
// of the cache; one warp per key block, lane l takes keys l, l+32, ...; block max over the
// warp.  Memory-bound: each index key is read exactly once.
// ---------------------------------------------------------------------------------------
template <typename T, int DI, int NI>
__global__ void __launch_bounds__(256) index_scores_decode_scan(
    const T* __restrict__ iq, const T* __restrict__ ik, float* __restrict__ scores, Dims p) {
  __shared__ float qs[NI][DI];
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < NI * DI; i += blockDim.x)
    qs[i / DI][i % DI] = to_f32(iq[(size_t)b * NI * DI + i]);
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int warps_total = gridDim.x * (blockDim.x / 32);
  for (int blk = blockIdx.x * (blockDim.x / 32) + warp; blk < p.nB; blk += warps_total) {
    const int j0 = blk * p.Bk;
    const int nk = min(p.Bk, p.Sk - j0);
    float mx[NI];
#pragma unroll
    for (int h = 0; h < NI; ++h) mx[h] = -INFINITY;
    for (int jj = lane; jj < nk; jj += 32) {
      const T* kp = ik + ((size_t)b * p.Sk + j0 + jj) * DI;
      float acc[NI];
#pragma unroll
      for (int h = 0; h < NI; ++h) acc[h] = 0.f;
#pragma unroll
      for (int c = 0; c < DI; c += Vec16<T>::N) {
        float kv[Vec16<T>::N];
        Vec16<T>::load(kp + c, kv);
#pragma unroll
        for (int e = 0; e < Vec16<T>::N; ++e)
#pragma unroll
          for (int h = 0; h < NI; ++h) acc[h] = fmaf(qs[h][c + e], kv[e], acc[h]);
      }
#pragma unroll
      for (int h = 0; h < NI; ++h) mx[h] = fmaxf(mx[h], acc[h]);
    }
#pragma unroll
    for (int h = 0; h < NI; ++h)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], o));
    if (lane < NI) {
      float v = mx[0];
#pragma unroll
      for (int h = 1; h < NI; ++h)
        if (lane == h) v = mx[h];
      scores[((size_t)b * NI + lane) * p.nB + blk] = v * p.index_scale;
    }
  }
}

template <typename T, int DI>
static cudaError_t launch_prefill_simt(const Dims& p, const void* iq, const void* ik,
                                       float* scores, cudaStream_t st) {
  const int rows = p.Hkv * p.Qt;               // validated: rows <= 256
  const int threads = ((rows + 31) / 32) * 32;
  const size_t smem = ((size_t)p.Bk * DI + (size_t)threads) * sizeof(float);
  auto kern = index_scores_prefill_simt<T, DI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.nR, p.B);
  kern<<<grid, threads, smem, st>>>((const T*)iq, (const T*)ik, scores, p);
  return cudaGetLastError();
}

template <typename T, int DI>
static cudaError_t launch_decode_scan(const Dims& p, const void* iq, const void* ik,
                                      float* scores, cudaStream_t st) {
  const int warps = 8;
  int ctas = (p.nB + warps - 1) / warps;
  if (ctas > 4096) ctas = 4096;
  dim3 grid(ctas, p.B);
  switch (p.Hkv) {
    case 4: index_scores_decode_scan<T, DI, 4><<<grid, warps * 32, 0, st>>>(
        (const T*)iq, (const T*)ik, scores, p); break;
    case 8: index_scores_decode_scan<T, DI, 8><<<grid, warps * 32, 0, st>>>(
        (const T*)iq, (const T*)ik, scores, p); break;
    case 2: index_scores_decode_scan<T, DI, 2><<<grid, warps * 32, 0, st>>>(
        (const T*)iq, (const T*)ik, scores, p); break;
    case 1: index_scores_decode_scan<T, DI, 1><<<grid, warps * 32, 0, st>>>(
        (const T*)iq, (const T*)ik, scores, p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <typename T>
static cudaError_t dispatch_dim(const Dims& p, const void* iq, const void* ik, float* scores,
                                cudaStream_t st) {
  if (p.decode) {
    return p.dI == 128 ? launch_decode_scan<T, 128>(p, iq, ik, scores, st)
                       : launch_decode_scan<T, 64>(p, iq, ik, scores, st);
  }
  return p.dI == 128 ? launch_prefill_simt<T, 128>(p, iq, ik, scores, st)
                     : launch_prefill_simt<T, 64>(p, iq, ik, scores, st);
}

cudaError_t launch_index_scores(const Dims& p, const void* idx_q, const void* idx_k,
                                float* scores, cudaStream_t st, int* dev_status) {
  if (p.dtype == 1) {
    if (index_tc_supported(p))
      return launch_index_scores_tc(p, idx_q, idx_k, scores, nullptr, st, dev_status);
    if (index_scan_tc_supported(p))
      return launch_index_scan_tc(p, idx_q, idx_k, scores, st, dev_status);
    return dispatch_dim<__nv_bfloat16>(p, idx_q, idx_k, scores, st);
  }
  return dispatch_dim<float>(p, idx_q, idx_k, scores, st);
}

}  // namespace msa
