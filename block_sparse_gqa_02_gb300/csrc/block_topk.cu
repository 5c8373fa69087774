// Per-KV-head block top-k of MSA: every KV head keeps its own selection, never merged
// across heads ("Sparse Attention Cannot Be Directly Ported Across Architectures",
// paragraph "MSA addresses these issues"; Chinese topic page on MSA, summary), over block
// candidates rather than tokens, which keeps the candidate count small (aietalks.com,
// "Block-level retrieval makes sparse attention easier to run on GPUs").
//
// One CTA per selection row (b, g, m).  The current block cb is always kept; the other
// k-1 are the largest of blocks 0..cb-1 under the total order (score desc, index asc).
// Scores map to order-preserving 32-bit keys (-0 folded onto +0); a 4-pass 8-bit radix
// select finds the (k-1)-th largest key tau and how many copies of tau to keep; the
// selected blocks are then compacted in index order, which writes them ascending without
// a sort.  Bit-exact and deterministic.
#include "common.cuh"

namespace msa {

namespace {


__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) == 0) u = 0;                       // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);      // larger float -> larger key
}

// Exclusive prefix sum of one value per thread over the CTA; also returns the total.
template <int kThreads>
__device__ __forceinline__ int cta_exclusive_scan(int v, int* warp_sums, int& total) {
  constexpr int kWarps = kThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) warp_sums[lane] = w;                 // inclusive warp totals
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  total = warp_sums[kWarps - 1];
  __syncthreads();
  return before;
}

// shared != 0: the row is (b, m) and its candidates are the fp32 sums over the KV heads of
// their block scores (added in head order 0, 1, ...); the one selection is written to every
// head's row (the aggregated selection the pages contrast MSA with).
template <int kThreads>
__global__ void __launch_bounds__(kThreads) block_topk_kernel(const float* __restrict__ scores,
                                                              int32_t* __restrict__ sel, Dims p,
                                                              int shared) {
  constexpr int kWarps = kThreads / 32;
  extern __shared__ uint32_t keys[];                        // [cb]
  __shared__ uint32_t hist[256];
  __shared__ int warp_sums[kWarps];
  __shared__ uint32_t s_digit;
  __shared__ int s_remaining;

  // row = (b * Hkv + g) * nR + m, or b * nR + m for the shared selection
  const int row = blockIdx.x;
  const int m = row % p.nR;
  const int b = shared ? row / p.nR : row / (p.Hkv * p.nR);
  // ragged decode: the query of sequence b sits at its own cache length - 1
  const int last = p.seq_lens ? seq_len_of(p, b) - 1 : row_last_pos(p, m);
  const float* srow = scores + (size_t)row * p.nB;
  int32_t* out = sel + (size_t)row * p.k;
  const size_t head_stride = (size_t)p.nR * p.nB;           // between heads, same (b, m)
  if (shared) {
    srow = scores + ((size_t)b * p.Hkv * p.nR + m) * p.nB;
    out = sel + ((size_t)b * p.Hkv * p.nR + m) * p.k;
  }
  const int n_out = shared ? p.Hkv : 1;
  const size_t out_stride = (size_t)p.nR * p.k;
  if (last < 0) {                                           // empty sequence: nothing visible
    for (int h = 0; h < n_out; ++h)
      for (int i = threadIdx.x; i < p.k; i += kThreads) out[h * out_stride + i] = -1;
    return;
  }
  const int cb = last / p.Bk;

  if (cb + 1 <= p.k) {                                      // every candidate fits
    for (int h = 0; h < n_out; ++h)
      for (int i = threadIdx.x; i < p.k; i += kThreads) out[h * out_stride + i] = i <= cb ? i : -1;
    return;
  }
  const int want = p.k - 1;                                 // picked from blocks 0..cb-1
  if (want == 0) {
    if (threadIdx.x < n_out) out[threadIdx.x * out_stride] = cb;
    return;
  }
  const int n = cb;
  if (!shared) {
    // eight loads in flight per thread before any is used (a row of 8192 candidates is
    // eight rounds of the CTA)
    constexpr int kBatch = 8;
    for (int i0 = threadIdx.x; i0 < n; i0 += kThreads * kBatch) {
      float xs[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + u * kThreads;
        xs[u] = i < n ? __ldg(srow + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + u * kThreads;
        if (i < n) keys[i] = order_key(xs[u]);
      }
    }
  } else {
    for (int i = threadIdx.x; i < n; i += kThreads) {
      float x = srow[i];
      for (int h = 1; h < p.Hkv; ++h) x = __fadd_rn(x, srow[h * head_stride + i]);
      keys[i] = order_key(x);
    }
  }

  // radix select of the want-th largest key, 8 bits at a time from the top
  uint32_t prefix = 0, mask = 0;
  int remaining = want;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t key = keys[i];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      uint32_t c[8];
      int sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {                          // lane 0 holds bins 255..248
        c[e] = hist[255 - 8 * lane - e];
        sum += (int)c[e];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - sum;
      if (excl < remaining && remaining <= incl) {           // exactly one lane
        int cum = excl;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (cum + (int)c[e] >= remaining) {
            s_digit = 255u - 8u * lane - e;
            s_remaining = remaining - cum;
            break;
          }
          cum += (int)c[e];
        }
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 255u << shift;
    remaining = s_remaining;
    __syncthreads();
  }
  const uint32_t tau = prefix;                              // the want-th largest key
  const int take_eq = remaining;                            // copies of tau to keep

  // compaction in index order: thread t owns the contiguous slice [t*c, t*c + c)
  const int c = (n + kThreads - 1) / kThreads;
  const int lo = min(n, threadIdx.x * c), hi = min(n, lo + c);
  int n_eq = 0;
  for (int i = lo; i < hi; ++i) n_eq += keys[i] == tau;
  int total;
  const int eq_before = cta_exclusive_scan<kThreads>(n_eq, warp_sums, total);
  int n_take = 0;
  {
    int rank = eq_before;
    for (int i = lo; i < hi; ++i) {
      const uint32_t key = keys[i];
      if (key > tau) ++n_take;
      else if (key == tau) n_take += (rank++ < take_eq);
    }
  }
  const int pos0 = cta_exclusive_scan<kThreads>(n_take, warp_sums, total);
  {
    int rank = eq_before, pos = pos0;
    for (int i = lo; i < hi; ++i) {
      const uint32_t key = keys[i];
      const bool take = key > tau || (key == tau && rank++ < take_eq);
      if (take) {
        for (int h = 0; h < n_out; ++h) out[h * out_stride + pos] = i;
        ++pos;
      }
    }
  }
  if (threadIdx.x < n_out) out[threadIdx.x * out_stride + want] = cb;   // cb > every earlier
}

}  // namespace

template <int kThreads>
static cudaError_t launch_rows(const Dims& p, const float* scores, int32_t* sel, cudaStream_t st,
                               int shared) {
  const int rows = shared ? p.B * p.nR : p.B * p.Hkv * p.nR;
  const size_t smem = (size_t)p.nB * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(block_topk_kernel<kThreads>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  block_topk_kernel<kThreads><<<rows, kThreads, smem, st>>>(scores, sel, p, shared);
  return cudaGetLastError();
}

cudaError_t launch_block_topk(const Dims& p, const float* scores, int32_t* sel,
                              cudaStream_t st, int shared) {
  if (p.B * p.Hkv * p.nR == 0) return cudaSuccess;
  // long rows (decode at 1M context: 8192 candidates) get more threads per row
  if (p.nB > 2048) return launch_rows<1024>(p, scores, sel, st, shared);
  return launch_rows<256>(p, scores, sel, st, shared);
}

}  // namespace msa
