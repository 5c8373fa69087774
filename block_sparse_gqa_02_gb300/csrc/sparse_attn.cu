// Main branch of MSA: exact softmax attention of every query head over the key blocks its
// KV head selected ("How MiniMax M3 was built", aietalks.com, section "MSA uses a
// lightweight index branch before sparse attention": the sparse branch attends only to
// the selected blocks; Chinese topic page on MSA, summary: exact attention on the chosen
// blocks).  All G query heads of a KV group share the group's selection.
//
// This file holds the CUDA-core kernels: prefill for fp32 and for shapes the tensor-core
// kernel does not cover, and the split-KV decode with its log-sum-exp merge.
#include "common.cuh"
#include "sparse_decode_mma.cuh"
#include "sparse_prefill_tc.cuh"

namespace msa {

namespace {

constexpr int kRows = 64;          // query rows per CTA
constexpr int kTPR = 4;            // threads per row
constexpr int kThreads = kRows * kTPR;
constexpr int kKC = 32;            // keys staged per step
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Online-softmax attention of up to kRows query rows over a list of key blocks.
// Row state lives in the kTPR threads of the row: each holds D/kTPR output dims (dims
// 4*lane + 4*kTPR*i .. +3) and the full running max / sum.
template <typename T, int D>
struct RowAttention {
  static constexpr int DPT = D / kTPR;       // dims per thread
  float q[DPT], acc[DPT];
  float mrow, lrow;                          // running max (log2 units), running sum

  __device__ void init(const T* qrow, bool active, float scale_log2) {
    const int sub = threadIdx.x % kTPR;
#pragma unroll
    for (int i = 0; i < DPT / 4; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int dim = 4 * sub + 4 * kTPR * i + e;
        q[4 * i + e] = active ? to_f32(qrow[dim]) * scale_log2 : 0.f;
        acc[4 * i + e] = 0.f;
      }
    mrow = -INFINITY;
    lrow = 0.f;
  }

  // Keys [j0, j0 + nk) of one KV head (rows of kv_k / kv_v), staged kKC at a time.
  __device__ void run_keys(const T* kbase, const T* vbase, int j0, int nk, int pos,
                           float* ks, float* vs) {
    const int sub = threadIdx.x % kTPR;
    for (int c0 = 0; c0 < nk; c0 += kKC) {
      const int nc = min(kKC, nk - c0);
      __syncthreads();
      for (int e = threadIdx.x * Vec16<T>::N; e < kKC * D; e += kThreads * Vec16<T>::N) {
        if (e < nc * D) {
          Vec16<T>::load(kbase + (size_t)(j0 + c0) * D + e, ks + e);
          Vec16<T>::load(vbase + (size_t)(j0 + c0) * D + e, vs + e);
        } else {
#pragma unroll
          for (int x = 0; x < Vec16<T>::N; ++x) ks[e + x] = vs[e + x] = 0.f;
        }
      }
      __syncthreads();
      float s[kKC];
      float cmax = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < kKC; ++jj) {
        const float4* kr = reinterpret_cast<const float4*>(ks + jj * D) + sub;
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < DPT / 4; ++i) {
          float4 kv = kr[kTPR * i];
          dot = fmaf(q[4 * i], kv.x, dot);
          dot = fmaf(q[4 * i + 1], kv.y, dot);
          dot = fmaf(q[4 * i + 2], kv.z, dot);
          dot = fmaf(q[4 * i + 3], kv.w, dot);
        }
#pragma unroll
        for (int o = 1; o < kTPR; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        const bool vis = jj < nc && (j0 + c0 + jj) <= pos;
        s[jj] = vis ? dot : -INFINITY;
        cmax = fmaxf(cmax, s[jj]);
      }
      const float mnew = fmaxf(mrow, cmax);
      if (mnew == -INFINITY) continue;                      // nothing visible yet
      const float alpha = exp2f(mrow - mnew);
      lrow *= alpha;
#pragma unroll
      for (int i = 0; i < DPT; ++i) acc[i] *= alpha;
#pragma unroll
      for (int jj = 0; jj < kKC; ++jj) {
        const float pj = exp2f(s[jj] - mnew);
        lrow += pj;
        const float4* vr = reinterpret_cast<const float4*>(vs + jj * D) + sub;
#pragma unroll
        for (int i = 0; i < DPT / 4; ++i) {
          float4 vv = vr[kTPR * i];
          acc[4 * i] = fmaf(pj, vv.x, acc[4 * i]);
          acc[4 * i + 1] = fmaf(pj, vv.y, acc[4 * i + 1]);
          acc[4 * i + 2] = fmaf(pj, vv.z, acc[4 * i + 2]);
          acc[4 * i + 3] = fmaf(pj, vv.w, acc[4 * i + 3]);
        }
      }
      mrow = mnew;
    }
  }

  // Natural-log lse, -inf for an empty row.
  __device__ float lse() const {
    return lrow > 0.f ? mrow * kLn2 + logf(lrow) : -INFINITY;
  }
};

// Prefill: grid (row chunks of kRows, selection rows nR, B * Hkv).  Row r of tile m:
// token m*Qt + r / G, head g*G + r % G.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) sparse_prefill_simt(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const int32_t* __restrict__ sel, T* __restrict__ out, float* __restrict__ lse, Dims p) {
  extern __shared__ float smem[];
  float* ks = smem;
  float* vs = smem + kKC * D;
  const int m = blockIdx.y, bg = blockIdx.z, b = bg / p.Hkv, g = bg % p.Hkv;
  const int r = blockIdx.x * kRows + threadIdx.x / kTPR;
  const int tl = r / p.G, h = g * p.G + r % p.G;
  const int t = m * p.Qt + tl;
  const bool active = tl < p.Qt && t < p.Sq;
  const float scale_log2 = p.sm_scale * kLog2e;

  const int32_t* srow = sel + ((size_t)bg * p.nR + m) * p.k;

  RowAttention<T, D> ra;
  ra.init(q + (((size_t)b * p.Sq + (active ? t : 0)) * p.Hq + h) * D, active, scale_log2);
  const T* kbase = k + (size_t)bg * p.Sk * D;
  const T* vbase = v + (size_t)bg * p.Sk * D;
  const int pos = active ? p.q_off + t : -1;
  for (int i = 0; i < p.k; ++i) {
    const int blk = srow[i];
    if (blk < 0 || blk >= p.nB) continue;
    const int j0 = blk * p.Bk;
    ra.run_keys(kbase, vbase, j0, min(p.Bk, p.Sk - j0), pos, ks, vs);
  }
  if (!active) return;
  const int sub = threadIdx.x % kTPR;
  const float inv = ra.lrow > 0.f ? 1.f / ra.lrow : 0.f;
  T* orow = out + (((size_t)b * p.Sq + t) * p.Hq + h) * D;
#pragma unroll
  for (int i = 0; i < RowAttention<T, D>::DPT / 4; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) orow[4 * sub + 4 * kTPR * i + e] = from_f32<T>(ra.acc[4 * i + e] * inv);
  if (lse && sub == 0) lse[((size_t)b * p.Hq + h) * p.Sq + t] = ra.lse();
}

// Decode partials: grid (splits, 1, B * Hkv); rows are the G heads of the group (G <= 64).
// Split s covers selection entries [s * per, (s + 1) * per).  Writes normalised partial
// outputs and their natural-log lse into the workspace.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) sparse_decode_partial_simt(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const int32_t* __restrict__ sel, float* __restrict__ ws_o, float* __restrict__ ws_l,
    Dims p, int n_split, int per) {
  extern __shared__ float smem[];
  float* ks = smem;
  float* vs = smem + kKC * D;
  const int s = blockIdx.x, bg = blockIdx.z, b = bg / p.Hkv, g = bg % p.Hkv;
  const int r = threadIdx.x / kTPR;
  const bool active = r < p.G;
  const int h = g * p.G + (active ? r : 0);
  RowAttention<T, D> ra;
  ra.init(q + ((size_t)b * p.Hq + h) * D, active, p.sm_scale * kLog2e);
  const int32_t* srow = sel + (size_t)bg * p.k;
  const T* kbase = k + (size_t)bg * p.Sk * D;
  const T* vbase = v + (size_t)bg * p.Sk * D;
  const int pos = p.Sk - 1;
  const int i1 = min(p.k, (s + 1) * per);
  for (int i = s * per; i < i1; ++i) {
    const int blk = srow[i];
    if (blk < 0 || blk >= p.nB) continue;
    const int j0 = blk * p.Bk;
    ra.run_keys(kbase, vbase, j0, min(p.Bk, p.Sk - j0), pos, ks, vs);
  }
  if (!active) return;
  const int sub = threadIdx.x % kTPR;
  const size_t slot = ((size_t)b * p.Hq + h) * n_split + s;
  const float inv = ra.lrow > 0.f ? 1.f / ra.lrow : 0.f;
#pragma unroll
  for (int i = 0; i < RowAttention<T, D>::DPT / 4; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      ws_o[slot * D + 4 * sub + 4 * kTPR * i + e] = ra.acc[4 * i + e] * inv;
  if (sub == 0) ws_l[slot] = ra.lse();
}

// o = sum_s exp(lse_s - lse) o_s with lse = log sum_s exp(lse_s).  One CTA per (b, h).
template <typename T, int D>
__global__ void __launch_bounds__(D) decode_combine(const float* __restrict__ ws_o,
                                                   const float* __restrict__ ws_l,
                                                   T* __restrict__ out, float* __restrict__ lse,
                                                   Dims p, int n_split) {
  const int bh = blockIdx.x;
  const float* l = ws_l + (size_t)bh * n_split;
  float mx = -INFINITY;
  for (int s = 0; s < n_split; ++s) mx = fmaxf(mx, l[s]);
  float acc = 0.f, den = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < n_split; ++s) {
      const float w = expf(l[s] - mx);
      den += w;
      acc = fmaf(w, ws_o[((size_t)bh * n_split + s) * D + threadIdx.x], acc);
    }
  }
  out[(size_t)bh * D + threadIdx.x] = from_f32<T>(den > 0.f ? acc / den : 0.f);
  if (lse && threadIdx.x == 0) lse[bh] = den > 0.f ? mx + logf(den) : -INFINITY;
}

template <typename T, int D>
cudaError_t prefill_simt(const Dims& p, const void* q, const void* k, const void* v,
                         const int32_t* sel, void* out, float* lse, cudaStream_t st) {
  const size_t smem = 2 * (size_t)kKC * D * sizeof(float);
  auto kern = sparse_prefill_simt<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.Qt * p.G + kRows - 1) / kRows, p.nR, p.B * p.Hkv);
  kern<<<grid, kThreads, smem, st>>>((const T*)q, (const T*)k, (const T*)v, sel, (T*)out, lse, p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t decode_split(const Dims& p, const void* q, const void* k, const void* v,
                         const int32_t* sel, void* out, float* lse, float* ws, cudaStream_t st,
                         int* dev_status) {
  const int n_split = decode_num_splits(p);
  const int per = (p.k + n_split - 1) / n_split;
  float* ws_o = ws;
  float* ws_l = ws + (size_t)p.B * p.Hq * n_split * D;
  cudaError_t e;
  if (sparse_decode_mma_supported(p)) {
    e = launch_sparse_decode_mma(p, q, k, v, sel, ws_o, ws_l, n_split, per, st, dev_status);
  } else {
    const size_t smem = 2 * (size_t)kKC * D * sizeof(float);
    auto kern = sparse_decode_partial_simt<T, D>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(n_split, 1, p.B * p.Hkv);
    kern<<<grid, kThreads, smem, st>>>((const T*)q, (const T*)k, (const T*)v, sel, ws_o, ws_l,
                                       p, n_split, per);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  decode_combine<T, D><<<p.B * p.Hq, D, 0, st>>>(ws_o, ws_l, (T*)out, lse, p, n_split);
  return cudaGetLastError();
}

}  // namespace

int decode_num_splits(const Dims& p) {
  // one wave of CTAs over the 152 SMs (one resident CTA per SM): each CTA then streams a
  // long run of blocks through its TMA ring instead of paying the ring's fill and drain
  // several times; never more splits than blocks
  const int units = p.B * p.Hkv;
  int s = 152 / units;
  if (s > p.k) s = p.k;
  if (s < 1) s = 1;
  return s;
}

size_t decode_workspace_bytes(const Dims& p) {
  const size_t slots = (size_t)p.B * p.Hq * decode_num_splits(p);
  return slots * ((size_t)p.d + 1) * sizeof(float);
}

cudaError_t launch_sparse_prefill(const Dims& p, const void* q, const void* k, const void* v,
                                  const int32_t* sel, void* out, float* lse, cudaStream_t st,
                                  int* dev_status) {
  if (p.dtype == 1 && sparse_prefill_tc_supported(p))
    return launch_sparse_prefill_tc(p, q, k, v, sel, out, lse, st, dev_status);
  if (p.dtype == 1)
    return p.d == 128 ? prefill_simt<__nv_bfloat16, 128>(p, q, k, v, sel, out, lse, st)
                      : prefill_simt<__nv_bfloat16, 64>(p, q, k, v, sel, out, lse, st);
  return p.d == 128 ? prefill_simt<float, 128>(p, q, k, v, sel, out, lse, st)
                    : prefill_simt<float, 64>(p, q, k, v, sel, out, lse, st);
}

cudaError_t launch_sparse_decode(const Dims& p, const void* q, const void* k, const void* v,
                                 const int32_t* sel, void* out, float* lse, float* ws,
                                 cudaStream_t st, int* dev_status) {
  if (p.dtype == 1)
    return p.d == 128
               ? decode_split<__nv_bfloat16, 128>(p, q, k, v, sel, out, lse, ws, st, dev_status)
               : decode_split<__nv_bfloat16, 64>(p, q, k, v, sel, out, lse, ws, st, dev_status);
  return p.d == 128 ? decode_split<float, 128>(p, q, k, v, sel, out, lse, ws, st, dev_status)
                    : decode_split<float, 64>(p, q, k, v, sel, out, lse, ws, st, dev_status);
}

}  // namespace msa
