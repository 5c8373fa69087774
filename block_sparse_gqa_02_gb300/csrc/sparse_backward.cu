// Training: gradients of MSA's main branch, the sparse attention over the selected blocks
// (the pages mention kernels for training: "Sparse Attention Cannot Be Directly Ported
// Across Architectures", paragraph "MSA addresses these issues"; aietalks.com, section
// "Block-level retrieval makes sparse attention easier to run on GPUs").
//
// For each query row (token t, head h of KV group g) over its keys J (selected blocks, j <= t):
//   p_j = exp(sm_scale q.k_j - lse),  D = dout . out,  dp_j = dout . v_j,
//   ds_j = p_j (dp_j - D),  dq = sm_scale sum_j ds_j k_j,
//   dk_j += sm_scale ds_j q,  dv_j += p_j dout   (summed over every row that sees key j).
// CTA = 64 rows of one (sequence, KV head, query tile), as in the CUDA-core forward.  Per
// 32-key chunk, each row's 4 threads compute p and ds, keep dq in registers, and the CTA then
// forms the chunk's dk / dv partials (ds^T Q and p^T dout over its 64 rows) from shared memory
// and adds them to fp32 dk / dv with atomics, because a block is shared by all the tiles
// that selected it.  CUDA cores, fp32 throughout; a first implementation of the training
// path (the tensor-core forward kernels are the optimised hot path).
#include "common.cuh"
#include "sparse_backward_tc.cuh"

namespace msa {

namespace {

constexpr int kRows = 64;
constexpr int kTPR = 4;
constexpr int kThreads = kRows * kTPR;
constexpr int kKC = 32;
constexpr float kLog2e = 1.4426950408889634f;

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) sparse_backward_simt(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const int32_t* __restrict__ sel, const T* __restrict__ out, const float* __restrict__ lse,
    const T* __restrict__ dout, float* __restrict__ dq, float* __restrict__ dk,
    float* __restrict__ dv, Dims p) {
  constexpr int DPT = D / kTPR;
  extern __shared__ float smem[];
  float* ks = smem;                        // [kKC][D]
  float* vs = ks + kKC * D;                // [kKC][D]
  float* qs = vs + kKC * D;                // [kRows][D]  q
  float* dos = qs + kRows * D;             // [kRows][D]  dout
  float* ps = dos + kRows * D;             // [kRows][kKC] p
  float* dss = ps + kRows * kKC;           // [kRows][kKC] sm_scale * ds

  const int m = blockIdx.y, bg = blockIdx.z, b = bg / p.Hkv, g = bg % p.Hkv;
  const int rl = threadIdx.x / kTPR, sub = threadIdx.x % kTPR;
  const int r = blockIdx.x * kRows + rl;
  const int tl = r / p.G, h = g * p.G + r % p.G;
  const int t = m * p.Qt + tl;
  const bool active = tl < p.Qt && t < p.Sq;
  const int pos = active ? t : -1;

  // this row: q (scaled) and dout in registers and shared memory, lse, D = dout . out
  float qv[DPT], dov[DPT], dqv[DPT];
  float dsum = 0.f;
  const size_t row_off = (((size_t)b * p.Sq + (active ? t : 0)) * p.Hq + h) * D;
#pragma unroll
  for (int i = 0; i < DPT / 4; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int dim = 4 * sub + 4 * kTPR * i + e;
      const float qraw = active ? to_f32(q[row_off + dim]) : 0.f;
      const float dd = active ? to_f32(dout[row_off + dim]) : 0.f;
      const float oo = active ? to_f32(out[row_off + dim]) : 0.f;
      qv[4 * i + e] = qraw * p.sm_scale;
      dov[4 * i + e] = dd;
      dqv[4 * i + e] = 0.f;
      dsum = fmaf(dd, oo, dsum);
      qs[rl * D + dim] = qraw;
      dos[rl * D + dim] = dd;
    }
#pragma unroll
  for (int o = 1; o < kTPR; o <<= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
  const float lse2 = active ? lse[((size_t)b * p.Hq + h) * p.Sq + t] * kLog2e : 0.f;

  const int32_t* srow = sel + ((size_t)bg * p.nR + m) * p.k;
  const T* kbase = k + (size_t)bg * p.Sk * D;
  const T* vbase = v + (size_t)bg * p.Sk * D;
  float* dkbase = dk + (size_t)bg * p.Sk * D;
  float* dvbase = dv + (size_t)bg * p.Sk * D;
  for (int i = 0; i < p.k; ++i) {
    const int blk = srow[i];
    if (blk < 0 || blk >= p.nB) continue;
    const int j0 = blk * p.Bk;
    const int nk = min(p.Bk, p.Sk - j0);
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
      // per row: p and ds for the chunk's keys, dq accumulation
#pragma unroll 4
      for (int jj = 0; jj < kKC; ++jj) {
        const float4* kr = reinterpret_cast<const float4*>(ks + jj * D) + sub;
        const float4* vr = reinterpret_cast<const float4*>(vs + jj * D) + sub;
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int x = 0; x < DPT / 4; ++x) {
          const float4 kk = kr[kTPR * x], vv = vr[kTPR * x];
          s = fmaf(qv[4 * x], kk.x, fmaf(qv[4 * x + 1], kk.y,
              fmaf(qv[4 * x + 2], kk.z, fmaf(qv[4 * x + 3], kk.w, s))));
          dp = fmaf(dov[4 * x], vv.x, fmaf(dov[4 * x + 1], vv.y,
               fmaf(dov[4 * x + 2], vv.z, fmaf(dov[4 * x + 3], vv.w, dp))));
        }
#pragma unroll
        for (int o = 1; o < kTPR; o <<= 1) {
          s += __shfl_xor_sync(0xffffffffu, s, o);
          dp += __shfl_xor_sync(0xffffffffu, dp, o);
        }
        const bool vis = jj < nc && (j0 + c0 + jj) <= pos;
        const float pj = vis ? exp2f(fmaf(s, kLog2e, -lse2)) : 0.f;
        const float ds = pj * (dp - dsum) * p.sm_scale;
#pragma unroll
        for (int x = 0; x < DPT / 4; ++x) {
          const float4 kk = kr[kTPR * x];
          dqv[4 * x] = fmaf(ds, kk.x, dqv[4 * x]);
          dqv[4 * x + 1] = fmaf(ds, kk.y, dqv[4 * x + 1]);
          dqv[4 * x + 2] = fmaf(ds, kk.z, dqv[4 * x + 2]);
          dqv[4 * x + 3] = fmaf(ds, kk.w, dqv[4 * x + 3]);
        }
        if (sub == 0) {
          ps[rl * kKC + jj] = pj;
          dss[rl * kKC + jj] = ds;
        }
      }
      __syncthreads();
      // the chunk's dk_j = sum_rows (sm_scale ds) q and dv_j = sum_rows p dout: thread
      // (key jj, dims 4 s + 32 x .. +3) sums over the CTA's 64 rows (conflict-free float4
      // reads), then adds its float4s to global memory with vector atomics
      {
        constexpr int TPK = kThreads / kKC;                  // threads per key: 8
        constexpr int NV = D / (4 * TPK);                    // float4s per thread
        const int jj = threadIdx.x / TPK, sl = threadIdx.x % TPK;
        if (jj < nc) {
          float4 ak[NV], av[NV];
#pragma unroll
          for (int x = 0; x < NV; ++x) ak[x] = av[x] = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int rr = 0; rr < kRows; ++rr) {
            const float dsv = dss[rr * kKC + jj], pv = ps[rr * kKC + jj];
            if (dsv == 0.f && pv == 0.f) continue;
            const float4* qr4 = reinterpret_cast<const float4*>(qs + rr * D) + sl;
            const float4* dr4 = reinterpret_cast<const float4*>(dos + rr * D) + sl;
#pragma unroll
            for (int x = 0; x < NV; ++x) {
              const float4 a = qr4[TPK * x], d4 = dr4[TPK * x];
              ak[x].x = fmaf(dsv, a.x, ak[x].x); ak[x].y = fmaf(dsv, a.y, ak[x].y);
              ak[x].z = fmaf(dsv, a.z, ak[x].z); ak[x].w = fmaf(dsv, a.w, ak[x].w);
              av[x].x = fmaf(pv, d4.x, av[x].x); av[x].y = fmaf(pv, d4.y, av[x].y);
              av[x].z = fmaf(pv, d4.z, av[x].z); av[x].w = fmaf(pv, d4.w, av[x].w);
            }
          }
          float4* dkr = reinterpret_cast<float4*>(dkbase + (size_t)(j0 + c0 + jj) * D) + sl;
          float4* dvr = reinterpret_cast<float4*>(dvbase + (size_t)(j0 + c0 + jj) * D) + sl;
#pragma unroll
          for (int x = 0; x < NV; ++x) {
            atomicAdd(dkr + TPK * x, ak[x]);
            atomicAdd(dvr + TPK * x, av[x]);
          }
        }
      }
    }
  }
  if (!active) return;
  float* dqr = dq + row_off;
#pragma unroll
  for (int i = 0; i < DPT / 4; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dqr[4 * sub + 4 * kTPR * i + e] = dqv[4 * i + e];
}

template <typename T, int D>
cudaError_t backward(const Dims& p, const void* q, const void* k, const void* v,
                     const int32_t* sel, const void* out, const float* lse, const void* dout,
                     float* dq, float* dk, float* dv, cudaStream_t st) {
  const size_t kv_elems = (size_t)p.B * p.Hkv * p.Sk * D;
  cudaError_t e = cudaMemsetAsync(dk, 0, kv_elems * sizeof(float), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, kv_elems * sizeof(float), st);
  if (e != cudaSuccess) return e;
  const size_t smem = (2 * (size_t)kKC * D + 2 * (size_t)kRows * D + 2 * (size_t)kRows * kKC) *
                      sizeof(float);
  auto kern = sparse_backward_simt<T, D>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.Qt * p.G + kRows - 1) / kRows, p.nR, p.B * p.Hkv);
  kern<<<grid, kThreads, smem, st>>>((const T*)q, (const T*)k, (const T*)v, sel, (const T*)out,
                                     lse, (const T*)dout, dq, dk, dv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_prefill_backward(const Dims& p, const void* q, const void* k,
                                           const void* v, const int32_t* sel, const void* out,
                                           const float* lse, const void* dout, float* dq,
                                           float* dk, float* dv, void* workspace,
                                           cudaStream_t st, int* status) {
  if (sparse_backward_tc_supported(p))
    return launch_sparse_backward_tc(p, q, k, v, sel, out, lse, dout, dq, dk, dv, workspace, st,
                                     status);
  if (p.dtype == 1)
    return p.d == 128 ? backward<__nv_bfloat16, 128>(p, q, k, v, sel, out, lse, dout, dq, dk, dv, st)
                      : backward<__nv_bfloat16, 64>(p, q, k, v, sel, out, lse, dout, dq, dk, dv, st);
  return p.d == 128 ? backward<float, 128>(p, q, k, v, sel, out, lse, dout, dq, dk, dv, st)
                    : backward<float, 64>(p, q, k, v, sel, out, lse, dout, dq, dk, dv, st);
}

size_t backward_workspace_bytes(const Dims& p) {
  return sparse_backward_tc_supported(p) ? sparse_backward_tc_workspace_bytes(p) : 0;
}

}  // namespace msa
