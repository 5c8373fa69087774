// Training the index branch: KL loss toward the main branch's attention ("Sparse Attention
// Cannot Be Directly Ported Across Architectures", paragraph introducing MSA; aietalks.com,
// "MSA uses a lightweight index branch before sparse attention": the index branch is
// trained with a KL loss to match the attention scores of the main branch).
//
// For token t and KV head g over the keys J the main branch attends (selected blocks,
// j <= t): target p_T[j] = mean over the group's G query heads of exp(sm_scale q_h.k_j -
// lse_h) (held constant), index p_I = softmax over J of s_j = index_scale q_I.k_I[j];
// loss += KL(p_T || p_I); dL/ds_j = p_I[j] - p_T[j]; d idx_q[t,g] = index_scale sum_j
// (p_I - p_T)_j k_I[j]; d idx_k[j] += index_scale (p_I - p_T)_j q_I[t,g].
// CTA = 64 tokens x 4 threads of one (sequence, KV head, query tile); a tile of more than
// 64 tokens takes several CTAs.  Pass 1 runs the index
// logits over J for the row's log-normaliser; pass 2 recomputes them with the main-branch
// probabilities chunk by chunk, accumulates the loss and d idx_q in registers, and reduces
// d idx_k over the CTA's tokens in shared memory before fp32 atomics (index keys are shared
// by every tile and head).  CUDA cores, fp32.
#include "common.cuh"
#include "index_kl_tc.cuh"

namespace msa {

namespace {

constexpr int kTok = 64;
constexpr int kTPR = 4;
constexpr int kThreads = kTok * kTPR;
constexpr int kKC = 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename T, int D, int DI>
__global__ void __launch_bounds__(kThreads) index_kl_simt(
    const T* __restrict__ q, const T* __restrict__ k, const float* __restrict__ lse,
    const T* __restrict__ iq, const T* __restrict__ ik, const int32_t* __restrict__ sel,
    float* __restrict__ loss, float* __restrict__ diq, float* __restrict__ dik, Dims p) {
  constexpr int DPT = D / kTPR, IPT = DI / kTPR;
  extern __shared__ float smem[];
  float* ks = smem;                        // [kKC][D]   main keys of the chunk
  float* iks = ks + kKC * D;               // [kKC][DI]  index keys of the chunk
  float* iqs = iks + kKC * DI;             // [kTok][DI] index queries of the tile
  float* gs = iqs + kTok * DI;             // [kTok][kKC] index_scale * (p_I - p_T)
  __shared__ float loss_part[kThreads / 32];

  const int m = blockIdx.y, bg = blockIdx.z, b = bg / p.Hkv, g = bg % p.Hkv;
  const int rl = threadIdx.x / kTPR, sub = threadIdx.x % kTPR;   // CTA row, quarter of dims
  const int tl = blockIdx.x * kTok + rl;                           // token within the tile
  const int t = m * p.Qt + tl;
  const bool active = tl < p.Qt && t < p.Sq;
  const int pos = active ? t : -1;

  float qi[IPT], dqi[IPT];
#pragma unroll
  for (int i = 0; i < IPT / 4; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int dim = 4 * sub + 4 * kTPR * i + e;
      const float x = active ? to_f32(iq[(((size_t)b * p.Sq + t) * p.Hkv + g) * DI + dim]) : 0.f;
      qi[4 * i + e] = x * p.index_scale;
      dqi[4 * i + e] = 0.f;
      iqs[rl * DI + dim] = x;
    }
  float lse2[64];                          // main-branch lse of the group's heads, log2 units
  for (int hh = 0; hh < p.G; ++hh)
    lse2[hh] = active ? lse[((size_t)b * p.Hq + g * p.G + hh) * p.Sq + t] * kLog2e : 0.f;

  const int32_t* srow = sel + ((size_t)bg * p.nR + m) * p.k;
  const T* kbase = k + (size_t)bg * p.Sk * D;
  const T* ikbase = ik + (size_t)b * p.Sk * DI;
  const T* qrow = q + (((size_t)b * p.Sq + (active ? t : 0)) * p.Hq + (size_t)g * p.G) * D;

  // stage keys [j0, j0 + nc) of both kinds into shared memory
  auto stage = [&](int j0, int nc, bool with_main) {
    __syncthreads();
    for (int e = threadIdx.x * Vec16<T>::N; e < kKC * DI; e += kThreads * Vec16<T>::N) {
      if (e < nc * DI) Vec16<T>::load(ikbase + (size_t)j0 * DI + e, iks + e);
      else
        for (int x = 0; x < Vec16<T>::N; ++x) iks[e + x] = 0.f;
    }
    if (with_main)
      for (int e = threadIdx.x * Vec16<T>::N; e < kKC * D; e += kThreads * Vec16<T>::N) {
        if (e < nc * D) Vec16<T>::load(kbase + (size_t)j0 * D + e, ks + e);
        else
          for (int x = 0; x < Vec16<T>::N; ++x) ks[e + x] = 0.f;
      }
    __syncthreads();
  };
  auto index_logit = [&](int jj) {      // log2 units
    const float4* kr = reinterpret_cast<const float4*>(iks + jj * DI) + sub;
    float s = 0.f;
#pragma unroll
    for (int x = 0; x < IPT / 4; ++x) {
      const float4 kk = kr[kTPR * x];
      s = fmaf(qi[4 * x], kk.x, fmaf(qi[4 * x + 1], kk.y,
          fmaf(qi[4 * x + 2], kk.z, fmaf(qi[4 * x + 3], kk.w, s))));
    }
#pragma unroll
    for (int o = 1; o < kTPR; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s * kLog2e;
  };

  // pass 1: log-normaliser of the index distribution over the row's keys (log2 units)
  float mI = -INFINITY, lI = 0.f;
  for (int i = 0; i < p.k; ++i) {
    const int blk = srow[i];
    if (blk < 0 || blk >= p.nB) continue;
    const int jb = blk * p.Bk, nk = min(p.Bk, p.Sk - jb);
    for (int c0 = 0; c0 < nk; c0 += kKC) {
      const int nc = min(kKC, nk - c0);
      stage(jb + c0, nc, false);
      for (int jj = 0; jj < nc; ++jj) {
        const float s = index_logit(jj);
        if (jb + c0 + jj > pos) continue;
        const float mn = fmaxf(mI, s);
        lI = lI * exp2f(mI - mn) + exp2f(s - mn);
        mI = mn;
      }
    }
  }
  const float lseI = mI == -INFINITY ? 0.f : mI + log2f(lI);

  // pass 2: target, index probabilities, loss and gradients
  float lsum = 0.f;
  const float inv_g = 1.f / p.G;
  for (int i = 0; i < p.k; ++i) {
    const int blk = srow[i];
    if (blk < 0 || blk >= p.nB) continue;
    const int jb = blk * p.Bk, nk = min(p.Bk, p.Sk - jb);
    for (int c0 = 0; c0 < nk; c0 += kKC) {
      const int nc = min(kKC, nk - c0);
      stage(jb + c0, nc, true);
      float pt[kKC];
#pragma unroll
      for (int jj = 0; jj < kKC; ++jj) pt[jj] = 0.f;
      for (int hh = 0; hh < p.G; ++hh) {
        float qh[DPT];
#pragma unroll
        for (int x = 0; x < DPT; ++x)
          qh[x] = active ? to_f32(qrow[(size_t)hh * D + 4 * sub + 4 * kTPR * (x / 4) + (x % 4)]) *
                               p.sm_scale * kLog2e
                         : 0.f;
#pragma unroll
        for (int jj = 0; jj < kKC; ++jj) {
          const float4* kr = reinterpret_cast<const float4*>(ks + jj * D) + sub;
          float z = 0.f;
#pragma unroll
          for (int x = 0; x < DPT / 4; ++x) {
            const float4 kk = kr[kTPR * x];
            z = fmaf(qh[4 * x], kk.x, fmaf(qh[4 * x + 1], kk.y,
                fmaf(qh[4 * x + 2], kk.z, fmaf(qh[4 * x + 3], kk.w, z))));
          }
#pragma unroll
          for (int o = 1; o < kTPR; o <<= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
          pt[jj] += exp2f(z - lse2[hh]);
        }
      }
#pragma unroll
      for (int jj = 0; jj < kKC; ++jj) {
        const float s = index_logit(jj);
        const bool vis = jj < nc && jb + c0 + jj <= pos;
        const float tgt = vis ? pt[jj] * inv_g : 0.f;
        const float log_pi = s - lseI;                      // log2 units
        const float pi = vis ? exp2f(log_pi) : 0.f;
        if (tgt > 0.f) lsum += tgt * (log2f(tgt) - log_pi) * kLn2;
        const float gj = (pi - tgt) * p.index_scale;
        const float4* kr = reinterpret_cast<const float4*>(iks + jj * DI) + sub;
#pragma unroll
        for (int x = 0; x < IPT / 4; ++x) {
          const float4 kk = kr[kTPR * x];
          dqi[4 * x] = fmaf(gj, kk.x, dqi[4 * x]);
          dqi[4 * x + 1] = fmaf(gj, kk.y, dqi[4 * x + 1]);
          dqi[4 * x + 2] = fmaf(gj, kk.z, dqi[4 * x + 2]);
          dqi[4 * x + 3] = fmaf(gj, kk.w, dqi[4 * x + 3]);
        }
        if (sub == 0) gs[rl * kKC + jj] = gj;
      }
      __syncthreads();
      // d idx_k of the chunk's keys: thread (key jj, dims 4 s + 32 x .. +3) sums over the
      // 64 tokens (conflict-free float4 reads), then vector atomics
      {
        constexpr int TPK = kThreads / kKC;
        constexpr int NV = DI / (4 * TPK);
        const int jj = threadIdx.x / TPK, sl = threadIdx.x % TPK;
        if (jj < nc) {
          float4 a[NV];
#pragma unroll
          for (int x = 0; x < NV; ++x) a[x] = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int r = 0; r < kTok; ++r) {
            const float gv = gs[r * kKC + jj];
            if (gv == 0.f) continue;
            const float4* q4 = reinterpret_cast<const float4*>(iqs + r * DI) + sl;
#pragma unroll
            for (int x = 0; x < NV; ++x) {
              const float4 v4 = q4[TPK * x];
              a[x].x = fmaf(gv, v4.x, a[x].x); a[x].y = fmaf(gv, v4.y, a[x].y);
              a[x].z = fmaf(gv, v4.z, a[x].z); a[x].w = fmaf(gv, v4.w, a[x].w);
            }
          }
          float4* dst = reinterpret_cast<float4*>(dik + ((size_t)b * p.Sk + jb + c0 + jj) * DI) + sl;
#pragma unroll
          for (int x = 0; x < NV; ++x) atomicAdd(dst + TPK * x, a[x]);
        }
      }
    }
  }
  if (active) {
    float* dst = diq + (((size_t)b * p.Sq + t) * p.Hkv + g) * DI;
#pragma unroll
    for (int i = 0; i < IPT / 4; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) dst[4 * sub + 4 * kTPR * i + e] = dqi[4 * i + e];
  }
  // the CTA's loss: one row's value counted once (sub 0), warp then CTA reduction
  float lv = sub == 0 ? lsum : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lv += __shfl_xor_sync(0xffffffffu, lv, o);
  if ((threadIdx.x & 31) == 0) loss_part[threadIdx.x >> 5] = lv;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) tot += loss_part[w];
    atomicAdd(loss, tot);
  }
}

template <typename T, int D, int DI>
cudaError_t kl(const Dims& p, const void* q, const void* k, const float* lse, const void* iq,
               const void* ik, const int32_t* sel, float* loss, float* diq, float* dik,
               cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(loss, 0, sizeof(float), st);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(dik, 0, (size_t)p.B * p.Sk * DI * sizeof(float), st);
  if (e != cudaSuccess) return e;
  const size_t smem = ((size_t)kKC * D + (size_t)kKC * DI + (size_t)kTok * DI +
                       (size_t)kTok * kKC) * sizeof(float);
  auto kern = index_kl_simt<T, D, DI>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.Qt + kTok - 1) / kTok, p.nR, p.B * p.Hkv);
  kern<<<grid, kThreads, smem, st>>>((const T*)q, (const T*)k, lse, (const T*)iq, (const T*)ik,
                                     sel, loss, diq, dik, p);
  return cudaGetLastError();
}

}  // namespace

size_t index_kl_workspace_bytes(const Dims& p) {
  return index_kl_tc_supported(p) ? index_kl_tc_workspace_bytes(p) : 0;
}

cudaError_t launch_index_kl(const Dims& p, const void* q, const void* k, const float* lse,
                            const void* idx_q, const void* idx_k, const int32_t* sel,
                            float* loss, float* d_idx_q, float* d_idx_k, void* workspace,
                            cudaStream_t st, int* status) {
  if (index_kl_tc_supported(p))
    return launch_index_kl_tc(p, q, k, lse, idx_q, idx_k, sel, loss, d_idx_q, d_idx_k, workspace,
                              st, status);
  if (p.dtype == 1) {
    if (p.d == 128)
      return p.dI == 128 ? kl<__nv_bfloat16, 128, 128>(p, q, k, lse, idx_q, idx_k, sel, loss,
                                                       d_idx_q, d_idx_k, st)
                         : kl<__nv_bfloat16, 128, 64>(p, q, k, lse, idx_q, idx_k, sel, loss,
                                                      d_idx_q, d_idx_k, st);
    return p.dI == 128 ? kl<__nv_bfloat16, 64, 128>(p, q, k, lse, idx_q, idx_k, sel, loss,
                                                    d_idx_q, d_idx_k, st)
                       : kl<__nv_bfloat16, 64, 64>(p, q, k, lse, idx_q, idx_k, sel, loss,
                                                   d_idx_q, d_idx_k, st);
  }
  if (p.d == 128)
    return p.dI == 128 ? kl<float, 128, 128>(p, q, k, lse, idx_q, idx_k, sel, loss, d_idx_q,
                                             d_idx_k, st)
                       : kl<float, 128, 64>(p, q, k, lse, idx_q, idx_k, sel, loss, d_idx_q,
                                            d_idx_k, st);
  return p.dI == 128 ? kl<float, 64, 128>(p, q, k, lse, idx_q, idx_k, sel, loss, d_idx_q,
                                          d_idx_k, st)
                     : kl<float, 64, 64>(p, q, k, lse, idx_q, idx_k, sel, loss, d_idx_q,
                                         d_idx_k, st);
}

}  // namespace msa
