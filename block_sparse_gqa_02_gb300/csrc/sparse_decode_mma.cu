// Main branch of MSA, decode: the new token of each sequence attends, for each KV head, over
// the blocks that head selected (aietalks.com, "MSA uses a lightweight index branch before
// sparse attention"; per-token selection in decode).  Memory-bound: each selected 128-key
// K/V block (2 x 32 KiB, contiguous per head) is read once and shared by the G query heads
// of its group.
//
// One token's G <= 16 query heads of a group form exactly the M = 16 rows of
// mma.sync.m16n8k16, so the Q.K^T and P.V products run on the tensor cores with no padding
// beyond G; the tcgen05 UMMA shapes start at M = 64 and would waste most of the array here.
// CTA = (sequence, KV head, split of its selected blocks).  A TMA producer warp streams the
// split's K and V blocks (128-byte swizzle) through a 2-stage ring; 4 compute warps each
// take 32 keys of every block, keep S, P and O in registers (flash-attention style online
// softmax, log2 domain), then merge their partial (max, sum, O) through shared memory and
// write the split's normalised partial output and natural-log lse for the log-sum-exp merge.
#include "common.cuh"
#include "ptx.cuh"
#include "sparse_decode_mma.cuh"
#include "tma_host.cuh"

namespace msa {

namespace {

constexpr int kD = 128;
constexpr int kBk = 128;
constexpr int kRowBytes = 128;
constexpr int kBlockBytes = 2 * kBk * kRowBytes;   // one K or V block: [chunk][128][128 B]
constexpr int kStages = 2;
constexpr int kComputeWarps = 4;
constexpr int kThreads = (kComputeWarps + 1) * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// The warps' partial outputs reuse the K/V ring once every copy into it has landed.
struct __align__(1024) Smem {
  union {
    struct {
      uint8_t k[kStages][kBlockBytes];
      uint8_t v[kStages][kBlockBytes];
    };
    float o[kComputeWarps][16][kD + 4];
  };
  uint64_t full[kStages], empty[kStages];
  float m[kComputeWarps][16];
  float l[kComputeWarps][16];
  int abort;
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Address of the 16-byte unit u (8 dims) of row `row` in a [chunk][128 rows][128 B] tile
// written by TMA with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int u) {
  return base + (u >> 3) * (kBk * kRowBytes) + row * kRowBytes + (((u & 7) ^ (row & 7)) << 4);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreads)
sparse_decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ sel,
                         float* __restrict__ ws_o, float* __restrict__ ws_l, Dims p, int n_split,
                         int per, int* status) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, bg = blockIdx.y, b = bg / p.Hkv, g = bg % p.Hkv;
  const int G = p.G;
  const int32_t* srow = sel + (size_t)bg * p.k;
  const int i0 = split * per, i1 = min(p.k, i0 + per);
  const int L = seq_len_of(p, b);                          // this sequence's cache length
  const int nB_b = (L + kBk - 1) / kBk;
  const volatile int* abort = &s.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(&s.full[i], 1);
      ptx::mbar_init(&s.empty[i], kComputeWarps);
    }
    s.abort = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();

  // the split's valid blocks, in order (entries < 0 or >= nB are skipped)
  auto block_at = [&](int i) { return srow[i]; };
  auto valid = [&](int blk) { return blk >= 0 && blk < nB_b; };

  // a compute warp's running output, row maxima and row sums (rows gr and gr + 8)
  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

  int issued = 0;                                          // producer: copies issued
  if (warp == kComputeWarps) {
    // ------------------------------------------------------------- TMA producer
    int& j = issued;
    bool ok = true;
    for (int i = i0; i < i1; ++i) {
      const int blk = block_at(i);
      if (!valid(blk)) continue;
      const int st = j % kStages;
      if (!ptx::mbar_wait(&s.empty[st], ((j / kStages) & 1) ^ 1, abort)) { ok = false; break; }
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&s.full[st], 2 * kBlockBytes);
        // contiguous cache: (dims, key, sequence*Hkv + g); paged pool [P, Hkv, 128, d]:
        // (dims, key in block, physical block*Hkv + g)
        const int y = p.block_table ? 0 : blk * kBk;
        const int z = p.block_table ? p.block_table[(size_t)b * p.nB + blk] * p.Hkv + g : bg;
        debug_check(y >= 0 && y < p.Sk && z >= 0 &&
                        z < (p.block_table ? p.n_phys * p.Hkv : p.B * p.Hkv),
                    status, kDbgCoord);
        for (int kc = 0; kc < 2; ++kc) {
          ptx::tma_load_3d(s.k[st] + kc * kBk * kRowBytes, &tm_k, &s.full[st], kc * 64, y, z);
          ptx::tma_load_3d(s.v[st] + kc * kBk * kRowBytes, &tm_v, &s.full[st], kc * 64, y, z);
        }
      }
      ++j;
      __syncwarp();
    }
    if (!ok && lane == 0) {
      s.abort = 1;
      if (status) atomicExch(status, 0x401);
    }
  } else {
    // ------------------------------------------------------------ compute warps
    const int gr = lane >> 2, c = lane & 3;                  // fragment row / column pair
    const float c1 = p.sm_scale * kLog2e;
    // Q as A fragments: rows = query heads of the group (zero beyond G), 8 k-steps of 16 dims
    uint32_t qa[8][4];
    {
      const __nv_bfloat16* qb = q + ((size_t)b * p.Hq + (size_t)g * G) * kD;
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(qb + (size_t)gr * kD);
      const uint32_t* q1 = reinterpret_cast<const uint32_t*>(qb + (size_t)(gr + 8) * kD);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qa[kk][0] = gr < G ? q0[kk * 8 + c] : 0u;
        qa[kk][1] = gr + 8 < G ? q1[kk * 8 + c] : 0u;
        qa[kk][2] = gr < G ? q0[kk * 8 + 4 + c] : 0u;
        qa[kk][3] = gr + 8 < G ? q1[kk * 8 + 4 + c] : 0u;
      }
    }
    bool ok = true;
    int j = 0;
    for (int i = i0; i < i1; ++i) {
      const int blk = block_at(i);
      if (!valid(blk)) continue;
      const int st = j % kStages;
      if (!ptx::mbar_wait(&s.full[st], (j / kStages) & 1, abort)) { ok = false; break; }
      const uint32_t kb = ptx::smem_u32(s.k[st]), vb = ptx::smem_u32(s.v[st]);
      const int key0 = warp * 32;                            // this warp's 32 keys
      // S = Q K^T: 16 rows x 32 keys (4 n-tiles of 8 keys)
      float sc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        const int row = key0 + nt * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < 8; kk += 2) {
          uint32_t bf[4];
          ldsm_x4(swz(kb, row, 2 * kk + (lane >> 3)), bf);
          mma_bf16_16816(sc[nt], qa[kk], bf[0], bf[1]);
          mma_bf16_16816(sc[nt], qa[kk + 1], bf[2], bf[3]);
        }
      }
      // mask keys beyond the cache and find the row maxima (rows gr and gr + 8)
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = blk * kBk + key0 + nt * 8 + 2 * c + (e & 1);
          float x = key < L ? sc[nt][e] * c1 : -INFINITY;
          sc[nt][e] = x;
          mx[e >> 1] = fmaxf(mx[e >> 1], x);
        }
      float alpha[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float m_new = fmaxf(m_run[r], mx[r]);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        alpha[r] = ex2(m_run[r] - m_use);
        m_run[r] = m_new;
        l_run[r] *= alpha[r];
        mx[r] = m_use;
      }
      // P = exp2(S - m), bf16 A fragments for P.V (k = keys)
      uint32_t pa[2][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const float p0 = ex2(sc[nt][0] - mx[0]), p1 = ex2(sc[nt][1] - mx[0]);
        const float p2 = ex2(sc[nt][2] - mx[1]), p3 = ex2(sc[nt][3] - mx[1]);
        l_run[0] += p0 + p1;
        l_run[1] += p2 + p3;
        pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(p0, p1);
        pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(p2, p3);
      }
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        o[nt][0] *= alpha[0];
        o[nt][1] *= alpha[0];
        o[nt][2] *= alpha[1];
        o[nt][3] *= alpha[1];
      }
      // O += P V: 2 k-steps of 16 keys x 16 n-tiles of 8 dims
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const int row = key0 + ks * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
        for (int nt = 0; nt < 16; nt += 2) {
          uint32_t bf[4];
          ldsm_x4_t(swz(vb, row, nt + (lane >> 4)), bf);
          mma_bf16_16816(o[nt], pa[ks], bf[0], bf[1]);
          mma_bf16_16816(o[nt + 1], pa[ks], bf[2], bf[3]);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&s.empty[st]);
      ++j;
    }
    if (!ok && lane == 0) {
      s.abort = 1;
      if (status) atomicExch(status, 0x402);
    }
  }
  // Every warp has left its loop, so the abort flag is final.  Without an abort the compute
  // warps consumed every copy; after one (set by the producer or by a compute warp that gave
  // up), the producer waits for its last copies, which may still be in flight, before the
  // ring's memory is reused for the merge.
  __syncthreads();
  if (warp == kComputeWarps && lane == 0 && *abort)
    for (int x = issued > kStages ? issued - kStages : 0; x < issued; ++x)
      ptx::mbar_wait_timed(&s.full[x % kStages], (x / kStages) & 1);
  __syncthreads();
  if (warp < kComputeWarps) {
    const int gr = lane >> 2, c = lane & 3;
    // this warp's partial state -> shared memory (row sums reduced over the quad)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
    }
    if (c == 0) {
      s.m[warp][gr] = m_run[0];
      s.m[warp][gr + 8] = m_run[1];
      s.l[warp][gr] = l_run[0];
      s.l[warp][gr + 8] = l_run[1];
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      s.o[warp][gr][nt * 8 + 2 * c] = o[nt][0];
      s.o[warp][gr][nt * 8 + 2 * c + 1] = o[nt][1];
      s.o[warp][gr + 8][nt * 8 + 2 * c] = o[nt][2];
      s.o[warp][gr + 8][nt * 8 + 2 * c + 1] = o[nt][3];
    }
  }
  __syncthreads();

  // merge the 4 warps: 16 rows x 128 dims over 128 threads (8 threads per row)
  if (threadIdx.x < kComputeWarps * 32) {
    const int r = threadIdx.x >> 3, d0 = (threadIdx.x & 7) * 16;
    float mt = -INFINITY;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) mt = fmaxf(mt, s.m[w][r]);
    const float mu = mt == -INFINITY ? 0.f : mt;
    float lt = 0.f, wgt[kComputeWarps];
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) {
      wgt[w] = ex2(s.m[w][r] - mu);
      lt += wgt[w] * s.l[w][r];
    }
    const int h = g * G + r;
    if (r < G) {
      const size_t slot = ((size_t)b * p.Hq + h) * n_split + split;
      debug_check(h < p.Hq && split < n_split, status, kDbgStore);
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
      for (int dd = 0; dd < 16; ++dd) {
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kComputeWarps; ++w) acc = fmaf(wgt[w], s.o[w][r][d0 + dd], acc);
        ws_o[slot * kD + d0 + dd] = acc * inv;
      }
      if (d0 == 0) ws_l[slot] = lt > 0.f ? (mt + __log2f(lt)) * kLn2 : -INFINITY;
    }
  }
}

}  // namespace

bool sparse_decode_mma_supported(const Dims& p) {
  return p.dtype == 1 && p.decode && p.d == kD && p.Bk == kBk && p.G <= 16;
}

cudaError_t launch_sparse_decode_mma(const Dims& p, const void* q, const void* k, const void* v,
                                     const int32_t* sel, float* ws_o, float* ws_l, int n_split,
                                     int per, cudaStream_t st, int* status) {
  CUtensorMap tk, tv;
  // contiguous caches [B, Hkv, L, d] as (d, L, B*Hkv); paged pools [P, Hkv, 128, d] as
  // (d, 128, P*Hkv)
  const uint64_t rows = p.block_table ? (uint64_t)kBk : (uint64_t)p.Sk;
  const uint64_t outer = p.block_table ? (uint64_t)p.n_phys * p.Hkv : (uint64_t)p.B * p.Hkv;
  const uint64_t kd[3] = {(uint64_t)kD, rows, outer};
  const uint64_t ks[2] = {(uint64_t)kD * 2, rows * kD * 2};
  const uint32_t kbx[3] = {64, (uint32_t)kBk, 1};
  cudaError_t e = make_tensor_map_bf16(&tk, k, 3, kd, ks, kbx);
  if (e == cudaSuccess) e = make_tensor_map_bf16(&tv, v, 3, kd, ks, kbx);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(Smem) + 1024;
  e = cudaFuncSetAttribute(sparse_decode_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(n_split, p.B * p.Hkv);
  sparse_decode_mma_kernel<<<grid, kThreads, smem, st>>>(tk, tv, (const __nv_bfloat16*)q, sel,
                                                         ws_o, ws_l, p, n_split, per, status);
  return cudaGetLastError();
}

}  // namespace msa
