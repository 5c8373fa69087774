// Training, on the tcgen05 tensor cores: gradients of MSA's main branch, the sparse
// attention over the selected blocks (the pages mention kernels for training as well as
// inference: "Sparse Attention Cannot Be Directly Ported Across Architectures", paragraph
// "MSA addresses these issues"; aietalks.com, section "Block-level retrieval makes sparse
// attention easier to run on GPUs").  bf16 inputs, head_dim 128, 128-key blocks, 64-query
// tiles; fp32 accumulation and outputs.
//
// For a query row (token t, head h of KV group g) over its keys J (selected blocks, j <= t):
//   p_j = 2^(c1 s_j - lse2)  (s_j = q.k_j, c1 = sm_scale log2 e, lse2 = lse log2 e),
//   D = dout . out,  ds_j = p_j (dout . v_j - D),
//   dq = sm_scale sum_j ds_j k_j,  dk_j += sm_scale ds_j q,  dv_j += p_j dout.
//
// Two kernels, each accumulating in TMEM so that no partial product goes through HBM:
// * dQ (query-outer, one CTA per 128 (token, head) rows of a tile, as in the forward): per
//   selected block S = Q K^T and dP = dO V^T into TMEM, the softmax warps form dS (bf16, in
//   TMEM) and dQ += dS K accumulates in TMEM.  It also writes each 128-row group's lse2 and
//   D, in row order, as one 1 KiB record for the second kernel.
// * dK, dV (key-outer, one CTA per (sequence, KV head, key block, range of query tiles)):
//   the tiles that selected the block are read from a bitmap built first; for every 128-row
//   group of those tiles S^T = K Q^T and dP^T = V dO^T go to TMEM (keys on the TMEM lanes),
//   the elementwise warps form P^T there and release it (so dV += P^T dO, and the next
//   group's S^T, run while they go on), then dS^T (dK += dS^T Q); dK and dV accumulate in
//   TMEM over all of the CTA's groups.  A CTA adds its dK / dV to the fp32 outputs with
//   vector atomics (a heavily selected block is split over several CTAs).
// Warps: 16 elementwise warps (four per TMEM lane quadrant, each taking a quarter of the
// columns of S / dP or S^T / dP^T: with two, the warps waited mostly on the latency of their
// own loads and exponentials), a TMA producer and MMA issuers (a single thread's stream of
// N = 128 MMAs with commits in it keeps the tensor core busy only ~60 % of the time): three
// in the dQ kernel (S, dP, dQ), whose elementwise warps release S / dP as soon as they have
// loaded them so the next block's products run while dS is formed; two in the dK / dV
// kernel.  Every wait is bounded.
#include "common.cuh"
#include "ptx.cuh"
#include "sparse_backward_tc.cuh"
#include "tma_host.cuh"

namespace msa {

namespace {

constexpr int kD = 128;
constexpr int kBk = 128;
constexpr int kQt = 64;
constexpr int kRows = 128;                              // rows of one Q group
constexpr int kRowBytes = 128;
constexpr int kTileBytes = 2 * kRows * kRowBytes;       // [2 chunks][128 rows][128 B] = 32 KiB
constexpr int kMaxSel = 256;
constexpr int kMathWarps = 16;                          // four per TMEM lane quadrant
constexpr int kProducerWarp = kMathWarps, kMmaWarp = kMathWarps + 1;   // first MMA issuer: 17
constexpr int kThreads = (kMathWarps + 3) * 32;
constexpr int kDqThreads = (kMathWarps + 4) * 32;     // dQ pass: three MMA issuers
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescKK = ptx::idesc_bf16_f32(128, 128, 0, 0);   // both operands K-major
constexpr uint32_t kIdescMN = ptx::idesc_bf16_f32(128, 128, 0, 1);   // B MN-major
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxTilesPerCta = 2048;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed pairs of fp32 (one 64-bit register) for the paired FMA / ADD / MUL instructions.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void split_f32x2(uint64_t x, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// D[tmem] (+)= A[smem, K-major] B[smem, K-major]^T over 128 dims (8 steps of 16): S = Q K^T
// in the dQ kernel, S^T = K Q^T in the dK/dV kernel.
__device__ __forceinline__ void mma_kk(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t off = (kk >> 2) * (kRows * kRowBytes) + (kk & 3) * 32;
    ptx::umma_bf16_ss(d_tmem, ptx::smem_desc_k_sw128(a_smem + off),
                      ptx::smem_desc_k_sw128(b_smem + off), kIdescKK, kk > 0 ? 1u : 0u);
  }
}

// D[tmem] (+)= A[tmem, 128 x 128 bf16] B[smem, MN-major 128 x 128], the reduction over the
// 128 rows of B: dQ += dS K, dV += P^T dO, dK += dS^T Q.  When split, A's 32-row chunk c
// (16 packed columns) sits at columns 32c .. 32c+15 of its region (the columns the chunk's
// fp32 values came from); else the chunks follow one another.
__device__ __forceinline__ void mma_tmn(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem,
                                        bool accumulate, bool split = false) {
#pragma unroll
  for (int kk = 0; kk < 128 / 16; ++kk)
    ptx::umma_bf16_ts(d_tmem, a_tmem + (split ? 32 * (kk >> 1) + (kk & 1) * 8 : kk * 8),
                      ptx::smem_desc_mn_sw128(b_smem + kk * 16 * kRowBytes, kRows * kRowBytes, 1024),
                      kIdescMN, (accumulate || kk > 0) ? 1u : 0u);
}


__device__ __forceinline__ void raise_abort(int* abort_flag, int* status, int code) {
  *abort_flag = 1;
  if (status) atomicExch(status, code);
}

// ============================================================================ bitmap
// bit (bg, blk, m) set when query tile m of (sequence, KV head) bg selected key block blk.
__global__ void selection_bitmap_kernel(const int32_t* __restrict__ sel,
                                        uint32_t* __restrict__ bits, Dims p, int words) {
  const size_t n = (size_t)p.B * p.Hkv * p.nR * p.k;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const int blk = sel[e];
    if (blk < 0 || blk >= p.nB) continue;
    const size_t row = e / p.k;                          // bg * nR + m
    const int m = (int)(row % p.nR);
    const size_t bg = row / p.nR;
    atomicOr(&bits[(bg * p.nB + blk) * words + (m >> 5)], 1u << (m & 31));
  }
}

// ============================================================================ dQ kernel

// dQ pass: K rides a three-stage ring (read by S and, a block later, by dQ), V a two-stage
// ring (read by dP only, so free as soon as dP completes); with Q and dO this fills the
// 227 KiB a CTA may use
constexpr int kKStages = 3;

struct __align__(1024) SmemQ {
  uint8_t q[kTileBytes];
  uint8_t dO[kTileBytes];
  uint8_t k[kKStages][kTileBytes];
  uint8_t v[2][kTileBytes];
  uint64_t qd_full;
  uint64_t k_full[kKStages], k_empty[kKStages], v_full[2], v_empty[2];
  uint64_t s_full, s_free, ds_full, dq_done, drain[3];
  float dsum[kRows];
  int blocks[kMaxSel];
  int n_sel;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(SmemQ) + 1024 <= 227 * 1024, "dQ pass shared memory");


__global__ void __launch_bounds__(kDqThreads, 1)
backward_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const int32_t* __restrict__ sel, const __nv_bfloat16* __restrict__ out,
                      const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse,
                      float* __restrict__ dq, float* __restrict__ rowstat, Dims p,
                      int* status) {
  extern __shared__ uint8_t smem_raw[];
  SmemQ& s = *reinterpret_cast<SmemQ*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int part = blockIdx.x;                           // 128-row group of the tile
  const int m = p.nR - 1 - blockIdx.y;                   // heaviest tiles first
  const int bg = blockIdx.z, b = bg / p.Hkv, g = bg % p.Hkv;
  const int G = p.G;
  const int tok_per_group = kRows / G;
  const volatile int* abort = &s.abort;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&s.qd_full, 1);
    for (int i = 0; i < kKStages; ++i) {
      ptx::mbar_init(&s.k_full[i], 1);
      ptx::mbar_init(&s.k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s.v_full[i], 1);
      ptx::mbar_init(&s.v_empty[i], 1);
    }
    ptx::mbar_init(&s.s_full, 2);          // S and dP, one commit each
    ptx::mbar_init(&s.s_free, kMathWarps);
    ptx::mbar_init(&s.ds_full, kMathWarps);
    ptx::mbar_init(&s.dq_done, 1);
    for (int i = 0; i < 3; ++i) ptx::mbar_init(&s.drain[i], 1);
    s.abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&s.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 1) {
    // this tile's selection, entries < 0 or >= nB dropped, order kept
    const int32_t* srow = sel + ((size_t)bg * p.nR + m) * p.k;
    int n = 0;
    for (int i0 = 0; i0 < p.k; i0 += 32) {
      const int i = i0 + lane;
      const int blk = i < p.k ? srow[i] : -1;
      const bool ok = blk >= 0 && blk < p.nB;
      const unsigned mask = __ballot_sync(0xffffffffu, ok);
      if (ok) s.blocks[n + __popc(mask & ((1u << lane) - 1))] = blk;
      n += __popc(mask);
    }
    if (lane == 0) s.n_sel = n;
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = s.tmem_base;
  const int n_sel = s.n_sel;
  // TMEM columns: S [0,128), dP [128,256), dQ [256,384), dS (bf16) [384,448)
  constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------- TMA producer
    int issued_v = 0, issued_k = 0;
    bool ok = true;
    // test hook: issue nothing, so the consumers' bounded waits run out
    const int n_load = p.inject == 1 ? 0 : n_sel;
    if (lane == 0 && n_load > 0) {
      ptx::mbar_arrive_expect_tx(&s.qd_full, 2 * kTileBytes);
      const int t0 = m * kQt + part * tok_per_group;
      for (int kc = 0; kc < 2; ++kc) {
        ptx::tma_load_4d(s.q + kc * kRows * kRowBytes, &tm_q, &s.qd_full, kc * 64, g * G, t0, b);
        ptx::tma_load_4d(s.dO + kc * kRows * kRowBytes, &tm_do, &s.qd_full, kc * 64, g * G, t0,
                         b);
      }
    }
    for (int j = 0; j < n_load; ++j) {
      const int blk = s.blocks[j];
      const int sv = j & 1, sk = j % kKStages;
      if (!ptx::mbar_wait(&s.v_empty[sv], ((j >> 1) & 1) ^ 1, abort)) { ok = false; break; }
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&s.v_full[sv], kTileBytes);
        for (int kc = 0; kc < 2; ++kc)
          ptx::tma_load_3d(s.v[sv] + kc * kBk * kRowBytes, &tm_v, &s.v_full[sv], kc * 64,
                           blk * kBk, bg);
      }
      issued_v = j + 1;
      __syncwarp();
      if (!ptx::mbar_wait(&s.k_empty[sk], ((j / kKStages) & 1) ^ 1, abort)) { ok = false; break; }
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&s.k_full[sk], kTileBytes);
        for (int kc = 0; kc < 2; ++kc)
          ptx::tma_load_3d(s.k[sk] + kc * kBk * kRowBytes, &tm_k, &s.k_full[sk], kc * 64,
                           blk * kBk, bg);
      }
      issued_k = j + 1;
      __syncwarp();
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x501);
    if (*abort && lane == 0 && n_load > 0) {
      ptx::mbar_wait_timed(&s.qd_full, 0);
      for (int j = issued_v > 2 ? issued_v - 2 : 0; j < issued_v; ++j)
        ptx::mbar_wait_timed(&s.v_full[j & 1], (j >> 1) & 1);
      for (int j = issued_k > kKStages ? issued_k - kKStages : 0; j < issued_k; ++j)
        ptx::mbar_wait_timed(&s.k_full[j % kKStages], (j / kKStages) & 1);
    }
  } else if (warp >= kMmaWarp && warp <= kMmaWarp + 2) {
    // ------------------------------------------------------------- MMA issuers
    // the first: S = Q K^T of each block, the second: dP = dO V^T (each into TMEM once the
    // math warps have read the previous block's), the third: dQ += dS K once the math warps
    // have written dS.  One thread's stream of N = 128 MMAs with commits runs at ~105 clocks
    // an MMA, so S and dP (16 MMAs a block) on one thread held the block back; on two, the
    // next block's S and dP run while this block's elementwise step forms dS.
    const int who = warp - kMmaWarp;
    bool ok = true, issued_any = false;
    const uint32_t qa = ptx::smem_u32(s.q), da = ptx::smem_u32(s.dO);
    if (n_sel > 0 && who < 2) {
      ok = ptx::mbar_wait(&s.qd_full, 0, abort);
      for (int j = 0; ok && j < n_sel; ++j) {
        // S (first issuer) or dP (second) of block j once the math warps have read block j-1's
        if ((who == 0 ? !ptx::mbar_wait(&s.k_full[j % kKStages], (j / kKStages) & 1, abort)
                      : !ptx::mbar_wait(&s.v_full[j & 1], (j >> 1) & 1, abort)) ||
            (j > 0 && !ptx::mbar_wait(&s.s_free, (j - 1) & 1, abort))) { ok = false; break; }
        ptx::tc_fence_after_sync();
        if (lane == 0) {
          if (who == 0) {
            mma_kk(tmem + kColS, qa, ptx::smem_u32(s.k[j % kKStages]));
            ptx::umma_commit(&s.s_full);
          } else {
            mma_kk(tmem + kColDP, da, ptx::smem_u32(s.v[j & 1]));
            ptx::umma_commit(&s.s_full);
            ptx::umma_commit(&s.v_empty[j & 1]);           // dP was the only reader of V
          }
        }
        issued_any = true;
        __syncwarp();
      }
    } else if (n_sel > 0) {
      for (int j = 0; ok && j < n_sel; ++j) {
        if (!ptx::mbar_wait(&s.ds_full, j & 1, abort)) { ok = false; break; }
        ptx::tc_fence_after_sync();
        if (lane == 0) {
          mma_tmn(tmem + kColDQ, tmem + kColDS, ptx::smem_u32(s.k[j % kKStages]), j > 0);
          ptx::umma_commit(&s.dq_done);
          ptx::umma_commit(&s.k_empty[j % kKStages]);
        }
        issued_any = true;
        __syncwarp();
      }
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x502);
    if (*abort && lane == 0 && issued_any) {
      ptx::umma_commit(&s.drain[who]);                     // covers this thread's MMAs
      ptx::mbar_wait_timed(&s.drain[who], 0);
    }
  } else {
    // ------------------------- math warps 0-15: warp w takes row quadrant w % 4 and the key
    // columns (and dQ columns) 32 (w / 4) .. +31
    const int quad = warp & 3, half = warp >> 2;
    const int r = quad * 32 + lane;
    const int R = part * kRows + r;                      // row within the tile's Qt*G rows
    const int t = m * kQt + R / G;
    const int h = g * G + R % G;
    const bool valid = t < p.Sq;
    const float c1 = p.sm_scale * kLog2e;
    const size_t row_off = (((size_t)b * p.Sq + (valid ? t : 0)) * p.Hq + h) * kD;
    // D = dout . out of this row, formed by the quadrant's first warp and shared (every warp
    // of the quadrant needs it)
    float dsum = 0.f;
    if (valid && half == 0) {
      const uint4* o4 = reinterpret_cast<const uint4*>(out + row_off);
      const uint4* d4 = reinterpret_cast<const uint4*>(dout + row_off);
#pragma unroll 4
      for (int x = 0; x < kD / 8; ++x) {
        const uint4 a = o4[x], c = d4[x];
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[e]));
          const float2 fc = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&cv[e]));
          dsum = fmaf(fa.x, fc.x, fmaf(fa.y, fc.y, dsum));
        }
      }
    }
    if (half == 0) s.dsum[r] = dsum;
    asm volatile("bar.sync 1, %0;" ::"r"(kMathWarps * 32) : "memory");
    dsum = s.dsum[r];
    const float lse2 = valid ? lse[((size_t)b * p.Hq + h) * p.Sq + t] * kLog2e : INFINITY;
    if (half == 0) {
      // the group's record for the dK/dV pass: lse2 of its 128 rows, then their D
      float* rec = rowstat + (((size_t)bg * p.nR + m) * gridDim.x + part) * 2 * kRows;
      rec[r] = -lse2;                                    // negated: the dK/dV pass adds them
      rec[kRows + r] = -dsum;
    }
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    bool ok = true;
    for (int j = 0; j < n_sel; ++j) {
      const int blk = s.blocks[j];
      if (!ptx::mbar_wait(&s.s_full, j & 1, abort)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      const int lim = t - blk * kBk;                       // visible columns: c <= lim
      uint32_t sv[32], dv[32];
      ptx::tmem_ld_x32(tmem + lane_off + kColS + half * 32, sv);
      ptx::tmem_ld_x32(tmem + lane_off + kColDP + half * 32, dv);
      ptx::tmem_ld_wait();
      // this warp's S / dP columns are in registers: the next block may overwrite them
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&s.s_free);
      // The Q / dO barrier's only phase has completed, so this wait returns at once.  It is
      // here because it is a loop: without it the compiler schedules the exponentials below
      // ahead of the arrive, and the next block's S and dP wait for the whole elementwise
      // step (measured: 2.9K instead of 2.3K clocks a block).
      if (!ptx::mbar_wait(&s.qd_full, 0, abort)) { ok = false; break; }
      uint32_t pk[16];
      const uint64_t c1x2 = f32x2(c1, c1), nl2 = f32x2(-lse2, -lse2), nd2 = f32x2(-dsum, -dsum);
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        // two columns at a time in paired fp32
        float y0, y1;
        split_f32x2(fma_f32x2(f32x2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c1x2,
                              nl2), y0, y1);
        const float p0 = half * 32 + e <= lim ? ex2(y0) : 0.f;
        const float p1 = half * 32 + e + 1 <= lim ? ex2(y1) : 0.f;
        float d0, d1;
        split_f32x2(mul_f32x2(f32x2(p0, p1),
                              add_f32x2(f32x2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])),
                                        nd2)),
                    d0, d1);
        pk[e >> 1] = pack_bf16x2(d0, d1);
      }
      // the previous block's dQ MMA has finished reading dS (it ran while these were formed)
      if (j > 0 && !ptx::mbar_wait(&s.dq_done, (j - 1) & 1, abort)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      ptx::tmem_st_x16(tmem + lane_off + kColDS + half * 16, pk);
      ptx::tmem_st_wait();
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&s.ds_full);
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x503);
    bool have = ok && n_sel > 0 && ptx::mbar_wait(&s.dq_done, (n_sel - 1) & 1, abort);
    if (ok && n_sel > 0 && !have && lane == 0) raise_abort(&s.abort, status, 0x504);
    if (have) ptx::tc_fence_after_sync();
    // dq = sm_scale * dQ (zero for a row with no visible key), this warp's 32 columns;
    // tcgen05.ld is warp-collective, so every lane loads (`have` is the same in the whole
    // warp) and valid rows store
    float4* dst = reinterpret_cast<float4*>(dq + row_off);
#pragma unroll 1
    for (int u = 0; u < 1; ++u) {
      const int c = half + u;
      uint32_t v[32];
      if (have) {
        ptx::tmem_ld_x32(tmem + lane_off + kColDQ + c * 32, v);
        ptx::tmem_ld_wait();
      }
      if (valid) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          dst[c * 8 + e / 4] = have ? make_float4(__uint_as_float(v[e]) * p.sm_scale,
                                                  __uint_as_float(v[e + 1]) * p.sm_scale,
                                                  __uint_as_float(v[e + 2]) * p.sm_scale,
                                                  __uint_as_float(v[e + 3]) * p.sm_scale)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ======================================================================= dK / dV kernel

struct __align__(1024) SmemKV {
  uint8_t k[kTileBytes];
  uint8_t v[kTileBytes];
  uint8_t q[2][kTileBytes];
  uint8_t dO[2][kTileBytes];
  float rec[2][2 * kRows];       // a group's -lse2 [0,128) and -D [128,256), per stage
  uint64_t kv_full, g_full[2], g_empty[2];
  uint64_t s_full_s, s_full_dp, p_full_p, p_full_ds, acc_dk, acc_dv, drain[2];
  int tiles[kMaxTilesPerCta];
  int n_tiles;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(kThreads, 1)
backward_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_do,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const uint32_t* __restrict__ bits, const float* __restrict__ rowstat,
                        float* __restrict__ dk,
                        float* __restrict__ dv, Dims p, int words, int words_per_cta,
                        int* status) {
  extern __shared__ uint8_t smem_raw[];
  SmemKV& s = *reinterpret_cast<SmemKV*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x, blk = blockIdx.y, bg = blockIdx.z;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int G = p.G;
  const int parts = p.Qt * G / kRows;                    // 128-row groups per tile
  const int tok_per_group = kRows / G;

  // the tiles of this CTA's range that selected the block, ascending
  if (warp == 0) {
    const uint32_t* row = bits + ((size_t)bg * p.nB + blk) * words;
    const int w0 = chunk * words_per_cta, w1 = min(words, w0 + words_per_cta);
    int n = 0;
    for (int wb = w0; wb < w1; wb += 32) {
      const int w = wb + lane;
      const uint32_t word = w < w1 ? row[w] : 0u;
      const int cnt = __popc(word);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int pos = n + incl - cnt;
      for (uint32_t x = word; x; x &= x - 1) s.tiles[pos++] = w * 32 + __ffs(x) - 1;
      n += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s.n_tiles = n;
  }
  __syncthreads();
  const int n_tiles = s.n_tiles;
  if (n_tiles == 0) return;                              // the whole CTA leaves together
  const int n_groups = n_tiles * parts;
  const volatile int* abort = &s.abort;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&s.kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s.g_full[i], 1);
      ptx::mbar_init(&s.g_empty[i], 2);   // both issuers' MMAs read the group
    }
    ptx::mbar_init(&s.s_full_s, 1);         // S^T landed
    ptx::mbar_init(&s.s_full_dp, 1);        // dP^T landed
    ptx::mbar_init(&s.p_full_p, kMathWarps);    // P^T written
    ptx::mbar_init(&s.p_full_ds, kMathWarps);   // dS^T written
    ptx::mbar_init(&s.acc_dk, 1);
    ptx::mbar_init(&s.acc_dv, 1);
    ptx::mbar_init(&s.drain[0], 1);
    ptx::mbar_init(&s.drain[1], 1);
    s.abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&s.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = s.tmem_base;
  // TMEM columns: dV [0,128), dK [128,256), S^T [256,384) (P^T bf16 over its first 64),
  // dP^T [384,512) (dS^T bf16 over its first 64)
  constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 384;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------- TMA producer
    int issued = 0;
    bool ok = true;
    if (lane == 0) {
      ptx::mbar_arrive_expect_tx(&s.kv_full, 2 * kTileBytes);
      for (int kc = 0; kc < 2; ++kc) {
        ptx::tma_load_3d(s.k + kc * kBk * kRowBytes, &tm_k, &s.kv_full, kc * 64, blk * kBk, bg);
        ptx::tma_load_3d(s.v + kc * kBk * kRowBytes, &tm_v, &s.kv_full, kc * 64, blk * kBk, bg);
      }
    }
    for (int gi = 0; gi < n_groups; ++gi) {
      const int st = gi & 1;
      if (!ptx::mbar_wait(&s.g_empty[st], ((gi >> 1) & 1) ^ 1, abort)) { ok = false; break; }
      const int m = s.tiles[gi / parts], part = gi % parts;
      if (lane == 0) {
        // the group's per-row lse2 and D (+inf / 0 past the sequence), written in row order
        // by the dQ pass, and its Q and dO rows
        ptx::mbar_arrive_expect_tx(&s.g_full[st], 2 * kTileBytes + 2 * kRows * 4);
        ptx::bulk_load(s.rec[st], rowstat + (((size_t)bg * p.nR + m) * parts + part) * 2 * kRows,
                       2 * kRows * 4, &s.g_full[st]);
        const int t0 = m * kQt + part * tok_per_group;
        for (int kc = 0; kc < 2; ++kc) {
          ptx::tma_load_4d(s.q[st] + kc * kRows * kRowBytes, &tm_q, &s.g_full[st], kc * 64,
                           g * G, t0, b);
          ptx::tma_load_4d(s.dO[st] + kc * kRows * kRowBytes, &tm_do, &s.g_full[st], kc * 64,
                           g * G, t0, b);
        }
      }
      issued = gi + 1;
      __syncwarp();
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x601);
    if (*abort && lane == 0) {
      ptx::mbar_wait_timed(&s.kv_full, 0);
      for (int gi = issued > 2 ? issued - 2 : 0; gi < issued; ++gi)
        ptx::mbar_wait_timed(&s.g_full[gi & 1], (gi >> 1) & 1);
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ------------------------------------------------------------- MMA issuers
    // the first issuer: S^T = K Q^T, then dK += dS^T Q; the second: dP^T = V dO^T, then
    // dV += P^T dO.
    // P^T is written over S^T and read by dV, dS^T over dP^T and read by dK.  The first
    // issuer takes the S region (S^T, then dV once P^T is written), the second the dP
    // region (dP^T, then dK once dS^T is written): the math warps release P^T before they
    // form dS^T, so dV and the next group's S^T run while dS^T is being formed.  Each
    // issuer's next product overwrites what its own last one read, so it waits for that one.
    const int who = warp - kMmaWarp;
    bool ok = ptx::mbar_wait(&s.kv_full, 0, abort);
    bool issued_any = false;
    const uint32_t ka = ptx::smem_u32(s.k), va = ptx::smem_u32(s.v);
    uint64_t* my_acc = who == 0 ? &s.acc_dv : &s.acc_dk;
    uint64_t* my_sfull = who == 0 ? &s.s_full_s : &s.s_full_dp;
    uint64_t* my_pfull = who == 0 ? &s.p_full_p : &s.p_full_ds;
    for (int gi = 0; ok && gi < n_groups; ++gi) {
      const int st = gi & 1;
      if (!ptx::mbar_wait(&s.g_full[st], (gi >> 1) & 1, abort) ||
          (gi > 0 && !ptx::mbar_wait(my_acc, (gi - 1) & 1, abort))) { ok = false; break; }
      ptx::tc_fence_after_sync();
      if (lane == 0) {
        if (who == 0) mma_kk(tmem + kColS, ka, ptx::smem_u32(s.q[st]));
        else mma_kk(tmem + kColDP, va, ptx::smem_u32(s.dO[st]));
        ptx::umma_commit(my_sfull);
      }
      issued_any = true;
      __syncwarp();
      if (!ptx::mbar_wait(my_pfull, gi & 1, abort)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      if (lane == 0) {
        if (who == 0) mma_tmn(tmem + kColDV, tmem + kColS, ptx::smem_u32(s.dO[st]), gi > 0, true);
        else mma_tmn(tmem + kColDK, tmem + kColDP, ptx::smem_u32(s.q[st]), gi > 0, true);
        ptx::umma_commit(my_acc);
        ptx::umma_commit(&s.g_empty[st]);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x602);
    if (*abort && lane == 0 && issued_any) {
      ptx::umma_commit(&s.drain[who]);                     // covers this thread's MMAs
      ptx::mbar_wait_timed(&s.drain[who], 0);
    }
  } else {
    // ----------------- math warps 0-15: one key of the block per lane (quadrant w % 4); warp
    // w takes the group rows (and dV / dK columns) 32 (w / 4) .. +31
    const int quad = warp & 3, half = warp >> 2;
    const int key = blk * kBk + quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float c1 = p.sm_scale * kLog2e;
    bool ok = true;
    for (int gi = 0; gi < n_groups; ++gi) {
      const int st = gi & 1;
      const int m = s.tiles[gi / parts], part = gi % parts;
      // row x of the group holds token t0 + x / G; the key is masked for rows x < xlim
      const int t0 = m * kQt + part * tok_per_group;
      const int dj = key - t0;
      const int xlim = dj > 0 ? dj * G : 0;
      // g_full: the group's per-row lse2 / D have landed; then S^T
      if (!ptx::mbar_wait(&s.g_full[st], (gi >> 1) & 1, abort) ||
          !ptx::mbar_wait(&s.s_full_s, gi & 1, abort)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      const int c = half;                                  // this warp's 32-column chunk
      uint32_t sv[32];
      ptx::tmem_ld_x32(tmem + lane_off + kColS + c * 32, sv);
      ptx::tmem_ld_wait();
      // P^T, two rows at a time in paired fp32 (the record holds -lse2 and -D), released
      // to the dV product before dS^T is formed
      float pr[32];
      {
        uint32_t pp[16];
        const uint64_t c1x2 = f32x2(c1, c1);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int x = c * 32 + e;
          const uint64_t nl2 = *reinterpret_cast<const uint64_t*>(&s.rec[st][x]);
          float y0, y1;
          split_f32x2(fma_f32x2(f32x2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                c1x2, nl2), y0, y1);
          pr[e] = x >= xlim ? ex2(y0) : 0.f;
          pr[e + 1] = x + 1 >= xlim ? ex2(y1) : 0.f;
          pp[e >> 1] = pack_bf16x2(pr[e], pr[e + 1]);
        }
        // over columns this warp loaded: chunk c at columns 32c .. 32c+15
        ptx::tmem_st_x16(tmem + lane_off + kColS + 32 * c, pp);
        ptx::tmem_st_wait();
        ptx::tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&s.p_full_p);
      }
      // then dP^T and dS^T = P^T (dP^T - D)
      if (!ptx::mbar_wait(&s.s_full_dp, gi & 1, abort)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      uint32_t dpv[32];
      ptx::tmem_ld_x32(tmem + lane_off + kColDP + c * 32, dpv);
      ptx::tmem_ld_wait();
      {
        uint32_t dd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const uint64_t nd2 = *reinterpret_cast<const uint64_t*>(&s.rec[st][kRows + c * 32 + e]);
          float d0, d1;
          split_f32x2(mul_f32x2(f32x2(pr[e], pr[e + 1]),
                                add_f32x2(f32x2(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])), nd2)),
                      d0, d1);
          dd[e >> 1] = pack_bf16x2(d0, d1);
        }
        ptx::tmem_st_x16(tmem + lane_off + kColDP + 32 * c, dd);
        ptx::tmem_st_wait();
        ptx::tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&s.p_full_ds);
      }
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x603);
    bool have = ok && ptx::mbar_wait(&s.acc_dk, (n_groups - 1) & 1, abort) &&
                ptx::mbar_wait(&s.acc_dv, (n_groups - 1) & 1, abort);
    if (ok && !have && lane == 0) raise_abort(&s.abort, status, 0x604);
    if (have) {
      ptx::tc_fence_after_sync();
      const bool in_range = key < p.Sk;
      float4* dvr = reinterpret_cast<float4*>(dv + ((size_t)bg * p.Sk + (in_range ? key : 0)) * kD);
      float4* dkr = reinterpret_cast<float4*>(dk + ((size_t)bg * p.Sk + (in_range ? key : 0)) * kD);
#pragma unroll 1
      for (int u = 0; u < 1; ++u) {
        const int c = half + u;
        uint32_t a[32], bk[32];
        ptx::tmem_ld_x32(tmem + lane_off + kColDV + c * 32, a);
        ptx::tmem_ld_x32(tmem + lane_off + kColDK + c * 32, bk);
        ptx::tmem_ld_wait();
        if (in_range) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            atomicAdd(dvr + c * 8 + e / 4,
                      make_float4(__uint_as_float(a[e]), __uint_as_float(a[e + 1]),
                                  __uint_as_float(a[e + 2]), __uint_as_float(a[e + 3])));
            atomicAdd(dkr + c * 8 + e / 4,
                      make_float4(__uint_as_float(bk[e]) * p.sm_scale,
                                  __uint_as_float(bk[e + 1]) * p.sm_scale,
                                  __uint_as_float(bk[e + 2]) * p.sm_scale,
                                  __uint_as_float(bk[e + 3]) * p.sm_scale));
          }
        }
      }
    }
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_selection_bitmap(const Dims& p, const int32_t* sel, uint32_t* bits,
                                   cudaStream_t st) {
  const int words = (p.nR + 31) / 32;
  cudaError_t e = cudaMemsetAsync(bits, 0, (size_t)p.B * p.Hkv * p.nB * words * sizeof(uint32_t),
                                  st);
  if (e != cudaSuccess) return e;
  const size_t n = (size_t)p.B * p.Hkv * p.nR * p.k;
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  selection_bitmap_kernel<<<blocks, 256, 0, st>>>(sel, bits, p, words);
  return cudaGetLastError();
}

// Query tiles per key-block CTA: about nR / 16 (so a block every tile selected is split
// over ~16 CTAs), a multiple of 32 between 32 and kMaxTilesPerCta.
int tiles_per_cta(const Dims& p) {
  int t = (p.nR + 15) / 16;
  t = (t + 31) / 32 * 32;
  return t < 32 ? 32 : (t > kMaxTilesPerCta ? kMaxTilesPerCta : t);
}

bool sparse_backward_tc_supported(const Dims& p) {
  return p.dtype == 1 && !p.decode && p.d == kD && p.Bk == kBk && p.Qt == kQt && p.G >= 2 &&
         p.G <= kRows && (kRows % p.G) == 0 && p.k <= kMaxSel;
}

size_t sparse_backward_tc_workspace_bytes(const Dims& p) {
  // per 128-row group: lse2 and D of its rows (1 KiB), then the bitmap
  const size_t rowstat = (size_t)p.B * p.Hkv * p.nR * (p.Qt * p.G / kRows) * 2 * kRows * 4;
  const size_t words = (size_t)(p.nR + 31) / 32;
  const size_t bitmap = (size_t)p.B * p.Hkv * p.nB * words * sizeof(uint32_t);
  return rowstat + bitmap;
}

cudaError_t launch_sparse_backward_tc(const Dims& p, const void* q, const void* k,
                                      const void* v, const int32_t* sel, const void* out,
                                      const float* lse, const void* dout, float* dq, float* dk,
                                      float* dv, void* workspace, cudaStream_t st, int* status) {
  const size_t rowstat_bytes = (size_t)p.B * p.Hkv * p.nR * (p.Qt * p.G / kRows) * 2 * kRows * 4;
  float* rowstat = reinterpret_cast<float*>(workspace);
  uint32_t* bits = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(workspace) + rowstat_bytes);
  const int words = (p.nR + 31) / 32;
  const size_t kv_bytes = (size_t)p.B * p.Hkv * p.Sk * kD * sizeof(float);
  cudaError_t e = cudaMemsetAsync(dk, 0, kv_bytes, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, kv_bytes, st);
  if (e != cudaSuccess) return e;

  CUtensorMap tq, tdo, tk, tv;
  // q, dout [B, T, Hq, d] as (d, Hq, T, B); one box = 64 dims x G heads x (128 / G) tokens
  const uint64_t qd[4] = {(uint64_t)kD, (uint64_t)p.Hq, (uint64_t)p.Sq, (uint64_t)p.B};
  const uint64_t qs[3] = {(uint64_t)kD * 2, (uint64_t)p.Hq * kD * 2,
                          (uint64_t)p.Sq * p.Hq * kD * 2};
  const uint32_t qb[4] = {64, (uint32_t)p.G, (uint32_t)(kRows / p.G), 1};
  // k, v [B, Hkv, Sk, d] as (d, Sk, B * Hkv); one box = 64 dims x 128 keys
  const uint64_t kd[3] = {(uint64_t)kD, (uint64_t)p.Sk, (uint64_t)p.B * p.Hkv};
  const uint64_t ks[2] = {(uint64_t)kD * 2, (uint64_t)p.Sk * kD * 2};
  const uint32_t kb[3] = {64, (uint32_t)kBk, 1};
  e = make_tensor_map_bf16(&tq, q, 4, qd, qs, qb);
  if (e == cudaSuccess) e = make_tensor_map_bf16(&tdo, dout, 4, qd, qs, qb);
  if (e == cudaSuccess) e = make_tensor_map_bf16(&tk, k, 3, kd, ks, kb);
  if (e == cudaSuccess) e = make_tensor_map_bf16(&tv, v, 3, kd, ks, kb);
  if (e != cudaSuccess) return e;

  if ((e = launch_selection_bitmap(p, sel, bits, st)) != cudaSuccess) return e;
  {
    const size_t smem = sizeof(SmemQ) + 1024;
    e = cudaFuncSetAttribute(backward_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.Qt * p.G / kRows, p.nR, p.B * p.Hkv);
    backward_dq_tc_kernel<<<grid, kDqThreads, smem, st>>>(
        tq, tdo, tk, tv, sel, (const __nv_bfloat16*)out, (const __nv_bfloat16*)dout, lse, dq,
        rowstat, p, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    const size_t smem = sizeof(SmemKV) + 1024;
    e = cudaFuncSetAttribute(backward_dkdv_tc_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int wpc = tiles_per_cta(p) / 32;
    dim3 grid((words + wpc - 1) / wpc, p.nB, p.B * p.Hkv);
    backward_dkdv_tc_kernel<<<grid, kThreads, smem, st>>>(tq, tdo, tk, tv, bits, rowstat, dk,
                                                          dv, p, words, wpc, status);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace msa
