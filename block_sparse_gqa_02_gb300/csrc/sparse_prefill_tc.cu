// Main branch of MSA, prefill, on the tcgen05 tensor cores (bf16 inputs, fp32 softmax and
// accumulation): exact attention of every query head over the blocks its KV head selected
// ("How MiniMax M3 was built", aietalks.com, section "MSA uses a lightweight index branch
// before sparse attention"; MiniMax稀疏注意力 topic page, summary: exact attention on the
// selected blocks only).  The G query heads of a KV group share its selection, so one CTA
// stacks (token, head) rows of one 64-query tile and streams only the selected 128-key
// blocks of that KV head -- each block a contiguous 32 KiB run of the head-major K/V layout
// (the pages' point about contiguous per-head reads for GQA).
//
// CTA = 256 rows of one (sequence, KV head, 64-query tile): two 128-row Q tiles that
// ping-pong on the tensor core (while one tile's softmax runs, the other tile's MMAs do).
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512); P (bf16) is
// written over the first 64 columns of S and read by the P.V MMA straight from TMEM.
// Warps: 0-3 softmax + epilogue of Q tile 0, 4-7 of Q tile 1, 8 TMA producer, 9 issues every
// Q.K^T and 10 every P.V.  One thread's stream of N = 128 MMAs with commits in it keeps the
// tensor core busy only ~60 % of the time; two streams that meet only through the barriers
// (a tile's Q.K^T after its previous P.V, its P.V after its softmax) fill the gaps, and
// neither issuer ever waits for its own MMAs.
// Online softmax in the log2 domain with conditional rescaling: the running max used for
// the exponent only moves when a block would push the row's P past a bound (its sum past
// 2^9 in a later block; its maximum past 2^8 in a row's first or diagonal block), so the O
// accumulator is rarely rescaled.  Every wait is bounded.
#include "common.cuh"
#include "ptx.cuh"
#include "sparse_prefill_tc.cuh"
#include "tma_host.cuh"

namespace msa {

namespace {

constexpr int kD = 128;
constexpr int kBk = 128;
constexpr int kQt = 64;
constexpr int kTileRows = 128;
constexpr int kRowBytes = 128;
constexpr int kTileBytes = 2 * kTileRows * kRowBytes;   // [2 chunks][128 rows][128 B] = 32 KiB
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kMaxSel = 256;
constexpr int kThreads = 352;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;      // issues the Q.K^T MMAs; warp 10 issues the P.V MMAs
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(128, kBk, 0, 0);
constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, kD, 0, 1);
constexpr float kRescaleThreshold = 8.0f;   // log2 units, on a block's maximum
constexpr float kSumThreshold = 512.0f;     // on a block's P sum (bounds every P by 2^9)
constexpr float kLn2 = 0.6931471805599453f;

struct __align__(1024) Smem {
  uint8_t q[2][kTileBytes];
  uint8_t k[kKStages][kTileBytes];
  uint8_t v[kVStages][kTileBytes];
  uint64_t q_full;
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], p_full[2], pv_done[2], o_full[2], drain[2];
  int blocks[kMaxSel];
  int n_sel;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Packed pairs of fp32 (one 64-bit register) for the paired FMA / ADD instructions.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float lo_f32(uint64_t x) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
  return lo;
}
__device__ __forceinline__ float hi_f32(uint64_t x) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
  return hi;
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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void raise_abort(Smem& s, int* status, int code) {
  s.abort = 1;
  if (status) atomicExch(status, code);
}

// 11 warps; a thread fits in 168 registers without spilling.
__global__ void __launch_bounds__(kThreads, 1)
sparse_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const int32_t* __restrict__ sel, __nv_bfloat16* __restrict__ out,
                         float* __restrict__ lse, Dims p, int* status) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int part = blockIdx.x;                   // which 256 rows of the tile's 64*G rows
  const int m = p.nR - 1 - blockIdx.y;           // heaviest tiles first
  const int bg = blockIdx.z, b = bg / p.Hkv, g = bg % p.Hkv;
  const int G = p.G;
  const int tok_per_tile = kTileRows / G;        // tokens in one 128-row Q tile
  const volatile int* abort = &s.abort;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&s.q_full, 1);
    for (int i = 0; i < kKStages; ++i) {
      ptx::mbar_init(&s.k_full[i], 1);
      ptx::mbar_init(&s.k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      ptx::mbar_init(&s.v_full[i], 1);
      ptx::mbar_init(&s.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s.s_full[i], 1);
      ptx::mbar_init(&s.p_full[i], 4);
      ptx::mbar_init(&s.pv_done[i], 1);
      ptx::mbar_init(&s.o_full[i], 1);
      ptx::mbar_init(&s.drain[i], 1);
    }
    s.abort = 0;
    ptx::fence_barrier_init();
    // the CTA's two Q tiles depend on nothing else: their copy starts before the
    // selection is read (test hook: no copies at all)
    if (p.inject != 1) {
      ptx::tma_prefetch_desc(&tm_q);
      ptx::mbar_arrive_expect_tx(&s.q_full, 2 * kTileBytes);
      for (int i = 0; i < 2; ++i) {
        const int t0 = m * kQt + (part * 2 + i) * tok_per_tile;
        debug_check(t0 >= 0 && t0 < p.nR * kQt && bg < p.B * p.Hkv, status, kDbgCoord);
        for (int kc = 0; kc < 2; ++kc)
          ptx::tma_load_4d(s.q[i] + kc * kTileRows * kRowBytes, &tm_q, &s.q_full, kc * 64,
                           g * G, t0, b);
      }
    }
  }
  if (warp == 0) {
    ptx::tmem_alloc(&s.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 1) {
    // compact this row's selection (entries < 0 or >= nB are skipped), keeping its order
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

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------- TMA producer
    int k_issued = 0, v_issued = 0;
    bool ok = true;
    // test hook: issue nothing, so the consumers' bounded waits run out
    const int n_load = p.inject == 1 ? 0 : n_sel;
    if (lane == 0 && n_load > 0) {
      ptx::tma_prefetch_desc(&tm_k);
      ptx::tma_prefetch_desc(&tm_v);
    }
    for (int j = 0; j < n_load; ++j) {
      const int blk = s.blocks[j];
      const int ks = j % kKStages, vs = j % kVStages;
      if (!ptx::mbar_wait(&s.k_empty[ks], ((j / kKStages) & 1) ^ 1, abort)) { ok = false; break; }
      if (lane == 0) {
        debug_check(blk >= 0 && blk < p.nB, status, kDbgCoord);
        ptx::mbar_arrive_expect_tx(&s.k_full[ks], kTileBytes);
        ptx::tma_load_4d(s.k[ks], &tm_k, &s.k_full[ks], 0, blk * kBk, 0, bg);
      }
      k_issued = j + 1;
      if (!ptx::mbar_wait(&s.v_empty[vs], ((j / kVStages) & 1) ^ 1, abort)) { ok = false; break; }
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&s.v_full[vs], kTileBytes);
        ptx::tma_load_4d(s.v[vs], &tm_v, &s.v_full[vs], 0, blk * kBk, 0, bg);
      }
      v_issued = j + 1;
      __syncwarp();
    }
    if (!ok && lane == 0) raise_abort(s, status, 0x201);
    // the Q copy was issued before anyone knew whether a block would need it: it lands
    // before the CTA leaves (at once when the MMA warp has used it)
    if (lane == 0 && p.inject != 1) ptx::mbar_wait_timed(&s.q_full, 0);
    if (*abort && lane == 0 && n_load > 0) {
      for (int j = k_issued > kKStages ? k_issued - kKStages : 0; j < k_issued; ++j)
        ptx::mbar_wait_timed(&s.k_full[j % kKStages], (j / kKStages) & 1);
      for (int j = v_issued > kVStages ? v_issued - kVStages : 0; j < v_issued; ++j)
        ptx::mbar_wait_timed(&s.v_full[j % kVStages], (j / kVStages) & 1);
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ------------------------ MMA issuers: warp 9 every Q.K^T, warp 10 every P.V
    const bool is_qk = warp == kMmaWarp;
    bool ok = true;
    bool issued_any = false;
    if (n_sel > 0 && is_qk) {
      ok = ptx::mbar_wait(&s.q_full, 0, abort);
      for (int j = 0; ok && j < n_sel; ++j) {
        if (!ptx::mbar_wait(&s.k_full[j % kKStages], (j / kKStages) & 1, abort)) { ok = false; break; }
        for (int i = 0; i < 2; ++i) {
          // Q.K^T of block j overwrites S/P of tile i, which block j-1's P.V reads
          if (j > 0 && !ptx::mbar_wait(&s.pv_done[i], (j - 1) & 1, abort)) { ok = false; break; }
          ptx::tc_fence_after_sync();
          if (lane == 0) {
            const uint32_t qa = ptx::smem_u32(s.q[i]);
            const uint32_t kb = ptx::smem_u32(s.k[j % kKStages]);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint32_t off = (kk >> 2) * (kTileRows * kRowBytes) + (kk & 3) * 32;
              ptx::umma_bf16_ss(tmem + i * 128, ptx::smem_desc_k_sw128(qa + off),
                                ptx::smem_desc_k_sw128(kb + off), kIdescQK, kk > 0 ? 1u : 0u);
            }
            ptx::umma_commit(&s.s_full[i]);
            if (i == 1) ptx::umma_commit(&s.k_empty[j % kKStages]);
          }
          issued_any = true;
          __syncwarp();
        }
      }
    } else if (n_sel > 0) {
      for (int j = 0; ok && j < n_sel; ++j) {
        if (!ptx::mbar_wait(&s.v_full[j % kVStages], (j / kVStages) & 1, abort)) { ok = false; break; }
        for (int i = 0; i < 2; ++i) {
          if (!ptx::mbar_wait(&s.p_full[i], j & 1, abort)) { ok = false; break; }
          ptx::tc_fence_after_sync();
          if (lane == 0) {
            const uint32_t vb = ptx::smem_u32(s.v[j % kVStages]);
#pragma unroll
            for (int kk = 0; kk < kBk / 16; ++kk)
              ptx::umma_bf16_ts(tmem + 256 + i * 128, tmem + i * 128 + kk * 8,
                                ptx::smem_desc_mn_sw128(vb + kk * 16 * kRowBytes, kBk * kRowBytes, 1024),
                                kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
            ptx::umma_commit(&s.pv_done[i]);
            if (i == 1) ptx::umma_commit(&s.v_empty[j % kVStages]);
            if (j + 1 == n_sel) ptx::umma_commit(&s.o_full[i]);
          }
          issued_any = true;
          __syncwarp();
        }
      }
    }
    if (!ok && lane == 0) raise_abort(s, status, 0x202);
    if (*abort && lane == 0 && issued_any) {
      // drain: one more commit covers every MMA this thread issued
      ptx::umma_commit(&s.drain[is_qk ? 0 : 1]);
      ptx::mbar_wait_timed(&s.drain[is_qk ? 0 : 1], 0);
    }
  } else {
    // ------------------------------------------------ softmax + epilogue (warps 0-7)
    const int i = warp >> 2, quad = warp & 3;
    const int r = quad * 32 + lane;                          // row in this Q tile
    const int R = (part * 2 + i) * kTileRows + r;            // row in the 64*G tile rows
    const int t = m * kQt + R / G;
    const int h = g * G + R % G;
    const bool valid = t < p.Sq;
    const float c1 = p.sm_scale * 1.4426950408889634f;       // to log2 units
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + i * 128;
    const uint32_t o_addr = tmem + lane_off + 256 + i * 128;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_sel; ++j) {
      const int blk = s.blocks[j];
      if (!ptx::mbar_wait(&s.s_full[i], j & 1, abort)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      uint32_t sv[4][32];
      // keys j > t are masked; only a block reaching past this row's token needs it
      const int lim = t - blk * kBk;                         // visible columns: c <= lim
      const uint64_t c1x2 = f32x2(c1, c1);
      // P = 2^(s * c1 - base) from the S values in sv, written over S as bf16; returns the
      // row sum of P.  Pairs of columns go through packed fp32 FMA / ADD, with one sum chain
      // per 32-column chunk.
      auto p_from_sv = [&](float base) {
        const uint64_t negm = f32x2(-base, -base);
        uint64_t acc[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
          acc[c] = f32x2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const uint64_t y = fma_f32x2(
                f32x2(__uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1])), c1x2, negm);
            const float p0 = ex2(lo_f32(y)), p1 = ex2(hi_f32(y));
            acc[c] = add_f32x2(acc[c], f32x2(p0, p1));
            pk[e >> 1] = pack_bf16x2(p0, p1);
          }
          ptx::tmem_st_x16(s_addr + c * 16, pk);
        }
        const uint64_t accs = add_f32x2(add_f32x2(acc[0], acc[1]), add_f32x2(acc[2], acc[3]));
        return lo_f32(accs) + hi_f32(accs);
      };
      // O *= alpha in every row of the warp (alpha = 1 in rows that keep their base).  The
      // P.V of the previous block is complete (it precedes this block's Q.K^T), and O is
      // rescaled before this block's P is released to the MMA warp.
      auto rescale_o = [&](float alpha) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t ov[32];
          ptx::tmem_ld_x32(o_addr + c * 32, ov);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          ptx::tmem_st_x32(o_addr + c * 32, ov);
        }
      };
      // tcgen05.ld/st are warp-collective, so every branch around them is warp-uniform.
      if (__all_sync(0xffffffffu, m_used != -INFINITY && lim >= kBk - 1)) {
        // A later block with no masked key: P is formed with the running base while S
        // streams in from TMEM a chunk at a time (the next chunk loads while this one is
        // exponentiated), and the block's P sum is checked afterwards (no per-column maximum
        // is taken: a sum within the bound bounds every P).  P chunk c lands on S columns
        // 16c .. 16c+15, which were loaded before.
        const uint64_t negm = f32x2(-m_used, -m_used);
        uint64_t acc[4];
        ptx::tmem_ld_x32(s_addr, sv[0]);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c < 3) ptx::tmem_ld_x32(s_addr + (c + 1) * 32, sv[c + 1]);
          uint32_t pk[16];
          acc[c] = f32x2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float x0 = __uint_as_float(sv[c][e]), x1 = __uint_as_float(sv[c][e + 1]);
            const uint64_t y = fma_f32x2(f32x2(x0, x1), c1x2, negm);
            const float p0 = ex2(lo_f32(y)), p1 = ex2(hi_f32(y));
            acc[c] = add_f32x2(acc[c], f32x2(p0, p1));
            pk[e >> 1] = pack_bf16x2(p0, p1);
          }
          ptx::tmem_st_x16(s_addr + c * 16, pk);
          if (c < 3) ptx::tmem_ld_wait();
        }
        // the block's P sum bounds every P of the row: at most 2^9 keeps them all small
        const uint64_t accs = add_f32x2(add_f32x2(acc[0], acc[1]), add_f32x2(acc[2], acc[3]));
        const float lb = lo_f32(accs) + hi_f32(accs);
        const bool redo = !(lb <= kSumThreshold);
        if (__any_sync(0xffffffffu, redo)) {
          // rare: a row's P grew past the bound; the warp redoes the block from the block
          // maximum (rows that keep their base recompute the same P)
          float alpha = 1.f;
          if (redo) {
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int e = 0; e < 32; e += 2)
                mx[c] = max3(mx[c], __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]));
            const float mb = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c1;
            alpha = ex2(m_used - mb);
            m_used = mb;
          }
          l = l * alpha + p_from_sv(m_used);
          rescale_o(alpha);
        } else {
          l += lb;
        }
      } else {
        // a row's first block, or a block with masked keys: the block maximum first
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld_x32(s_addr + c * 32, sv[c]);
        ptx::tmem_ld_wait();
        // four independent max chains (one per 32-column chunk) keep the dependency short
        float mc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (lim >= kBk - 1) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; e += 2)
              mc[c] = max3(mc[c], __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]));
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float x = c * 32 + e <= lim ? __uint_as_float(sv[c][e]) : -INFINITY;
              sv[c][e] = __float_as_uint(x);
              mc[c] = fmaxf(mc[c], x);
            }
        }
        const float mb = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3])) * c1;
        float alpha = 1.f;
        bool rescale = false;
        if (mb > m_used + kRescaleThreshold) {
          if (m_used != -INFINITY) {
            alpha = ex2(m_used - mb);
            rescale = true;
            l *= alpha;
          }
          m_used = mb;
        }
        l += p_from_sv(m_used == -INFINITY ? 0.f : m_used);
        if (__any_sync(0xffffffffu, rescale)) rescale_o(alpha);
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&s.p_full[i]);
    }
    if (!ok && lane == 0) raise_abort(s, status, 0x203);
    // epilogue: O / l -> bf16 row of out, lse
    bool have_o = ok && n_sel > 0;
    if (have_o) {
      if (!ptx::mbar_wait(&s.o_full[i], 0, abort)) {
        have_o = false;
        if (lane == 0) raise_abort(s, status, 0x204);
      }
    }
    if (have_o) ptx::tc_fence_after_sync();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16* orow = out + (((size_t)b * p.Sq + t) * p.Hq + h) * kD;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t ov[32];
      if (have_o) {
        ptx::tmem_ld_x32(o_addr + c * 32, ov);
        ptx::tmem_ld_wait();
      }
      if (valid) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          pk[e >> 1] = have_o ? pack_bf16x2(__uint_as_float(ov[e]) * inv,
                                            __uint_as_float(ov[e + 1]) * inv)
                              : 0u;
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int w = 0; w < 4; ++w)
          dst[w] = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
      }
    }
    debug_check(!valid || h < p.Hq, status, kDbgStore);
    if (valid && lse)
      lse[((size_t)b * p.Hq + h) * p.Sq + t] =
          l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool sparse_prefill_tc_supported(const Dims& p) {
  return p.dtype == 1 && !p.decode && p.d == kD && p.Bk == kBk && p.Qt == kQt &&
         p.G >= 4 && p.G <= 128 && (kTileRows % p.G) == 0 && p.k <= kMaxSel;
}

cudaError_t launch_sparse_prefill_tc(const Dims& p, const void* q, const void* k, const void* v,
                                     const int32_t* sel, void* out, float* lse, cudaStream_t st,
                                     int* status) {
  CUtensorMap tq, tk, tv;
  // q [B, T, Hq, d] as (d, Hq, T, B); one box = 64 dims x G heads x (128 / G) tokens
  const uint64_t qd[4] = {(uint64_t)kD, (uint64_t)p.Hq, (uint64_t)p.Sq, (uint64_t)p.B};
  const uint64_t qs[3] = {(uint64_t)kD * 2, (uint64_t)p.Hq * kD * 2,
                          (uint64_t)p.Sq * p.Hq * kD * 2};
  const uint32_t qb[4] = {64, (uint32_t)p.G, (uint32_t)(kTileRows / p.G), 1};
  // k, v [B, Hkv, Sk, d] as (64 dims, Sk, 2 halves of d, B * Hkv): the half-of-d axis has the
  // smallest stride (128 B) but sits outside the key axis, so one box {64, 128, 2, 1} lands a
  // whole block as [half][128 keys][128 B], the two swizzled K-major chunks the UMMAs read
  // (one copy per block instead of one per half)
  const uint64_t kd[4] = {64, (uint64_t)p.Sk, 2, (uint64_t)p.B * p.Hkv};
  const uint64_t ks[3] = {(uint64_t)kD * 2, 128, (uint64_t)p.Sk * kD * 2};
  const uint32_t kb[4] = {64, (uint32_t)kBk, 2, 1};
  cudaError_t e = make_tensor_map_bf16(&tq, q, 4, qd, qs, qb);
  if (e == cudaSuccess) e = make_tensor_map_bf16(&tk, k, 4, kd, ks, kb);
  if (e == cudaSuccess) e = make_tensor_map_bf16(&tv, v, 4, kd, ks, kb);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(Smem) + 1024;
  e = cudaFuncSetAttribute(sparse_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.Qt * p.G / (2 * kTileRows), p.nR, p.B * p.Hkv);
  sparse_prefill_tc_kernel<<<grid, kThreads, smem, st>>>(tq, tk, tv, sel, (__nv_bfloat16*)out,
                                                         lse, p, status);
  return cudaGetLastError();
}

}  // namespace msa
