// Training the index branch on the tcgen05 tensor cores: the KL loss toward the main
// branch's attention and its gradients ("Sparse Attention Cannot Be Directly Ported Across
// Architectures", paragraph introducing MSA; aietalks.com, "MSA uses a lightweight index
// branch before sparse attention": the index branch is trained with a KL loss to match the
// main branch's attention).  bf16 inputs, head_dim = index_dim = 128, 128-key blocks,
// 64-query tiles, G = 2 .. 32 query heads per KV head; fp32 accumulation and outputs.
//
// For token t and KV head g over the keys J of the tile's selected blocks (j <= t):
//   target p_T[j] = mean over the group's G heads h of 2^(c1 s_hj - lse2_h)   (held constant)
//   index  p_I[j] = 2^(c2 z_j - lseI2),  z_j = idx_q[t,g] . idx_k[j],  c2 = index_scale log2 e
//   loss += sum_j p_T (ln p_T - ln p_I);  gz_j = p_I - p_T = dloss / d(index_scale z_j)
//   d idx_q[t,g] = index_scale sum_j gz_j idx_k[j];  d idx_k[j] += index_scale gz_j idx_q[t,g].
//
// Kernels:
// * norm (G >= 8; one CTA per two consecutive 64-query tiles of a (sequence, KV head)): the
//   index log-normaliser lseI2 of every token, with the 128 tokens as the rows of
//   Z = idx_q idx_k^T over the union of the two tiles' selections; it writes each 128-row
//   group's record for the key-block pass (the main branch's lse2 per row, lseI2 per token)
//   and zeroes d idx_q.
// * rows (G < 8; query-tile order, one CTA per 128 (token, head) rows like the forward): a
//   first walk forms lseI2 from Z with each row's idx_q replicated so that every row of a
//   token holds its token's index logits, and writes the same record; a second walk forms S
//   and Z again (S into one of two TMEM buffers, so a block's S and Z are computed while the
//   math warps work on the previous block), the math warps average the G rows of a token
//   with warp shuffles, accumulate the loss and write gz into TMEM, and d idx_q += gz idx_k
//   accumulates in TMEM.
// * keys (key-block order over the tiles that selected the block, as in the dK/dV pass of
//   the backward): S^T = K Q^T and Z^T = idx_k idx_q^T with the keys on the TMEM lanes, so a
//   token's G rows are adjacent columns; gz^T goes to TMEM and d idx_k += gz^T idx_q
//   accumulates there over all of the CTA's groups before one set of vector atomics.  With
//   G >= 8 (at most 16 tokens a group) it also forms the loss terms and, per group,
//   d idx_q^T = idx_k^T gz^T (the block's idx_k tile read MN-major, gz written K-major to
//   shared memory) into 16 TMEM columns, which the math warps add into d idx_q with fp32
//   atomics two groups later.
// Warps: 16 elementwise warps (four per TMEM lane quadrant, each taking a quarter of the
// columns; 8 for G = 32, where a thread needs more registers than 608 threads leave), a TMA
// producer and two MMA issuers (a single thread's stream of N = 128 MMAs with commits in it
// keeps the tensor core busy only ~60 % of the time).  The elementwise work waits mostly on
// the latency of its own loads and exponentials, so four warps per quadrant, not two, keep
// the schedulers busy.  Every wait is bounded.
#include "common.cuh"
#include "index_kl_tc.cuh"
#include "ptx.cuh"
#include "sparse_backward_tc.cuh"
#include "tma_host.cuh"

namespace msa {

namespace {

constexpr int kD = 128;
constexpr int kBk = 128;
constexpr int kQt = 64;
constexpr int kRows = 128;
constexpr int kRowBytes = 128;
constexpr int kTileBytes = 2 * kRows * kRowBytes;           // [2 chunks][128 rows][128 B]
constexpr int kMaxSel = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescKK = ptx::idesc_bf16_f32(128, 128, 0, 0);
constexpr uint32_t kIdescMN = ptx::idesc_bf16_f32(128, 128, 0, 1);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxTilesPerCta = 2048;

// With G >= 8 a 128-row group holds at most 16 tokens, and the key-block pass also forms
// d idx_q (as d idx_q^T = idx_k^T gz^T per group, into 16 spare TMEM columns) and the loss,
// so the query-tile pass only makes the walk for the index normaliser.
template <int G>
constexpr bool kKeysDQ = G >= 8;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed pairs of fp32 (one 64-bit register) for the paired FMA / ADD instructions.
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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// D[tmem] = A[smem, K-major, 128 rows] B[smem, K-major]^T over 128 (8 steps of 16); the B
// tile's two 64-element chunks lie b_chunk bytes apart.
__device__ __forceinline__ void mma_kk(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem,
                                       uint32_t b_chunk, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t in = (kk & 3) * 32;
    ptx::umma_bf16_ss(d_tmem, ptx::smem_desc_k_sw128(a_smem + (kk >> 2) * (kRows * kRowBytes) + in),
                      ptx::smem_desc_k_sw128(b_smem + (kk >> 2) * b_chunk + in), idesc,
                      kk > 0 ? 1u : 0u);
  }
}

__device__ __forceinline__ void raise_abort(int* abort_flag, int* status, int code) {
  *abort_flag = 1;
  if (status) atomicExch(status, code);
}

// ===================================================================== rows kernel

struct __align__(1024) SmemR {
  uint8_t q[kTileBytes];        // Q rows of the group
  uint8_t iqr[kTileBytes];      // row R: idx_q of R's token (K-major, 128-byte swizzle)
  uint8_t k[2][kTileBytes];
  uint8_t ik[2][kTileBytes];
  uint64_t q_full, ring_full[2], ring_empty[2];
  uint64_t z_full[2], z_free[2], pass1_done;
  uint64_t s_full[2], g_full[2], dq_done[2], z_free2, drain[2];
  float part_ml[4][2][kRows];   // pass 1: [column part][max, sum][row]
  int blocks[kMaxSel];
  int n_sel;
  uint32_t tmem_base;
  int abort;
};

// Warps of the query-tile pass: 4 math warps per TMEM lane quadrant (each a quarter of the
// key columns) when a thread of 608 has the registers (G <= 16), else 2.
template <int G>
struct RowsWarps {
  static constexpr int kPerQuad = G <= 16 ? 4 : 2;
  static constexpr int kMath = 4 * kPerQuad;
  static constexpr int kProducer = kMath, kMma = kMath + 1;
  static constexpr int kThreads = (kMath + 3) * 32;
};

template <int G>
__global__ void __launch_bounds__(RowsWarps<G>::kThreads, 1)
kl_rows_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_ik,
                  const __nv_bfloat16* __restrict__ idx_q, const int32_t* __restrict__ sel,
                  const float* __restrict__ lse, float* __restrict__ rowstat, float* __restrict__ loss,
                  float* __restrict__ d_idx_q, Dims p, int* status) {
  extern __shared__ uint8_t smem_raw[];
  SmemR& s = *reinterpret_cast<SmemR*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  constexpr int kTokPerGroup = kRows / G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int part = blockIdx.x;
  const int m = p.nR - 1 - blockIdx.y;
  const int bg = blockIdx.z, b = bg / p.Hkv, g = bg % p.Hkv;
  const int t0 = m * kQt + part * kTokPerGroup;
  const volatile int* abort = &s.abort;
  using W = RowsWarps<G>;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&s.q_full, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s.ring_full[i], 1);
      ptx::mbar_init(&s.ring_empty[i], 1);
      ptx::mbar_init(&s.z_full[i], 1);
      ptx::mbar_init(&s.z_free[i], W::kMath);
    }
    ptx::mbar_init(&s.pass1_done, W::kMath);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s.s_full[i], 1);
      ptx::mbar_init(&s.g_full[i], W::kMath);
      ptx::mbar_init(&s.dq_done[i], 1);
    }
    ptx::mbar_init(&s.z_free2, W::kMath);
    ptx::mbar_init(&s.drain[0], 1);
    ptx::mbar_init(&s.drain[1], 1);
    s.abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&s.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 1) {
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
  if (warp < 4) {
    // row r's copy of its token's index query, written in the 128-byte-swizzled K-major
    // layout the tensor core reads (16-byte unit u of row r at unit u ^ (r % 8))
    const int r = warp * 32 + lane;
    const int t = t0 + r / G;
    const uint4* src = reinterpret_cast<const uint4*>(idx_q + (((size_t)b * p.Sq + (t < p.Sq ? t : 0)) * p.Hkv + g) * kD);
#pragma unroll
    for (int u16 = 0; u16 < 16; ++u16) {
      const uint4 v = t < p.Sq ? src[u16] : make_uint4(0, 0, 0, 0);
      const int kc = u16 >> 3, u = u16 & 7;
      *reinterpret_cast<uint4*>(s.iqr + kc * (kRows * kRowBytes) + r * kRowBytes +
                                ((u ^ (r & 7)) << 4)) = v;
    }
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = s.tmem_base;
  const int n_sel = s.n_sel;
  // TMEM: pass 1 Z in [0,128) / [128,256) alternately; pass 2 S in [0,128) / [384,512)
  // alternately by block (gz bf16 over part of it), Z [128,256), dIQ [256,384)
  constexpr uint32_t kColZ = 128, kColDQ = 256;
  auto col_s = [](int j) -> uint32_t { return (j & 1) ? 384u : 0u; };

  if (warp == W::kProducer) {
    int issued = 0;
    bool ok = true;
    // test hook: issue nothing, so the consumers' bounded waits run out
    const int n_load = p.inject == 1 ? 0 : n_sel;
    constexpr int kWalks = kKeysDQ<G> ? 1 : 2;
    if (lane == 0 && n_load > 0 && !kKeysDQ<G>) {
      ptx::mbar_arrive_expect_tx(&s.q_full, kTileBytes);
      for (int kc = 0; kc < 2; ++kc)
        ptx::tma_load_4d(s.q + kc * kRows * kRowBytes, &tm_q, &s.q_full, kc * 64, g * G, t0, b);
    }
    // the block ring: pass 1 loads idx_k blocks, pass 2 idx_k and K blocks
    for (int rr = 0; rr < kWalks * n_load; ++rr) {
      const int st = rr & 1;
      if (!ptx::mbar_wait(&s.ring_empty[st], ((rr >> 1) & 1) ^ 1, abort)) { ok = false; break; }
      if (lane == 0) {
        const bool pass2 = rr >= n_sel;
        const int blk = s.blocks[pass2 ? rr - n_sel : rr];
        ptx::mbar_arrive_expect_tx(&s.ring_full[st], pass2 ? 2 * kTileBytes : kTileBytes);
        for (int kc = 0; kc < 2; ++kc) {
          ptx::tma_load_3d(s.ik[st] + kc * kBk * kRowBytes, &tm_ik, &s.ring_full[st], kc * 64,
                           blk * kBk, b);
          if (pass2)
            ptx::tma_load_3d(s.k[st] + kc * kBk * kRowBytes, &tm_k, &s.ring_full[st], kc * 64,
                             blk * kBk, bg);
        }
      }
      issued = rr + 1;
      __syncwarp();
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x701);
    if (*abort && lane == 0 && n_load > 0) {
      if (!kKeysDQ<G>) ptx::mbar_wait_timed(&s.q_full, 0);
      for (int rr = issued > 2 ? issued - 2 : 0; rr < issued; ++rr)
        ptx::mbar_wait_timed(&s.ring_full[rr & 1], (rr >> 1) & 1);
    }
  } else if (warp == W::kMma || warp == W::kMma + 1) {
    // the first issuer: pass 1's Z and pass 2's S and Z; the second: pass 2's dIQ += gz
    // idx_k (a single thread's stream of N = 128 MMAs with commits keeps the tensor core
    // busy only ~60 % of the time).  S of block j goes over the gz of block j-2, so it waits
    // for the second issuer's product of block j-2; Z over block j-1's Z, once the math
    // warps have loaded it.
    const int who = warp - W::kMma;
    bool ok = true, issued_any = false;
    const uint32_t qa = ptx::smem_u32(s.q), za = ptx::smem_u32(s.iqr);
    if (who == 0) {
      for (int j = 0; ok && j < n_sel; ++j) {                // pass 1
        const int st = j & 1, buf = j & 1;
        if (!ptx::mbar_wait(&s.ring_full[st], (j >> 1) & 1, abort) ||
            !ptx::mbar_wait(&s.z_free[buf], ((j >> 1) & 1) ^ 1, abort)) { ok = false; break; }
        ptx::tc_fence_after_sync();
        if (lane == 0) {
          mma_kk(tmem + buf * 128, za, ptx::smem_u32(s.ik[st]), kBk * kRowBytes, kIdescKK);
          ptx::umma_commit(&s.z_full[buf]);
          ptx::umma_commit(&s.ring_empty[st]);
        }
        issued_any = true;
        __syncwarp();
      }
      if (ok && n_sel > 0 && !kKeysDQ<G>)
        ok = ptx::mbar_wait(&s.pass1_done, 0, abort) && ptx::mbar_wait(&s.q_full, 0, abort);
      for (int j = 0; ok && !kKeysDQ<G> && j < n_sel; ++j) { // pass 2: S and Z
        const int rr = n_sel + j, st = rr & 1;
        // S of block j goes where block j-2's gz was (its dIQ product has read it); Z
        // where block j-1's Z was (the math warps have loaded it)
        if (!ptx::mbar_wait(&s.ring_full[st], (rr >> 1) & 1, abort) ||
            (j > 1 && !ptx::mbar_wait(&s.dq_done[j & 1], ((j >> 1) & 1) ^ 1, abort)) ||
            (j > 0 && !ptx::mbar_wait(&s.z_free2, (j - 1) & 1, abort))) { ok = false; break; }
        ptx::tc_fence_after_sync();
        if (lane == 0) {
          mma_kk(tmem + col_s(j), qa, ptx::smem_u32(s.k[st]), kBk * kRowBytes, kIdescKK);
          mma_kk(tmem + kColZ, za, ptx::smem_u32(s.ik[st]), kBk * kRowBytes, kIdescKK);
          ptx::umma_commit(&s.s_full[j & 1]);
        }
        __syncwarp();
      }
    } else {
      for (int j = 0; ok && !kKeysDQ<G> && j < n_sel; ++j) { // pass 2: dIQ += gz idx_k
        const int rr = n_sel + j, st = rr & 1;
        if (!ptx::mbar_wait(&s.g_full[j & 1], (j >> 1) & 1, abort)) { ok = false; break; }
        ptx::tc_fence_after_sync();
        if (lane == 0) {
          // gz (rows x keys) from TMEM (keys 32c .. 32c+31 packed at columns 32c .. 32c+15),
          // idx_k as the MN-major B operand; block j's ring stage is free once this product
          // finishes (its S and Z completed before the math warps formed gz)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            ptx::umma_bf16_ts(tmem + kColDQ, tmem + col_s(j) + 32 * (kk >> 1) + (kk & 1) * 8,
                              ptx::smem_desc_mn_sw128(ptx::smem_u32(s.ik[st]) + kk * 16 * kRowBytes,
                                                      kBk * kRowBytes, 1024),
                              kIdescMN, (j > 0 || kk > 0) ? 1u : 0u);
          ptx::umma_commit(&s.dq_done[j & 1]);
          ptx::umma_commit(&s.ring_empty[st]);
        }
        issued_any = true;
        __syncwarp();
      }
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x702);
    if (*abort && lane == 0 && issued_any) {
      ptx::umma_commit(&s.drain[who]);
      ptx::mbar_wait_timed(&s.drain[who], 0);
    }
  } else {
    // ------------------------- math warps: warp w takes row quadrant w % 4 and the key
    // columns (and d idx_q columns) of its part w / 4 (kCols32 chunks of 32)
    constexpr int kParts = W::kPerQuad;
    constexpr int kCols32 = 4 / kParts;
    const int quad = warp & 3, half = warp >> 2;
    const int r = quad * 32 + lane;
    const int t = t0 + r / G, hh = r % G, h = g * G + hh;
    const bool valid = t < p.Sq;
    const float c1 = p.sm_scale * kLog2e, c2 = p.index_scale * kLog2e;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    bool ok = true;
    // pass 1: log2-sum-exp of the index logits over the tile's visible keys.  The G rows
    // (lanes) of a token hold the same index logits, so lane hh takes keys hh, hh + G, ...
    // of this warp's half of the columns; the token's lanes, then the two halves, are
    // combined at the end.
    float mI = -INFINITY, lI = 0.f;
    for (int j = 0; j < n_sel; ++j) {
      const int buf = j & 1, lim = t - s.blocks[j] * kBk;
      if (!ptx::mbar_wait(&s.z_full[buf], (j >> 1) & 1, abort)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      uint32_t zv[kCols32][32];
#pragma unroll
      for (int u = 0; u < kCols32; ++u)
        ptx::tmem_ld_x32(tmem + lane_off + buf * 128 + (kCols32 * half + u) * 32, zv[u]);
      ptx::tmem_ld_wait();
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&s.z_free[buf]);
#pragma unroll
      for (int u = 0; u < kCols32; ++u) {
        const int c = kCols32 * half + u;
        float zk[32 / G];                                    // this lane's keys of the chunk
        float cm = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32 / G; ++i) {
          float z = __uint_as_float(zv[u][i * G]);
#pragma unroll
          for (int x = 1; x < G; ++x)
            if (hh == x) z = __uint_as_float(zv[u][i * G + x]);
          zk[i] = c * 32 + i * G + hh <= lim ? z * c2 : -INFINITY;
          cm = fmaxf(cm, zk[i]);
        }
        if (cm != -INFINITY) {
          const float mn = fmaxf(mI, cm);
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < 32 / G; ++i) acc += ex2(zk[i] - mn);
          lI = lI * ex2(mI - mn) + acc;
          mI = mn;
        }
      }
    }
    // combine the token's G lanes
#pragma unroll
    for (int o = 1; o < G; o <<= 1) {
      const float mo = __shfl_xor_sync(0xffffffffu, mI, o);
      const float lo = __shfl_xor_sync(0xffffffffu, lI, o);
      const float mn = fmaxf(mI, mo);
      if (mn != -INFINITY) {
        lI = lI * ex2(mI - mn) + lo * ex2(mo - mn);
        mI = mn;
      }
    }
    // every math warp reaches this barrier exactly once (also after a failed wait)
    s.part_ml[half][0][r] = mI;
    s.part_ml[half][1][r] = lI;
    asm volatile("bar.sync 1, %0;" ::"r"(W::kMath * 32) : "memory");
    // the parts, combined in part order (every part's warp gets the same result)
    mI = -INFINITY;
    lI = 0.f;
#pragma unroll
    for (int q = 0; q < kParts; ++q) {
      const float mo = s.part_ml[q][0][r], lo = s.part_ml[q][1][r];
      const float mn = fmaxf(mI, mo);
      if (mn != -INFINITY) {
        lI = lI * ex2(mI - mn) + lo * ex2(mo - mn);
        mI = mn;
      }
    }
    const float lseI2 = mI == -INFINITY ? -INFINITY : mI + __log2f(lI);
    ptx::tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&s.pass1_done);
    // pass 2: target, loss, gz.  Of every G consecutive keys, the G rows (lanes) of a token
    // each finish one: a reduce-scatter over the token's lanes leaves lane hh the token's
    // target for key hh of the G, and that lane alone forms p_I, the loss term and gz for
    // it.  Each lane writes its gz (zeros at the other keys) as its row of the d idx_q
    // operand, so the rows of a token hold partial d idx_q that are summed at the end.
    const float lse2 = valid ? lse[((size_t)b * p.Hq + h) * p.Sq + t] * kLog2e : INFINITY;
    if (half == 0) {
      // the group's record for the key-block pass: -lse2 per row, then -lseI2 per token
      // (negated, so that the key-block pass adds them in a paired FMA)
      float* rec = rowstat + (((size_t)bg * p.nR + m) * gridDim.x + part) * 2 * kRows;
      rec[r] = -lse2;
      if (hh == 0) rec[kRows + r / G] = -lseI2;
    }
    if constexpr (kKeysDQ<G>) {
      // d idx_q and the loss come from the key-block pass, which adds into d idx_q
      if (!ok && lane == 0) raise_abort(&s.abort, status, 0x703);
      if (valid && hh == 0) {
        float4* dst = reinterpret_cast<float4*>(d_idx_q + (((size_t)b * p.Sq + t) * p.Hkv + g) * kD);
#pragma unroll
        for (int u = 0; u < kCols32; ++u)
#pragma unroll
          for (int e = 0; e < 8; ++e) dst[(kCols32 * half + u) * 8 + e] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else {
    float lsum = 0.f;
    for (int j = 0; ok && j < n_sel; ++j) {
      const int lim = t - s.blocks[j] * kBk;
      if (!ptx::mbar_wait(&s.s_full[j & 1], (j >> 1) & 1, abort)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      const uint32_t cs = col_s(j);
      uint32_t sv[kCols32][32], zv[kCols32][32];
#pragma unroll
      for (int u = 0; u < kCols32; ++u) {
        ptx::tmem_ld_x32(tmem + lane_off + cs + (kCols32 * half + u) * 32, sv[u]);
        ptx::tmem_ld_x32(tmem + lane_off + kColZ + (kCols32 * half + u) * 32, zv[u]);
      }
      ptx::tmem_ld_wait();
      // Z is in registers: the next block's Z may overwrite it
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&s.z_free2);
      // The Q barrier's only phase has completed, so this wait returns at once; as a loop it
      // keeps the compiler from scheduling the exponentials below ahead of the arrive, which
      // would hold the next block's Z back for the whole elementwise step.
      if (!ptx::mbar_wait(&s.q_full, 0, abort)) { ok = false; break; }
#pragma unroll
      for (int u = 0; u < kCols32; ++u) {
        const int c = kCols32 * half + u;
        uint32_t pk[16];
#pragma unroll
        for (int e0 = 0; e0 < 32; e0 += G) {
          // this row's attention probability at keys e0 .. e0+G-1 (0 where not visible)
          float a[G];
#pragma unroll
          for (int x = 0; x < G; ++x)
            a[x] = c * 32 + e0 + x <= lim ? ex2(fmaf(__uint_as_float(sv[u][e0 + x]), c1, -lse2))
                                          : 0.f;
          // reduce-scatter over the token's G lanes: lane hh ends with key e0 + hh's sum
#pragma unroll
          for (int st = G / 2, n = G; st >= 1; st >>= 1, n >>= 1) {
            const bool up = (hh & st) != 0;
#pragma unroll
            for (int x = 0; x < n / 2; ++x) {
              const float keep = up ? a[x + n / 2] : a[x];
              const float send = up ? a[x] : a[x + n / 2];
              a[x] = keep + __shfl_xor_sync(0xffffffffu, send, st);
            }
          }
          const float pt = a[0] * (1.f / G);
          float z = __uint_as_float(zv[u][e0]);
#pragma unroll
          for (int x = 1; x < G; ++x)
            if (hh == x) z = __uint_as_float(zv[u][e0 + x]);
          const bool vis = c * 32 + e0 + hh <= lim;
          const float zl = fmaf(z, c2, -lseI2);                // log2 p_I
          const float pi = vis ? ex2(zl) : 0.f;
          if (pt > 0.f) lsum += pt * (__log2f(pt) - zl);
          const float gz = pi - pt;
#pragma unroll
          for (int x = 0; x < G; x += 2)
            pk[(e0 + x) >> 1] = pack_bf16x2(hh == x ? gz : 0.f, hh == x + 1 ? gz : 0.f);
        }
        // gz over S columns this warp loaded: chunk c at columns 32c .. 32c+15
        ptx::tmem_st_x16(tmem + lane_off + cs + 32 * c, pk);
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&s.g_full[j & 1]);
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x703);
    const bool have = ok && n_sel > 0 &&
                      ptx::mbar_wait(&s.dq_done[(n_sel - 1) & 1], ((n_sel - 1) >> 1) & 1, abort);
    if (have) ptx::tc_fence_after_sync();
    float* dst = d_idx_q + (((size_t)b * p.Sq + (valid ? t : 0)) * p.Hkv + g) * kD;
#pragma unroll 1
    for (int u = 0; u < kCols32; ++u) {
      const int c = kCols32 * half + u;
      uint32_t v[32];
      if (have) {
        ptx::tmem_ld_x32(tmem + lane_off + kColDQ + c * 32, v);
        ptx::tmem_ld_wait();
      }
      // the token's d idx_q: the sum of its G rows' partial sums
      float dv[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        float x = have ? __uint_as_float(v[e]) : 0.f;
#pragma unroll
        for (int o = 1; o < G; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        dv[e] = x * p.index_scale;
      }
      if (valid && hh == 0) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(dst + c * 32 + e) =
              make_float4(dv[e], dv[e + 1], dv[e + 2], dv[e + 3]);
      }
    }
    // the loss of this warp's keys (each (token, key) term on one lane), natural log
    float lv = lsum * kLn2;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lv += __shfl_xor_sync(0xffffffffu, lv, o);
    if (lane == 0 && lv != 0.f) atomicAdd(loss, lv);
    }
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ============================================================== normaliser kernel (G >= 8)
// The index log-normaliser lseI2 of every token over the visible keys of its tile's
// selection, with the tokens themselves as the MMA's 128 rows: a CTA takes two consecutive
// 64-query tiles of one (sequence, KV head) and walks the union of their selections; a row
// skips the blocks its own tile did not select.  Each token's index query is used once (the
// query-tile form repeats it over the G rows of its heads).  Writes each 128-row group's
// record for the key-block pass (lse2 per row, lseI2 per token) and zeroes d idx_q.

// An even number of stages: stage u % kNormStages is always read by issuer u % 2, so each
// issuer waits for a stage's phases in order (with an odd count a stage's consecutive
// phases alternate between the issuers, and a parity wait could pass a phase early).
constexpr int kNormStages = 4;
constexpr int kNormMaxU = 2 * kMaxSel;
constexpr int kNormMath = 16;                                // four per TMEM lane quadrant
constexpr int kNormProducer = kNormMath, kNormMma = kNormMath + 1;   // issuers: 17, 18
constexpr int kNormThreads = (kNormMath + 3) * 32;
constexpr uint32_t kNormTmemCols = 256;

struct __align__(1024) SmemN {
  uint8_t iq[kTileBytes];                 // idx_q of the 128 tokens (K-major, 128-byte swizzle)
  uint8_t ik[kNormStages][kTileBytes];
  uint64_t iq_full, ring_full[kNormStages], ring_empty[kNormStages];
  uint64_t z_full[2], z_free[2], drain[2];
  float part_ml[4][2][kRows];             // [column part][max, sum][token]
  int ublk[kNormMaxU];                    // the union, first tile's blocks first
  int umask[kNormMaxU];                   // bit 0: the first tile selected it, bit 1: the second
  int n_u;
  uint32_t tmem_base;
  int abort;
};

template <int G>
__global__ void __launch_bounds__(kNormThreads, 1)
kl_norm_tc_kernel(const __grid_constant__ CUtensorMap tm_ik, const __grid_constant__ CUtensorMap tm_iq,
                  const int32_t* __restrict__ sel, const float* __restrict__ lse,
                  float* __restrict__ rowstat, float* __restrict__ d_idx_q, Dims p, int* status) {
  extern __shared__ uint8_t smem_raw[];
  SmemN& s = *reinterpret_cast<SmemN*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  constexpr int kTok = kRows / G;                             // tokens of a 128-row group
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = 2 * (gridDim.x - 1 - blockIdx.x);            // later tiles first
  const int bg = blockIdx.y, b = bg / p.Hkv, g = bg % p.Hkv;
  const int parts = p.Qt * G / kRows;                         // 128-row groups per tile
  const volatile int* abort = &s.abort;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&s.iq_full, 1);
    for (int i = 0; i < kNormStages; ++i) {
      ptx::mbar_init(&s.ring_full[i], 1);
      ptx::mbar_init(&s.ring_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s.z_full[i], 1);
      ptx::mbar_init(&s.z_free[i], kNormMath);
      ptx::mbar_init(&s.drain[i], 1);
    }
    s.abort = 0;
    ptx::fence_barrier_init();
    if (p.inject != 1) {                                      // test hook: no copies at all
      ptx::tma_prefetch_desc(&tm_iq);
      ptx::mbar_arrive_expect_tx(&s.iq_full, kTileBytes);
      debug_check(m0 < p.nR && bg < p.B * p.Hkv, status, kDbgCoord);
      for (int kc = 0; kc < 2; ++kc)
        ptx::tma_load_4d(s.iq + kc * kRows * kRowBytes, &tm_iq, &s.iq_full, kc * 64, g,
                         m0 * kQt, b);
    }
  }
  if (warp == 0) {
    ptx::tmem_alloc(&s.tmem_base, kNormTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 1) {
    // the union of the two tiles' selections (entries < 0 or >= nB are skipped)
    const int32_t* row0 = sel + ((size_t)bg * p.nR + m0) * p.k;
    int n = 0;
    for (int i0 = 0; i0 < p.k; i0 += 32) {
      const int i = i0 + lane;
      const int blk = i < p.k ? row0[i] : -1;
      const bool ok = blk >= 0 && blk < p.nB;
      const unsigned mask = __ballot_sync(0xffffffffu, ok);
      if (ok) {
        const int at = n + __popc(mask & ((1u << lane) - 1));
        s.ublk[at] = blk;
        s.umask[at] = 1;
      }
      n += __popc(mask);
    }
    __syncwarp();
    const int n0 = n;
    if (m0 + 1 < p.nR) {
      const int32_t* row1 = row0 + p.k;
      for (int i0 = 0; i0 < p.k; i0 += 32) {
        const int i = i0 + lane;
        const int blk = i < p.k ? row1[i] : -1;
        bool add = blk >= 0 && blk < p.nB;
        if (add) {
          for (int j = 0; j < n0; ++j)
            if (s.ublk[j] == blk) {                           // selected by both tiles
              atomicOr(&s.umask[j], 2);
              add = false;
              break;
            }
        }
        const unsigned mask = __ballot_sync(0xffffffffu, add);
        if (add) {
          const int at = n + __popc(mask & ((1u << lane) - 1));
          s.ublk[at] = blk;
          s.umask[at] = 2;
        }
        n += __popc(mask);
      }
    }
    if (lane == 0) s.n_u = n;
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = s.tmem_base;
  const int n_u = s.n_u;

  if (warp == kNormProducer) {
    int issued = 0;
    bool ok = true;
    const int n_load = p.inject == 1 ? 0 : n_u;
    if (lane == 0 && n_load > 0) ptx::tma_prefetch_desc(&tm_ik);
    for (int u = 0; u < n_load; ++u) {
      const int st = u % kNormStages;
      if (!ptx::mbar_wait(&s.ring_empty[st], ((u / kNormStages) & 1) ^ 1, abort)) { ok = false; break; }
      if (lane == 0) {
        const int blk = s.ublk[u];
        debug_check(blk >= 0 && blk < p.nB, status, kDbgCoord);
        ptx::mbar_arrive_expect_tx(&s.ring_full[st], kTileBytes);
        for (int kc = 0; kc < 2; ++kc)
          ptx::tma_load_3d(s.ik[st] + kc * kBk * kRowBytes, &tm_ik, &s.ring_full[st], kc * 64,
                           blk * kBk, b);
      }
      issued = u + 1;
      __syncwarp();
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x721);
    if (*abort && lane == 0 && p.inject != 1) {
      if (n_u > 0) ptx::mbar_wait_timed(&s.iq_full, 0);
      for (int u = issued > kNormStages ? issued - kNormStages : 0; u < issued; ++u)
        ptx::mbar_wait_timed(&s.ring_full[u % kNormStages], (u / kNormStages) & 1);
    }
  } else if (warp == kNormMma || warp == kNormMma + 1) {
    // the two issuers take alternate blocks, each into its own Z buffer
    const int who = warp - kNormMma;
    bool ok = n_u > 0 ? ptx::mbar_wait(&s.iq_full, 0, abort) : true;
    bool issued_any = false;
    const uint32_t qa = ptx::smem_u32(s.iq);
    for (int u = who; ok && u < n_u; u += 2) {
      const int st = u % kNormStages, buf = u & 1;
      if (!ptx::mbar_wait(&s.ring_full[st], (u / kNormStages) & 1, abort) ||
          (u >= 2 && !ptx::mbar_wait(&s.z_free[buf], ((u >> 1) & 1) ^ 1, abort))) { ok = false; break; }
      ptx::tc_fence_after_sync();
      if (lane == 0) {
        mma_kk(tmem + buf * 128, qa, ptx::smem_u32(s.ik[st]), kBk * kRowBytes, kIdescKK);
        ptx::umma_commit(&s.z_full[buf]);
        ptx::umma_commit(&s.ring_empty[st]);
      }
      issued_any = true;
      __syncwarp();
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x722);
    if (*abort && lane == 0 && issued_any) {
      ptx::umma_commit(&s.drain[who]);
      ptx::mbar_wait_timed(&s.drain[who], 0);
    }
  } else {
    // ------------------ math warps: warp w takes tokens 32 (w % 4) .. +31 (a TMEM lane
    // quadrant; quadrants 0-1 are the first tile, 2-3 the second) and key columns
    // 32 (w / 4) .. +31 of every block
    const int quad = warp & 3, part_w = warp >> 2;
    const int r = quad * 32 + lane;                           // token row of the CTA
    const int t = m0 * kQt + r;
    const int tile_bit = quad < 2 ? 1 : 2;
    const float c2 = p.index_scale * kLog2e;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    float mI = -INFINITY, lI = 0.f;
    bool ok = true;
    for (int u = 0; u < n_u; ++u) {
      const int buf = u & 1;
      if (!ptx::mbar_wait(&s.z_full[buf], (u >> 1) & 1, abort)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      uint32_t zv[32];
      ptx::tmem_ld_x32(tmem + lane_off + buf * 128 + part_w * 32, zv);
      ptx::tmem_ld_wait();
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&s.z_free[buf]);
      if (s.umask[u] & tile_bit) {                            // the same in the whole warp
        const int lim = t - s.ublk[u] * kBk - part_w * 32;    // visible columns: c <= lim
        float zk[32];
        float cm = -INFINITY;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          zk[c] = c <= lim ? __uint_as_float(zv[c]) * c2 : -INFINITY;
          cm = fmaxf(cm, zk[c]);
        }
        if (cm != -INFINITY) {
          const float mn = fmaxf(mI, cm);
          float acc = 0.f;
#pragma unroll
          for (int c = 0; c < 32; ++c) acc += ex2(zk[c] - mn);
          lI = lI * ex2(mI - mn) + acc;
          mI = mn;
        }
      }
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x723);
    // every math warp reaches this barrier exactly once (also after a failed wait)
    s.part_ml[part_w][0][r] = mI;
    s.part_ml[part_w][1][r] = lI;
    asm volatile("bar.sync 1, %0;" ::"r"(kNormMath * 32) : "memory");
    mI = -INFINITY;
    lI = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float mo = s.part_ml[q][0][r], lo = s.part_ml[q][1][r];
      const float mn = fmaxf(mI, mo);
      if (mn != -INFINITY) {
        lI = lI * ex2(mI - mn) + lo * ex2(mo - mn);
        mI = mn;
      }
    }
    const float lseI2 = mI == -INFINITY ? -INFINITY : mI + __log2f(lI);
    // the token's entries of its group's record (negated, as the key-block pass reads them):
    // -lse2 of its G rows, then -lseI2
    const int mt = m0 + (r >> 6), it = r & 63;
    const bool valid = t < p.Sq;
    if (mt < p.nR) {
      const int grp = it / kTok, tok = it % kTok;
      float* rec = rowstat + (((size_t)bg * p.nR + mt) * parts + grp) * 2 * kRows;
      if (part_w == 0) rec[kRows + tok] = -lseI2;
      for (int hh = part_w; hh < G; hh += 4)
        rec[tok * G + hh] = valid ? -lse[((size_t)b * p.Hq + g * G + hh) * p.Sq + t] * kLog2e
                                  : -INFINITY;
    }
    if (valid) {
      // d idx_q is added into by the key-block pass
      float4* dst = reinterpret_cast<float4*>(d_idx_q + (((size_t)b * p.Sq + t) * p.Hkv + g) * kD);
#pragma unroll
      for (int e = 0; e < 8; ++e) dst[part_w * 8 + e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kNormTmemCols);
  }
}

// ===================================================================== keys kernel

constexpr int kIqRows = 64;                                   // idx_q rows of a group, padded
constexpr int kIqBytes = 2 * kIqRows * kRowBytes;             // [2 chunks][64 rows][128 B]

// A group's q, idx_q and record ride a three-stage ring: a stage is refilled only once the
// group's d idx_k product has read its idx_q, so with two stages the next copies waited for
// that product and the S^T / Z^T behind them, and the math warps for both.
constexpr int kGStages = 3;

struct __align__(1024) SmemK {
  uint8_t k[kTileBytes];
  uint8_t ik[kTileBytes];
  uint8_t q[kGStages][kTileBytes];
  uint8_t iq[kGStages][kIqBytes];
  uint8_t gzs[2][2 * 16 * kRowBytes];   // gz (16 tokens x 128 keys, K-major) for d idx_q^T
  float rec[kGStages][2 * kRows];   // a group's -lse2 per row [0,128), -lseI2 per token [128,..)
  uint64_t kv_full, g_full[kGStages], g_empty[kGStages];
  uint64_t s_full[2], p_full[2], acc_done[2], drain[2];   // per S^T / gz^T buffer
  uint16_t tiles[kMaxTilesPerCta];   // query tiles (< 65536) that selected the block
  int n_tiles;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(SmemK) + 1024 <= 227 * 1024, "key-block pass shared memory");


// Warps of the key-block pass: 4 math warps per TMEM lane quadrant (each a quarter of a
// group's rows) when a quarter holds whole packed gz^T columns (G <= 16), else 2.
template <int G>
struct KeysWarps {
  static constexpr int kPerQuad = G <= 16 ? 4 : 2;
  static constexpr int kMath = 4 * kPerQuad;
  static constexpr int kProducer = kMath, kMma = kMath + 1;
  static constexpr int kThreads = (kMath + 3) * 32;
};

template <int G>
__global__ void __launch_bounds__(KeysWarps<G>::kThreads, 1)
kl_keys_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_ik, const __grid_constant__ CUtensorMap tm_iq,
                  const uint32_t* __restrict__ bits, const float* __restrict__ rowstat,
                  float* __restrict__ d_idx_k, float* __restrict__ d_idx_q,
                  float* __restrict__ loss, Dims p, int words,
                  int words_per_cta, int* status) {
  extern __shared__ uint8_t smem_raw[];
  SmemK& s = *reinterpret_cast<SmemK*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  constexpr int kTok = kRows / G;                             // tokens of a 128-row group
  constexpr int kNTok = kTok < 16 ? 16 : kTok;                // UMMA N (and K of d idx_k)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x, blk = blockIdx.y, bg = blockIdx.z;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int parts = p.Qt * G / kRows;

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
      for (uint32_t x = word; x; x &= x - 1) s.tiles[pos++] = (uint16_t)(w * 32 + __ffs(x) - 1);
      n += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s.n_tiles = n;
  }
  __syncthreads();
  const int n_tiles = s.n_tiles;
  if (n_tiles == 0) return;                                   // the whole CTA leaves together
  const int n_groups = n_tiles * parts;
  const volatile int* abort = &s.abort;

  // the idx_q rows past a group's tokens stay zero (the copies write only kTok rows)
  using W = KeysWarps<G>;
  for (int i = threadIdx.x; i < kGStages * kIqBytes / 16; i += W::kThreads)
    reinterpret_cast<uint4*>(&s.iq[0][0])[i] = make_uint4(0, 0, 0, 0);
  // so do the gz rows past a group's tokens in the d idx_q^T operand
  for (int i = threadIdx.x; i < (int)sizeof(s.gzs) / 16; i += W::kThreads)
    reinterpret_cast<uint4*>(&s.gzs[0][0])[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    ptx::mbar_init(&s.kv_full, 1);
    for (int i = 0; i < kGStages; ++i) {
      ptx::mbar_init(&s.g_full[i], 1);
      ptx::mbar_init(&s.g_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s.s_full[i], 1);
      ptx::mbar_init(&s.p_full[i], W::kMath);
      ptx::mbar_init(&s.acc_done[i], 1);
      ptx::mbar_init(&s.drain[i], 1);
    }
    s.abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&s.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = s.tmem_base;
  // TMEM: S^T (keys x rows, 128 columns), Z^T (keys x tokens, kNTok), gz^T (bf16, kNTok / 2),
  // dIK [256,384) (keys x index dims).  With at most 32 tokens a group (G >= 4) the first
  // three are double-buffered -- S^T at 0 and 384, Z^T at 128 and 160, gz^T at 192 and 224 --
  // so the next group's S^T and Z^T are computed while the math warps work on this group;
  // with 64 (G = 2) they are single: S^T 0, Z^T [128,192), gz^T [192,224).
  constexpr int kNBuf = kNTok <= 32 ? 2 : 1;
  constexpr uint32_t kColDK = 256;
  // d idx_q^T of a group (index dims x its 16 token columns), per buffer (G >= 8 only)
  auto col_dq = [](int b) -> uint32_t { return b == 0 ? 208u : 240u; };
  constexpr uint32_t kIdescDQ = ptx::idesc_bf16_f32(128, 16, 1, 0);   // A (idx_k^T) MN-major
  auto col_s = [](int b) -> uint32_t { return b == 0 ? 0u : 384u; };
  auto col_z = [](int b) -> uint32_t { return b == 0 ? 128u : 160u; };
  auto col_g = [](int b) -> uint32_t { return b == 0 ? 192u : 224u; };
  constexpr uint32_t kIdescZ = ptx::idesc_bf16_f32(128, kNTok, 0, 0);

  if (warp == W::kProducer) {
    int issued = 0;
    bool ok = true;
    if (lane == 0) {
      ptx::mbar_arrive_expect_tx(&s.kv_full, 2 * kTileBytes);
      for (int kc = 0; kc < 2; ++kc) {
        ptx::tma_load_3d(s.k + kc * kBk * kRowBytes, &tm_k, &s.kv_full, kc * 64, blk * kBk, bg);
        ptx::tma_load_3d(s.ik + kc * kBk * kRowBytes, &tm_ik, &s.kv_full, kc * 64, blk * kBk, b);
      }
    }
    for (int gi = 0; gi < n_groups; ++gi) {
      const int st = gi % kGStages;
      if (!ptx::mbar_wait(&s.g_empty[st], ((gi / kGStages) & 1) ^ 1, abort)) { ok = false; break; }
      const int m = s.tiles[gi / parts], part = gi % parts;
      const int t0 = m * kQt + part * kTok;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&s.g_full[st], kTileBytes + 2 * kTok * kRowBytes + 2 * kRows * 4);
        ptx::bulk_load(s.rec[st], rowstat + (((size_t)bg * p.nR + m) * parts + part) * 2 * kRows,
                       2 * kRows * 4, &s.g_full[st]);
        for (int kc = 0; kc < 2; ++kc) {
          ptx::tma_load_4d(s.q[st] + kc * kRows * kRowBytes, &tm_q, &s.g_full[st], kc * 64,
                           g * G, t0, b);
          ptx::tma_load_4d(s.iq[st] + kc * kIqRows * kRowBytes, &tm_iq, &s.g_full[st], kc * 64,
                           g, t0, b);
        }
      }
      issued = gi + 1;
      __syncwarp();
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x711);
    if (*abort && lane == 0) {
      ptx::mbar_wait_timed(&s.kv_full, 0);
      for (int gi = issued > kGStages ? issued - kGStages : 0; gi < issued; ++gi)
        ptx::mbar_wait_timed(&s.g_full[gi % kGStages], (gi / kGStages) & 1);
    }
  } else if (warp == W::kMma || warp == W::kMma + 1) {
    // the first issuer: S^T and Z^T of each group (after the math warps released the
    // buffer's previous group); the second: dIK += gz^T idx_q
    const int who = warp - W::kMma;
    bool ok = ptx::mbar_wait(&s.kv_full, 0, abort);
    bool issued_any = false;
    const uint32_t ka = ptx::smem_u32(s.k), ia = ptx::smem_u32(s.ik);
    for (int gi = 0; ok && gi < n_groups; ++gi) {
      const int st = gi % kGStages, bf = gi % kNBuf;
      const uint32_t ph = (gi / kNBuf) & 1;
      if (who == 0) {
        // S^T and Z^T of group gi, into a buffer the math warps have finished with
        if (!ptx::mbar_wait(&s.g_full[st], (gi / kGStages) & 1, abort) ||
            (gi >= kNBuf && !ptx::mbar_wait(&s.p_full[bf], ph ^ 1, abort))) { ok = false; break; }
        ptx::tc_fence_after_sync();
        if (lane == 0) {
          mma_kk(tmem + col_s(bf), ka, ptx::smem_u32(s.q[st]), kRows * kRowBytes, kIdescKK);
          mma_kk(tmem + col_z(bf), ia, ptx::smem_u32(s.iq[st]), kIqRows * kRowBytes, kIdescZ);
          ptx::umma_commit(&s.s_full[bf]);
        }
      } else {
        if (!ptx::mbar_wait(&s.p_full[bf], ph, abort)) { ok = false; break; }
        ptx::tc_fence_after_sync();
        if (lane == 0) {
          // dIK += gz^T (keys x tokens, TMEM) idx_q (tokens x index dims, MN-major B)
#pragma unroll
          for (int kk = 0; kk < kNTok / 16; ++kk)
            ptx::umma_bf16_ts(tmem + kColDK, tmem + col_g(bf) + kk * 8,
                              ptx::smem_desc_mn_sw128(ptx::smem_u32(s.iq[st]) + kk * 16 * kRowBytes,
                                                      kIqRows * kRowBytes, 1024),
                              kIdescMN, (gi > 0 || kk > 0) ? 1u : 0u);
          if constexpr (kKeysDQ<G>) {
            // d idx_q^T = idx_k^T (index dims x keys: the block's idx_k tile read MN-major)
            // gz^T (keys x tokens: gz K-major in shared memory)
            const uint32_t gb = ptx::smem_u32(s.gzs[bf]);
#pragma unroll
            for (int kk = 0; kk < kBk / 16; ++kk)
              ptx::umma_bf16_ss(tmem + col_dq(bf),
                                ptx::smem_desc_mn_sw128(ia + kk * 16 * kRowBytes, kBk * kRowBytes, 1024),
                                ptx::smem_desc_k_sw128(gb + (kk >> 2) * (16 * kRowBytes) + (kk & 3) * 32),
                                kIdescDQ, kk > 0 ? 1u : 0u);
          }
          ptx::umma_commit(&s.acc_done[bf]);
          ptx::umma_commit(&s.g_empty[st]);
        }
      }
      issued_any = true;
      __syncwarp();
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x712);
    if (*abort && lane == 0 && issued_any) {
      ptx::umma_commit(&s.drain[who]);
      ptx::mbar_wait_timed(&s.drain[who], 0);
    }
  } else {
    // ----------------- math warps: one key of the block per lane (quadrant w % 4); warp w
    // takes the group rows kRowsW (w / 4) .. +kRowsW - 1, i.e. its tokens, and the d idx_k
    // columns kRowsW (w / 4) .. +kRowsW - 1
    constexpr int kParts = W::kPerQuad;
    constexpr int kRowsW = kRows / kParts;                    // rows of a warp
    constexpr int kTokW = kTok / kParts;                      // tokens of a warp
    constexpr int kCols32 = kRowsW / 32;                      // 32-column chunks of a warp
    const int quad = warp & 3, part_w = warp >> 2;
    const int key = blk * kBk + quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float c1 = p.sm_scale * kLog2e, c2 = p.index_scale * kLog2e;
    if (part_w == 0 && kTok < 16) {
      // gz^T columns past the group's tokens (the padding up to the UMMA's K of 16) stay zero
      uint32_t z8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) z8[e] = 0u;
      for (int bf = 0; bf < kNBuf; ++bf) ptx::tmem_st_x8(tmem + lane_off + col_g(bf), z8);
      ptx::tmem_st_wait();
    }
    bool ok = true;
    float lsum = 0.f;                                         // this lane's loss terms (log2)
    // d idx_q of group gd (its d idx_q^T MMA complete): this warp's tokens of it, this lane's
    // index dimension.  dq_load issues the TMEM load (waited for with the caller's other
    // loads), dq_add adds the values into the output.
    constexpr int kTokQ = kTokW == 2 || kTokW == 4 ? kTokW : 2;
    uint32_t dqv[kTokQ];
    auto dq_load = [&](int gd) {
      if constexpr (kKeysDQ<G>) {
        static_assert(kTokW == 2 || kTokW == 4, "d idx_q columns per warp");
        const uint32_t a = tmem + lane_off + col_dq(gd % kNBuf) + part_w * kTokW;
        if constexpr (kTokW == 4) ptx::tmem_ld_x4(a, dqv);
        else ptx::tmem_ld_x2(a, dqv);
      }
    };
    auto dq_add = [&](int gd) {
      if constexpr (kKeysDQ<G>) {
        const int md = s.tiles[gd / parts], pd = gd % parts;
        const int tw = md * kQt + pd * kTok + part_w * kTokW;   // this warp's first token
        float* dst = d_idx_q + (((size_t)b * p.Sq + tw) * p.Hkv + g) * kD + quad * 32 + lane;
#pragma unroll
        for (int x = 0; x < kTokW; ++x)
          if (tw + x < p.Sq) atomicAdd(dst + (size_t)x * p.Hkv * kD, __uint_as_float(dqv[x]) * p.index_scale);
      }
    };
    for (int gi = 0; gi < n_groups; ++gi) {
      const int st = gi % kGStages, bf = gi % kNBuf;
      const uint32_t ph = (gi / kNBuf) & 1;
      const int m = s.tiles[gi / parts], part = gi % parts;
      const int t0 = m * kQt + part * kTok;
      if (!ptx::mbar_wait(&s.g_full[st], (gi / kGStages) & 1, abort) ||
          !ptx::mbar_wait(&s.s_full[bf], ph, abort) ||
          // the d idx_k MMA of the group that last used this gz^T buffer has read it
          (gi >= kNBuf && !ptx::mbar_wait(&s.acc_done[bf], ph ^ 1, abort))) { ok = false; break; }
      ptx::tc_fence_after_sync();
      const bool have_dq = kKeysDQ<G> && gi >= kNBuf;
      if (have_dq) dq_load(gi - kNBuf);
      uint32_t sv[kCols32][32];
#pragma unroll
      for (int u = 0; u < kCols32; ++u)
        ptx::tmem_ld_x32(tmem + lane_off + col_s(bf) + (kCols32 * part_w + u) * 32, sv[u]);
      // this warp's tokens' Z^T columns (loaded 16 at a time; a 16-column load that runs past
      // the Z^T columns reads unused TMEM and those values are not used)
      constexpr int kZLoads = kTokW < 16 ? 1 : kTokW / 16;
      uint32_t zv[kZLoads][16];
#pragma unroll
      for (int c = 0; c < kZLoads; ++c)
        ptx::tmem_ld_x16(tmem + lane_off + col_z(bf) + part_w * kTokW + c * 16, zv[c]);
      ptx::tmem_ld_wait();
      if (have_dq) dq_add(gi - kNBuf);
      // the target: per token, the sum over its G rows (adjacent columns) of
      // 2^(c1 s - lse2), two rows at a time in paired fp32 (G >= 2: a pair is one token's)
      float pt[kTokW];
      {
        const uint64_t c1x2 = f32x2(c1, c1);
        uint64_t acc[kTokW];
#pragma unroll
        for (int x = 0; x < kTokW; ++x) acc[x] = f32x2(0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kCols32; ++u)
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int x = part_w * kRowsW + u * 32 + e;      // row of the group
            const int tok = (u * 32 + e) / G;                // this warp's token index
            const uint64_t nl = *reinterpret_cast<const uint64_t*>(&s.rec[st][x]);   // -lse2 pair
            const uint64_t y = fma_f32x2(f32x2(__uint_as_float(sv[u][e]), __uint_as_float(sv[u][e + 1])),
                                         c1x2, nl);
            float y0, y1;
            split_f32x2(y, y0, y1);
            if (key <= t0 + part_w * kTokW + tok) acc[tok] = add_f32x2(acc[tok], f32x2(ex2(y0), ex2(y1)));
          }
#pragma unroll
        for (int x = 0; x < kTokW; ++x) {
          float a0, a1;
          split_f32x2(acc[x], a0, a1);
          pt[x] = a0 + a1;
        }
      }
      uint32_t pk[kTokW / 2 > 0 ? kTokW / 2 : 1];
#pragma unroll
      for (int tk = 0; tk < kTokW; tk += 2) {
        float gz2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int tok = part_w * kTokW + tk + u;            // token of the group
          const bool vis = key <= t0 + tok && t0 + tok < p.Sq;
          const float zl = fmaf(__uint_as_float(zv[(tk + u) / 16][(tk + u) % 16]), c2,
                                s.rec[st][kRows + tok]);       // log2 p_I
          const float pi = vis ? ex2(zl) : 0.f;
          const float ptm = pt[tk + u] * (1.f / G);
          if constexpr (kKeysDQ<G>) {
            if (ptm > 0.f) lsum += ptm * (__log2f(ptm) - zl);
          }
          gz2[u] = pi - ptm;
        }
        pk[tk >> 1] = pack_bf16x2(gz2[0], gz2[1]);
        if constexpr (kKeysDQ<G>) {
          // gz of this key for the two tokens, into the K-major operand of d idx_q^T: row =
          // token, 16-byte unit (key % 64) / 8 swizzled with the row, chunk = key / 64
          const int kl = quad * 32 + lane;
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int n = part_w * kTokW + tk + u;
            const uint32_t off = (kl >> 6) * (16 * kRowBytes) + n * kRowBytes +
                                 ((((kl & 63) >> 3) ^ (n & 7)) << 4) + (kl & 7) * 2;
            *reinterpret_cast<__nv_bfloat16*>(&s.gzs[bf][off]) = __float2bfloat16_rn(gz2[u]);
          }
        }
      }
      // this warp's tokens' gz^T columns (2 tokens per column)
      const uint32_t gcol = tmem + lane_off + col_g(bf) + part_w * (kTokW / 2);
      if constexpr (kTokW / 2 == 1) ptx::tmem_st_x1(gcol, pk);
      else if constexpr (kTokW / 2 == 2) ptx::tmem_st_x2(gcol, pk);
      else if constexpr (kTokW / 2 == 4) ptx::tmem_st_x4(gcol, pk);
      else if constexpr (kTokW / 2 == 8) ptx::tmem_st_x8(gcol, pk);
      else ptx::tmem_st_x16(gcol, pk);
      ptx::tmem_st_wait();
      if constexpr (kKeysDQ<G>) ptx::fence_proxy_async_smem();   // gz for the tensor core
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&s.p_full[bf]);
    }
    if (!ok && lane == 0) raise_abort(&s.abort, status, 0x713);
    if constexpr (kKeysDQ<G>) {
      // the last groups' d idx_q (each buffer's last MMA, then its product)
      for (int gd = n_groups > kNBuf ? n_groups - kNBuf : 0; ok && gd < n_groups; ++gd) {
        if (!ptx::mbar_wait(&s.acc_done[gd % kNBuf], (gd / kNBuf) & 1, abort)) { ok = false; break; }
        ptx::tc_fence_after_sync();
        dq_load(gd);
        ptx::tmem_ld_wait();
        dq_add(gd);
      }
      float lv = lsum * kLn2;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lv += __shfl_xor_sync(0xffffffffu, lv, o);
      if (lane == 0 && lv != 0.f) atomicAdd(loss, lv);
    }
    // the last d idx_k MMA (one issuing thread: it follows all the others)
    const bool have = ok && ptx::mbar_wait(&s.acc_done[(n_groups - 1) % kNBuf],
                                           ((n_groups - 1) / kNBuf) & 1, abort);
    if (have) {
      ptx::tc_fence_after_sync();
      const bool in_range = key < p.Sk;
      float4* dst = reinterpret_cast<float4*>(d_idx_k + ((size_t)b * p.Sk + (in_range ? key : 0)) * kD);
#pragma unroll 1
      for (int u = 0; u < kCols32; ++u) {
        const int c = kCols32 * part_w + u;
        uint32_t a[32];
        ptx::tmem_ld_x32(tmem + lane_off + kColDK + c * 32, a);
        ptx::tmem_ld_wait();
        if (in_range) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            atomicAdd(dst + c * 8 + e / 4,
                      make_float4(__uint_as_float(a[e]) * p.index_scale,
                                  __uint_as_float(a[e + 1]) * p.index_scale,
                                  __uint_as_float(a[e + 2]) * p.index_scale,
                                  __uint_as_float(a[e + 3]) * p.index_scale));
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

template <int G>
cudaError_t launch_kl_tc(const Dims& p, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tik, const void* idx_q, const int32_t* sel,
                         const float* lse, float* loss, float* d_idx_q, float* d_idx_k,
                         float* rowstat, uint32_t* bits, cudaStream_t st, int* status) {
  CUtensorMap tiq;
  // idx_q [B, T, Hkv, dI] as (dI, Hkv, T, B); one box = 64 dims x 1 head x (128 / G) tokens
  const uint64_t qd[4] = {(uint64_t)kD, (uint64_t)p.Hkv, (uint64_t)p.Sq, (uint64_t)p.B};
  const uint64_t qs[3] = {(uint64_t)kD * 2, (uint64_t)p.Hkv * kD * 2,
                          (uint64_t)p.Sq * p.Hkv * kD * 2};
  const uint32_t qb[4] = {64, 1, (uint32_t)(kRows / G), 1};
  cudaError_t e = make_tensor_map_bf16(&tiq, idx_q, 4, qd, qs, qb);
  if (e != cudaSuccess) return e;
  if constexpr (kKeysDQ<G>) {
    // idx_q as (dI, Hkv, T, B) with one box = 64 dims x 1 head x 128 tokens (two tiles)
    CUtensorMap tiq128;
    const uint32_t qb128[4] = {64, 1, (uint32_t)kRows, 1};
    e = make_tensor_map_bf16(&tiq128, idx_q, 4, qd, qs, qb128);
    if (e != cudaSuccess) return e;
    auto kern = kl_norm_tc_kernel<G>;
    const size_t smem = sizeof(SmemN) + 1024;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.nR + 1) / 2, p.B * p.Hkv);
    kern<<<grid, kNormThreads, smem, st>>>(tik, tiq128, sel, lse, rowstat, d_idx_q, p, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  } else {
    auto kern = kl_rows_tc_kernel<G>;
    const size_t smem = sizeof(SmemR) + 1024;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.Qt * G / kRows, p.nR, p.B * p.Hkv);
    kern<<<grid, RowsWarps<G>::kThreads, smem, st>>>(tq, tk, tik, (const __nv_bfloat16*)idx_q, sel, lse,
                                       rowstat, loss, d_idx_q, p, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    auto kern = kl_keys_tc_kernel<G>;
    const size_t smem = sizeof(SmemK) + 1024;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int words = (p.nR + 31) / 32;
    const int wpc = tiles_per_cta(p) / 32;
    // a CTA lists at most wpc * 32 tiles in its shared tile list
    if (wpc * 32 > kMaxTilesPerCta) return cudaErrorInvalidValue;
    dim3 grid((words + wpc - 1) / wpc, p.nB, p.B * p.Hkv);
    kern<<<grid, KeysWarps<G>::kThreads, smem, st>>>(tq, tk, tik, tiq, bits, rowstat, d_idx_k,
                                                     d_idx_q, loss, p, words, wpc, status);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

bool index_kl_tc_supported(const Dims& p) {
  return p.dtype == 1 && !p.decode && p.d == kD && p.dI == kD && p.Bk == kBk && p.Qt == kQt &&
         (p.G == 2 || p.G == 4 || p.G == 8 || p.G == 16 || p.G == 32) && p.k <= kMaxSel &&
         p.nR <= 65536;   // tile indices held in 16 bits (the shape check allows 65535)
}

size_t index_kl_tc_workspace_bytes(const Dims& p) {
  // per 128-row group: a 1 KiB record of lse2 / lseI2, then the bitmap
  const size_t rowstat = (size_t)p.B * p.Hkv * p.nR * (p.Qt * p.G / kRows) * 2 * kRows * 4;
  const size_t words = (size_t)(p.nR + 31) / 32;
  return rowstat + (size_t)p.B * p.Hkv * p.nB * words * sizeof(uint32_t);
}

cudaError_t launch_index_kl_tc(const Dims& p, const void* q, const void* k, const float* lse,
                               const void* idx_q, const void* idx_k, const int32_t* sel,
                               float* loss, float* d_idx_q, float* d_idx_k, void* workspace,
                               cudaStream_t st, int* status) {
  const size_t rowstat_bytes = (size_t)p.B * p.Hkv * p.nR * (p.Qt * p.G / kRows) * 2 * kRows * 4;
  float* rowstat = reinterpret_cast<float*>(workspace);
  uint32_t* bits = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(workspace) + rowstat_bytes);
  cudaError_t e = cudaMemsetAsync(loss, 0, sizeof(float), st);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(d_idx_k, 0, (size_t)p.B * p.Sk * kD * sizeof(float), st);
  if (e != cudaSuccess) return e;
  if ((e = launch_selection_bitmap(p, sel, bits, st)) != cudaSuccess) return e;

  CUtensorMap tq, tk, tik;
  const uint64_t qd[4] = {(uint64_t)kD, (uint64_t)p.Hq, (uint64_t)p.Sq, (uint64_t)p.B};
  const uint64_t qs[3] = {(uint64_t)kD * 2, (uint64_t)p.Hq * kD * 2,
                          (uint64_t)p.Sq * p.Hq * kD * 2};
  const uint32_t qb[4] = {64, (uint32_t)p.G, (uint32_t)(kRows / p.G), 1};
  const uint64_t kd[3] = {(uint64_t)kD, (uint64_t)p.Sk, (uint64_t)p.B * p.Hkv};
  const uint64_t ks[2] = {(uint64_t)kD * 2, (uint64_t)p.Sk * kD * 2};
  const uint32_t kb[3] = {64, (uint32_t)kBk, 1};
  // idx_k [B, T, dI] as (dI, T, B)
  const uint64_t ikd[3] = {(uint64_t)kD, (uint64_t)p.Sk, (uint64_t)p.B};
  e = make_tensor_map_bf16(&tq, q, 4, qd, qs, qb);
  if (e == cudaSuccess) e = make_tensor_map_bf16(&tk, k, 3, kd, ks, kb);
  if (e == cudaSuccess) e = make_tensor_map_bf16(&tik, idx_k, 3, ikd, ks, kb);
  if (e != cudaSuccess) return e;
  switch (p.G) {
    case 2: return launch_kl_tc<2>(p, tq, tk, tik, idx_q, sel, lse, loss, d_idx_q, d_idx_k, rowstat, bits, st, status);
    case 4: return launch_kl_tc<4>(p, tq, tk, tik, idx_q, sel, lse, loss, d_idx_q, d_idx_k, rowstat, bits, st, status);
    case 8: return launch_kl_tc<8>(p, tq, tk, tik, idx_q, sel, lse, loss, d_idx_q, d_idx_k, rowstat, bits, st, status);
    case 16: return launch_kl_tc<16>(p, tq, tk, tik, idx_q, sel, lse, loss, d_idx_q, d_idx_k, rowstat, bits, st, status);
    default: return launch_kl_tc<32>(p, tq, tk, tik, idx_q, sel, lse, loss, d_idx_q, d_idx_k, rowstat, bits, st, status);
  }
}

}  // namespace msa
