// Index branch of MSA on the tcgen05 tensor cores (bf16 inputs, fp32 accumulation).
//
// The index branch is a lightweight causal full attention of one index query head per KV
// head against one shared index key head ("Sparse Attention Cannot Be Directly Ported
// Across Architectures", paragraph introducing MSA), reduced to block scores for
// block-level retrieval (aietalks.com, "Block-level retrieval makes sparse attention
// easier to run on GPUs").  For one query tile (64 tokens x 4 index heads = 256 rows) the
// logits against one key block (128 keys) are a dense [256 x 128] = [256 x 128] x [128 x 128]^T
// contraction, so it runs as two M=128, N=128 UMMAs per 16-wide K step into TMEM; the
// epilogue reads the accumulator back, applies the causal mask on the diagonal block and
// max-pools each head's 64 rows x 128 columns into one score.
//
// CTA = one (sequence, query tile), heaviest tiles launched first.  Warps:
//   0-7  epilogue (warp w reads TMEM lanes 32*(w%4)..+31 of accumulator half w/4),
//   8    TMA producer (query tile once, then key blocks through a 4-stage ring),
//   9, 10 MMA issuers (one thread each: rows 0-127 and rows 128-255 of the tile), into
//        double-buffered accumulators (2 x 256 TMEM columns).  One thread's stream of
//        N = 128 MMAs with commits in it keeps the tensor core busy only ~60 % of the time;
//        two interleaved streams fill it.
// Shared memory operands use the 128-byte swizzle written by TMA; every wait is bounded.
#include "common.cuh"
#include "index_tc.cuh"
#include "ptx.cuh"
#include "tma_host.cuh"

namespace msa {

namespace {

constexpr int kQt = 64;            // queries per tile
constexpr int kNI = 4;             // index heads
constexpr int kRows = kQt * kNI;   // 256 accumulator rows per tile
constexpr int kBk = 128;           // keys per block
constexpr int kDI = 128;           // index dim: 2 swizzle chunks of 64
constexpr int kStages = 4;
constexpr int kRowBytes = 128;     // one swizzled row: 64 bf16
constexpr int kABytes = 2 * kRows * kRowBytes;   // [chunk][256 rows][128 B] = 64 KiB
constexpr int kBBytes = 2 * kBk * kRowBytes;     // [chunk][128 rows][128 B] = 32 KiB
constexpr int kEpiWarps = 8;
constexpr int kThreads = (kEpiWarps + 3) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, kBk);
constexpr int kMaxWant = 255;      // fused top-k: up to 255 blocks besides the current one

struct __align__(1024) Smem {
  uint8_t a[kABytes];
  uint8_t b[kStages][kBBytes];
  uint64_t full[kStages], empty[kStages];
  uint64_t a_full, acc_full[2], acc_empty[2], drain[2];
  uint64_t pair_bar[kEpiWarps / 2][2];
  float part[2][kEpiWarps];
  // fused top-k: per head, the best blocks seen so far (unordered) and how many
  float tk_s[kNI][kMaxWant];
  int tk_i[kNI][kMaxWant];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void raise_abort(Smem& s, int* status, int code) {
  s.abort = 1;
  if (status) atomicExch(status, code);
}

__global__ void __launch_bounds__(kThreads, 1)
index_scores_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k, float* __restrict__ scores,
                       int32_t* __restrict__ sel, Dims p, int* status) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = p.nR - 1 - blockIdx.x;            // heaviest (longest causal range) first
  const int b = blockIdx.y;
  const int cb = row_last_pos(p, m) / kBk;        // current block
  const int nblk = cb + 1;
  const volatile int* abort = &s.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(&s.full[i], 1);
      ptx::mbar_init(&s.empty[i], 2);          // both issuers' MMAs read the stage
    }
    ptx::mbar_init(&s.a_full, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s.acc_full[i], 2);       // both halves of the accumulator
      ptx::mbar_init(&s.drain[i], 1);
      ptx::mbar_init(&s.acc_empty[i], kEpiWarps);
    }
    for (int i = 0; i < kEpiWarps / 2; ++i) {
      ptx::mbar_init(&s.pair_bar[i][0], 2);
      ptx::mbar_init(&s.pair_bar[i][1], 2);
    }
    s.abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&s.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  // scores layout [B, NI, nR, nB]; blocks after the current one see no key
  float* srow = scores ? scores + ((size_t)b * kNI * p.nR + m) * p.nB : nullptr;
  const size_t head_stride = (size_t)p.nR * p.nB;
  const int n_after = p.nB - nblk;
  if (scores)
    for (int i = threadIdx.x; i < kNI * n_after; i += kThreads)
      srow[(size_t)(i / n_after) * head_stride + nblk + i % n_after] = -INFINITY;
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = s.tmem_base;

  if (warp == kEpiWarps) {
    // ------------------------------------------------------------- TMA producer
    int issued = 0;
    bool ok = true;
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_q);
      ptx::tma_prefetch_desc(&tm_k);
      ptx::mbar_arrive_expect_tx(&s.a_full, kABytes);
      // A rows ordered [head][token]: head g's 64 tokens at rows 64g..64g+63 of each chunk
      for (int g = 0; g < kNI; ++g)
        for (int kc = 0; kc < 2; ++kc)
          ptx::tma_load_4d(s.a + kc * kRows * kRowBytes + g * kQt * kRowBytes, &tm_q, &s.a_full,
                           kc * 64, g, m * kQt, b);
    }
    for (int i = 0; i < nblk; ++i) {
      const int st = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      if (!ptx::mbar_wait(&s.empty[st], ph ^ 1, abort)) { ok = false; break; }
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&s.full[st], kBBytes);
        for (int kc = 0; kc < 2; ++kc)
          ptx::tma_load_3d(s.b[st] + kc * kBk * kRowBytes, &tm_k, &s.full[st], kc * 64,
                           i * kBk, b);
      }
      issued = i + 1;
      __syncwarp();
    }
    if (!ok) {
      if (lane == 0) raise_abort(s, status, 0x101);
    }
    if (*abort && lane == 0) {
      // let copies already in flight land before the CTA's shared memory goes away
      ptx::mbar_wait_timed(&s.a_full, 0);
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
        ptx::mbar_wait_timed(&s.full[i % kStages], (i / kStages) & 1);
    }
  } else if (warp == kEpiWarps + 1 || warp == kEpiWarps + 2) {
    // ------------------------------------------------ MMA issuers, one per 128 rows
    const int h = warp - (kEpiWarps + 1);
    int issued = 0;
    bool ok = ptx::mbar_wait(&s.a_full, 0, abort);
    for (int i = 0; ok && i < nblk; ++i) {
      const int st = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      const int buf = i & 1;
      const uint32_t bph = (i >> 1) & 1;
      if (!ptx::mbar_wait(&s.full[st], ph, abort) ||
          !ptx::mbar_wait(&s.acc_empty[buf], bph ^ 1, abort)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after_sync();
      if (lane == 0) {
        const uint32_t a0 = ptx::smem_u32(s.a), b0 = ptx::smem_u32(s.b[st]);
#pragma unroll
        for (int kk = 0; kk < kDI / 16; ++kk) {
          const uint32_t ka = (kk >> 2) * (kRows * kRowBytes) + (kk & 3) * 32;
          const uint32_t kb = (kk >> 2) * (kBk * kRowBytes) + (kk & 3) * 32;
          ptx::umma_bf16_ss(tmem + buf * 256 + h * 128,
                            ptx::smem_desc_k_sw128(a0 + ka + h * 128 * kRowBytes),
                            ptx::smem_desc_k_sw128(b0 + kb), kIdesc, kk > 0 ? 1u : 0u);
        }
        ptx::umma_commit(&s.empty[st]);      // stage reusable once both halves' MMAs finish
        ptx::umma_commit(&s.acc_full[buf]);  // accumulator ready once both halves are done
      }
      issued = i + 1;
      __syncwarp();
    }
    if (!ok) {
      if (lane == 0) raise_abort(s, status, 0x102);
    }
    if (*abort && lane == 0 && issued > 0) {
      // the tensor core must be done with TMEM and shared memory before teardown: one more
      // commit covers every MMA this thread issued
      ptx::umma_commit(&s.drain[h]);
      ptx::mbar_wait_timed(&s.drain[h], 0);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int h = warp >> 2, quad = warp & 3;
    const int head = 2 * h + (quad >> 1);
    const int t = m * kQt + (quad & 1) * 32 + lane;      // this thread's query token
    const bool valid = t < p.Sq;
    const int pair = warp >> 1;
    bool ok = true;
    // fused top-k state of this head (used by the even warp of the pair, all lanes)
    const int want = sel ? min(p.k - 1, cb) : 0;   // blocks kept besides the current one
    int n_kept = 0, worst_pos = 0;
    float worst_s = INFINITY;
    bool search = false;
    for (int i = 0; i < nblk; ++i) {
      const int buf = i & 1;
      const uint32_t bph = (i >> 1) & 1;
      if (!ptx::mbar_wait(&s.acc_full[buf], bph, abort)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      uint32_t r[4][32];
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + buf * 256 + h * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld_x32(taddr + c * 32, r[c]);
      ptx::tmem_ld_wait();
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&s.acc_empty[buf]);
      float mx = -INFINITY;
      if (valid) {
        if (i < cb) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(r[c][j]));
        } else {                                         // diagonal block: keys j <= t
          const int lim = t - i * kBk;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c * 32 + j <= lim) mx = fmaxf(mx, __uint_as_float(r[c][j]));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      // the two warps holding this head's 64 rows meet through an mbarrier
      if (lane == 0) {
        s.part[i & 1][warp] = mx;
        ptx::mbar_arrive(&s.pair_bar[pair][i & 1]);
      }
      if (!ptx::mbar_wait(&s.pair_bar[pair][i & 1], (i >> 1) & 1, abort)) { ok = false; break; }
      if ((warp & 1) == 0) {
        const float v = fmaxf(s.part[i & 1][warp], s.part[i & 1][warp + 1]);
        const float score = v == -INFINITY ? -INFINITY : v * p.index_scale;
        if (srow && lane == 0) srow[(size_t)head * head_stride + i] = score;
        if (i < cb && want > 0) {
          // blocks arrive in index order, so a newcomer displaces the worst kept block only
          // when its score is strictly higher (on a tie the lower index stays)
          if (n_kept < want) {
            if (lane == 0) {
              s.tk_s[head][n_kept] = score;
              s.tk_i[head][n_kept] = i;
            }
            ++n_kept;
            search = n_kept == want;
          } else if (score > worst_s) {
            if (lane == 0) {
              s.tk_s[head][worst_pos] = score;
              s.tk_i[head][worst_pos] = i;
            }
            search = true;
          }
          if (search) {
            search = false;
            __syncwarp();
            // the worst kept block: lowest score, and of equal scores the highest index
            float ws = INFINITY;
            int wi = -1, wp = 0;
            for (int e = lane; e < want; e += 32) {
              const float cs = s.tk_s[head][e];
              const int ci = s.tk_i[head][e];
              if (cs < ws || (cs == ws && ci > wi)) { ws = cs; wi = ci; wp = e; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              const float os = __shfl_xor_sync(0xffffffffu, ws, o);
              const int oi = __shfl_xor_sync(0xffffffffu, wi, o);
              const int op = __shfl_xor_sync(0xffffffffu, wp, o);
              if (os < ws || (os == ws && oi > wi)) { ws = os; wi = oi; wp = op; }
            }
            worst_s = ws;
            worst_pos = wp;
          }
          __syncwarp();
        }
      }
    }
    if (ok && sel && (warp & 1) == 0) {
      // kept blocks in ascending index order, then the current block, then -1 padding
      int32_t* out = sel + (((size_t)b * kNI + head) * p.nR + m) * p.k;
      for (int e = lane; e < n_kept; e += 32) {
        const int ci = s.tk_i[head][e];
        int rank = 0;
        for (int f = 0; f < n_kept; ++f) rank += s.tk_i[head][f] < ci;
        out[rank] = ci;
      }
      for (int e = n_kept + lane; e < p.k; e += 32) out[e] = e == n_kept ? cb : -1;
    }
    if (!ok && lane == 0) raise_abort(s, status, 0x103);
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool index_topk_fused_supported(const Dims& p) { return index_tc_supported(p) && p.k <= kMaxWant + 1; }

bool index_tc_supported(const Dims& p) {
  return p.dtype == 1 && !p.decode && p.dI == kDI && p.Bk == kBk && p.Qt == kQt &&
         p.Hkv == kNI;
}

cudaError_t launch_index_scores_tc(const Dims& p, const void* idx_q, const void* idx_k,
                                   float* scores, int32_t* sel, cudaStream_t st, int* status) {
  CUtensorMap tq, tk;
  // idx_q [B, T, NI, dI] as (dI, NI, T, B); one box = 64 dims x 1 head x 64 tokens
  const uint64_t qd[4] = {(uint64_t)kDI, (uint64_t)kNI, (uint64_t)p.Sq, (uint64_t)p.B};
  const uint64_t qs[3] = {(uint64_t)kDI * 2, (uint64_t)kNI * kDI * 2,
                          (uint64_t)p.Sq * kNI * kDI * 2};
  const uint32_t qb[4] = {64, 1, (uint32_t)kQt, 1};
  // idx_k [B, T, dI] as (dI, T, B); one box = 64 dims x 128 keys
  const uint64_t kd[3] = {(uint64_t)kDI, (uint64_t)p.Sk, (uint64_t)p.B};
  const uint64_t ks[2] = {(uint64_t)kDI * 2, (uint64_t)p.Sk * kDI * 2};
  const uint32_t kbx[3] = {64, (uint32_t)kBk, 1};
  cudaError_t e = make_tensor_map_bf16(&tq, idx_q, 4, qd, qs, qb);
  if (e != cudaSuccess) return e;
  e = make_tensor_map_bf16(&tk, idx_k, 3, kd, ks, kbx);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(Smem) + 1024;
  e = cudaFuncSetAttribute(index_scores_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.nR, p.B);
  index_scores_tc_kernel<<<grid, kThreads, smem, st>>>(tq, tk, scores, sel, p, status);
  return cudaGetLastError();
}

}  // namespace msa
