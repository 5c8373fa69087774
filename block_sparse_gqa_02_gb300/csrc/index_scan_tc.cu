// Decode index scan of MSA: the new token's index queries (one per KV head) against every
// key of the index-key cache, max-pooled per 128-key block ("Sparse Attention Cannot Be
// Directly Ported Across Architectures", paragraph introducing MSA: lightweight full
// attention with four query heads and one key head; selection per token in decode).
//
// The scan is bound by HBM: every index key is read once (2 GiB for 8 sequences of 1M
// tokens) and used for 4 dot products.  Each CTA streams a contiguous range of key blocks
// of one sequence through a 6-stage TMA ring (32 KiB per block, 128-byte swizzle).  One
// thread issues the block's 4-head logits as UMMAs with the keys as the M=128 operand and
// the 4 queries, zero-padded to N=16, as the other, so the SMs only move bytes; 4 epilogue
// warps read the [128 keys x 16] accumulator from TMEM and max-pool it.
// Warps: 0-3 epilogue (TMEM lane quadrants), 4 TMA producer, 5 MMA issuer.  Every wait is
// bounded.
#include "common.cuh"
#include "index_scan_tc.cuh"
#include "ptx.cuh"
#include "tma_host.cuh"

namespace msa {

namespace {

constexpr int kNI = 4;
constexpr int kN = 16;             // UMMA N: 4 query heads padded with zero rows
constexpr int kBk = 128;
constexpr int kDI = 128;
constexpr int kStages = 6;
constexpr int kRowBytes = 128;
constexpr int kBlockBytes = 2 * kBk * kRowBytes;       // [chunk][128 keys][128 B] = 32 KiB
constexpr int kQBytes = 2 * kN * kRowBytes;            // [chunk][16 rows][128 B] = 4 KiB
constexpr int kThreads = 6 * 32;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr uint32_t kTmemCols = 32;                     // 2 accumulators x 16 columns
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, kN);

struct __align__(1024) Smem {
  uint8_t a[kStages][kBlockBytes];
  uint8_t q[kQBytes];
  uint64_t full[kStages], empty[kStages];
  uint64_t acc_full[2], acc_empty[2], red[2];
  float part[2][4][kNI];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void raise_abort(Smem& s, int* status, int code) {
  s.abort = 1;
  if (status) atomicExch(status, code);
}

// Which blocks a CTA scans.  Equal lengths: gridDim.x CTAs per sequence (blockIdx.y), each a
// contiguous range of blocks_per_cta blocks.  Ragged lengths (blocks_per_cta == 0): a 1-D grid
// whose CTAs are shared out in proportion to the sequences' block counts, every sequence
// getting at least one, so that a short sequence does not leave its share of the SMs idle
// while the longest one is still being read.
struct ScanRange {
  int b;          // sequence
  int blk0;       // first block of the range
  int nblk;       // blocks of the range inside the sequence
  int rank, cnt;  // this CTA among the sequence's CTAs (they share the -inf tail)
};

__device__ ScanRange scan_range(const Dims& p, int blocks_per_cta) {
  ScanRange r;
  if (blocks_per_cta > 0) {
    r.b = blockIdx.y;
    r.blk0 = blockIdx.x * blocks_per_cta;
    const int nB_b = (seq_len_of(p, r.b) + kBk - 1) / kBk;
    r.nblk = max(0, min(nB_b, r.blk0 + blocks_per_cta) - r.blk0);
    r.rank = blockIdx.x;
    r.cnt = gridDim.x;
    return r;
  }
  const int ctas = gridDim.x, c = blockIdx.x;   // ctas >= p.B, checked by the launcher
  long long total = 0;
  for (int bb = 0; bb < p.B; ++bb) total += (seq_len_of(p, bb) + kBk - 1) / kBk;
  total = max(total, 1ll);
  long long prefix = 0;
  r.b = p.B - 1; r.blk0 = 0; r.nblk = 0; r.rank = 0; r.cnt = 1;
  for (int bb = 0; bb < p.B; ++bb) {
    const int nb = (seq_len_of(p, bb) + kBk - 1) / kBk;
    const int lo = bb + (int)((long long)(ctas - p.B) * prefix / total);
    const int hi = bb + 1 + (int)((long long)(ctas - p.B) * (prefix + nb) / total);
    if (c >= lo && c < hi) {
      const int cnt = hi - lo, per = (nb + cnt - 1) / cnt;
      r.b = bb;
      r.rank = c - lo;
      r.cnt = cnt;
      r.blk0 = r.rank * per;
      r.nblk = max(0, min(nb, r.blk0 + per) - r.blk0);
      break;
    }
    prefix += nb;
  }
  return r;
}

__global__ void __launch_bounds__(kThreads, 1)
index_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __nv_bfloat16* __restrict__ iq,
                     float* __restrict__ scores, Dims p, int blocks_per_cta, int* status) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ScanRange rg = scan_range(p, blocks_per_cta);
  const int b = rg.b, blk0 = rg.blk0, nblk = rg.nblk;
  const int L = seq_len_of(p, b);                       // this sequence's cache length
  const int nB_b = (L + kBk - 1) / kBk;
  const volatile int* abort = &s.abort;
  // blocks past the sequence's end hold no key: the sequence's CTAs share them out
  for (int e = rg.rank * kThreads + threadIdx.x; e < (p.nB - nB_b) * kNI;
       e += rg.cnt * kThreads)
    scores[((size_t)b * kNI + e % kNI) * p.nB + nB_b + e / kNI] = -INFINITY;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(&s.full[i], 1);
      ptx::mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s.acc_full[i], 1);
      ptx::mbar_init(&s.acc_empty[i], 4);
      ptx::mbar_init(&s.red[i], 4);
    }
    s.abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&s.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  // the B operand: rows 0-3 = this sequence's index queries, rows 4-15 zero, K-major with
  // the 128-byte swizzle (16-byte unit u of row n lives at unit u ^ (n % 8))
  for (int i = threadIdx.x; i < kN * kDI / 8; i += kThreads) {
    const int n = i / (kDI / 8), u16 = i % (kDI / 8);          // row, 16-byte unit (8 dims)
    const int chunk = u16 >> 3, u = u16 & 7;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (n < kNI) val = *reinterpret_cast<const uint4*>(iq + ((size_t)b * kNI + n) * kDI + u16 * 8);
    *reinterpret_cast<uint4*>(s.q + chunk * kN * kRowBytes + n * kRowBytes + ((u ^ (n & 7)) << 4)) = val;
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = s.tmem_base;

  if (warp == kProducerWarp) {
    int issued = 0;
    bool ok = true;
    if (lane == 0) ptx::tma_prefetch_desc(&tm_k);
    for (int i = 0; i < nblk; ++i) {
      const int st = i % kStages;
      if (!ptx::mbar_wait(&s.empty[st], ((i / kStages) & 1) ^ 1, abort)) { ok = false; break; }
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&s.full[st], kBlockBytes);
        // contiguous cache: (dims, key, sequence); paged pool: (dims, key in block, block)
        const int blk = blk0 + i;
        const int y = p.block_table ? 0 : blk * kBk;
        const int z = p.block_table ? p.block_table[(size_t)b * p.nB + blk] : b;
        debug_check(blk >= 0 && blk < p.nB && y >= 0 && y < p.Sk && z >= 0 &&
                        z < (p.block_table ? p.n_phys : p.B),
                    status, kDbgCoord);
        for (int kc = 0; kc < 2; ++kc)
          ptx::tma_load_3d(s.a[st] + kc * kBk * kRowBytes, &tm_k, &s.full[st], kc * 64, y, z);
      }
      issued = i + 1;
      __syncwarp();
    }
    if (!ok && lane == 0) raise_abort(s, status, 0x301);
    if (*abort && lane == 0)
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
        ptx::mbar_wait_timed(&s.full[i % kStages], (i / kStages) & 1);
  } else if (warp == kMmaWarp) {
    int issued = 0;
    bool ok = true;
    const uint32_t q0 = ptx::smem_u32(s.q);
    for (int i = 0; i < nblk; ++i) {
      const int st = i % kStages, buf = i & 1;
      if (!ptx::mbar_wait(&s.full[st], (i / kStages) & 1, abort) ||
          !ptx::mbar_wait(&s.acc_empty[buf], ((i >> 1) & 1) ^ 1, abort)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      if (lane == 0) {
        const uint32_t a0 = ptx::smem_u32(s.a[st]);
#pragma unroll
        for (int kk = 0; kk < kDI / 16; ++kk)
          ptx::umma_bf16_ss(tmem + buf * kN,
                            ptx::smem_desc_k_sw128(a0 + (kk >> 2) * (kBk * kRowBytes) + (kk & 3) * 32),
                            ptx::smem_desc_k_sw128(q0 + (kk >> 2) * (kN * kRowBytes) + (kk & 3) * 32),
                            kIdesc, kk > 0 ? 1u : 0u);
        ptx::umma_commit(&s.empty[st]);
        ptx::umma_commit(&s.acc_full[buf]);
      }
      issued = i + 1;
      __syncwarp();
    }
    if (!ok && lane == 0) raise_abort(s, status, 0x302);
    if (*abort && lane == 0 && issued > 0)
      ptx::mbar_wait_timed(&s.acc_full[(issued - 1) & 1], ((issued - 1) >> 1) & 1);
  } else {
    // epilogue warps 0-3: warp w holds keys 32w..32w+31 of each block
    bool ok = true;
    for (int i = 0; i < nblk; ++i) {
      const int buf = i & 1;
      if (!ptx::mbar_wait(&s.acc_full[buf], (i >> 1) & 1, abort)) { ok = false; break; }
      ptx::tc_fence_after_sync();
      uint32_t r[16];
      ptx::tmem_ld_x16(tmem + ((uint32_t)(warp * 32) << 16) + buf * kN, r);
      ptx::tmem_ld_wait();
      ptx::tc_fence_before_sync();
      __syncwarp();
      // warps 1-3 release the accumulator now; warp 0 only after it has combined the
      // partial maxima below, so no warp can run two blocks ahead and overwrite them
      if (warp != 0 && lane == 0) ptx::mbar_arrive(&s.acc_empty[buf]);
      const int key = (blk0 + i) * kBk + warp * 32 + lane;
      float mx[kNI];
#pragma unroll
      for (int h = 0; h < kNI; ++h) {
        mx[h] = key < L ? __uint_as_float(r[h]) : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], o));
      }
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < kNI; ++h) s.part[i & 1][warp][h] = mx[h];
        ptx::mbar_arrive(&s.red[i & 1]);
      }
      if (warp == 0) {
        if (!ptx::mbar_wait(&s.red[i & 1], (i >> 1) & 1, abort)) { ok = false; break; }
        if (lane < kNI) {
          float v = fmaxf(fmaxf(s.part[i & 1][0][lane], s.part[i & 1][1][lane]),
                          fmaxf(s.part[i & 1][2][lane], s.part[i & 1][3][lane]));
          scores[((size_t)b * kNI + lane) * p.nB + blk0 + i] = v * p.index_scale;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&s.acc_empty[buf]);
      }
    }
    if (!ok && lane == 0) raise_abort(s, status, 0x303);
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool index_scan_tc_supported(const Dims& p) {
  return p.dtype == 1 && p.decode && p.dI == kDI && p.Bk == kBk && p.Hkv == kNI;
}

cudaError_t launch_index_scan_tc(const Dims& p, const void* idx_q, const void* idx_k,
                                 float* scores, cudaStream_t st, int* status) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  CUtensorMap tk;
  // contiguous idx_k [B, L, dI] as (dI, L, B); a paged pool [P, 128, dI] as (dI, 128, P)
  const uint64_t rows = p.block_table ? (uint64_t)kBk : (uint64_t)p.Sk;
  const uint64_t outer = p.block_table ? (uint64_t)p.n_phys : (uint64_t)p.B;
  const uint64_t kd[3] = {(uint64_t)kDI, rows, outer};
  const uint64_t ks[2] = {(uint64_t)kDI * 2, rows * kDI * 2};
  const uint32_t kbx[3] = {64, (uint32_t)kBk, 1};
  e = make_tensor_map_bf16(&tk, idx_k, 3, kd, ks, kbx);
  if (e != cudaSuccess) return e;
  // one CTA per SM: split evenly over the sequences when they have one length, in
  // proportion to their lengths (read on the device) when they may differ
  const bool ragged = p.seq_lens != nullptr && p.B <= sms;
  const int ctas_per_seq = max(1, (sms + p.B - 1) / p.B);
  const int blocks_per_cta = ragged ? 0 : (p.nB + ctas_per_seq - 1) / ctas_per_seq;
  const int ctas = ragged ? sms : (p.nB + blocks_per_cta - 1) / blocks_per_cta;
  const size_t smem = sizeof(Smem) + 1024;
  e = cudaFuncSetAttribute(index_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(ctas, ragged ? 1 : p.B);
  index_scan_tc_kernel<<<grid, kThreads, smem, st>>>(tk, (const __nv_bfloat16*)idx_q, scores, p,
                                                     blocks_per_cta, status);
  return cudaGetLastError();
}

}  // namespace msa
