// C-ABI entry points of the MSA library (declared in include/msa.h): argument checks,
// shape derivation, dispatch to the kernels, error reporting.  No entry point allocates.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "index_tc.cuh"
#include "msa.h"

namespace msa {

// Device status word: kernels that give up a bounded wait write a nonzero code here.
__device__ int g_device_status = 0;

namespace {

thread_local char g_last_error[512] = "";
int g_fault_mode = 0;   // msa_debug_set_fault

msa_status fail(msa_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
msa_status fail(msa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

msa_status cuda_fail(cudaError_t e, const char* where) {
  return fail(MSA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; }

int* status_ptr() {
  static thread_local int dev = -1;
  static thread_local int* ptr = nullptr;
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return nullptr;
  if (dev != cur) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    ptr = static_cast<int*>(p);
    dev = cur;
  }
  return ptr;
}

// Validates the shape and derives the kernel dimensions.
msa_status make_dims(const msa_shape* s, Dims* d) {
  if (!s) return fail(MSA_ERR_INVALID_ARG, "shape is NULL");
  if (s->batch < 1 || s->seq_q < 1 || s->seq_k < 1)
    return fail(MSA_ERR_INVALID_ARG, "batch, seq_q and seq_k must be >= 1 (got %d, %d, %d)",
                s->batch, s->seq_q, s->seq_k);
  if (s->n_heads_kv < 1 || s->n_heads_q < 1 || s->n_heads_q % s->n_heads_kv != 0)
    return fail(MSA_ERR_INVALID_ARG, "n_heads_q (%d) must be a positive multiple of n_heads_kv (%d)",
                s->n_heads_q, s->n_heads_kv);
  if (s->block_size < 1 || s->top_k < 1 || s->q_tile < 1)
    return fail(MSA_ERR_INVALID_ARG, "block_size, top_k and q_tile must be >= 1");
  if (s->dtype != MSA_F32 && s->dtype != MSA_BF16)
    return fail(MSA_ERR_INVALID_ARG, "dtype must be MSA_F32 or MSA_BF16 (got %d)", s->dtype);
  if (!(s->sm_scale >= 0.f) || !(s->index_scale >= 0.f) || isinf(s->sm_scale) ||
      isinf(s->index_scale))
    return fail(MSA_ERR_INVALID_ARG, "sm_scale and index_scale must be finite and >= 0");
  const bool decode = s->seq_q == 1 && s->q_tile == 1;
  if (!decode) {
    if (s->seq_q != s->seq_k)
      return fail(MSA_ERR_INVALID_ARG,
                  "prefill needs seq_q == seq_k (got %d, %d); decode needs seq_q == q_tile == 1",
                  s->seq_q, s->seq_k);
    if (s->block_size % s->q_tile != 0)
      return fail(MSA_ERR_INVALID_ARG, "block_size (%d) must be a multiple of q_tile (%d)",
                  s->block_size, s->q_tile);
  }
  if (s->head_dim != 64 && s->head_dim != 128)
    return fail(MSA_ERR_UNSUPPORTED, "head_dim %d: supported 64, 128", s->head_dim);
  if (s->index_dim != 64 && s->index_dim != 128)
    return fail(MSA_ERR_UNSUPPORTED, "index_dim %d: supported 64, 128", s->index_dim);
  const long long nB = ((long long)s->seq_k + s->block_size - 1) / s->block_size;
  if (nB > kMaxBlocks)
    return fail(MSA_ERR_UNSUPPORTED, "%lld blocks per sequence: at most %d", nB, kMaxBlocks);
  // query tiles and (sequence, KV head) pairs index grid dimensions of at most 65535
  const long long nR = ((long long)s->seq_q + s->q_tile - 1) / s->q_tile;
  if (nR > 65535)
    return fail(MSA_ERR_UNSUPPORTED, "%lld query tiles per sequence: at most 65535", nR);
  if ((long long)s->batch * s->n_heads_kv > 65535)
    return fail(MSA_ERR_UNSUPPORTED, "batch * n_heads_kv = %lld: at most 65535",
                (long long)s->batch * s->n_heads_kv);
  d->B = s->batch;
  d->Sq = s->seq_q;
  d->Sk = s->seq_k;
  d->Hq = s->n_heads_q;
  d->Hkv = s->n_heads_kv;
  d->G = s->n_heads_q / s->n_heads_kv;
  d->d = s->head_dim;
  d->dI = s->index_dim;
  d->Bk = s->block_size;
  d->k = s->top_k;
  d->Qt = s->q_tile;
  d->nB = (int)nB;
  d->nR = (s->seq_q + s->q_tile - 1) / s->q_tile;
  d->q_off = decode ? s->seq_k - 1 : 0;
  d->decode = decode ? 1 : 0;
  d->dtype = s->dtype;
  d->sm_scale = s->sm_scale > 0.f ? s->sm_scale : 1.f / sqrtf((float)s->head_dim);
  d->index_scale = s->index_scale > 0.f ? s->index_scale : 1.f / sqrtf((float)s->index_dim);
  d->inject = g_fault_mode;
  d->seq_lens = nullptr;
  d->block_table = nullptr;
  d->n_phys = 0;
  return MSA_OK;
}

msa_status check_ptr(const void* p, const char* name, bool nullable = false) {
  if (!p) return nullable ? MSA_OK : fail(MSA_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(MSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return MSA_OK;
}

#define MSA_TRY(expr)                    \
  do {                                   \
    msa_status st_ = (expr);             \
    if (st_ != MSA_OK) return st_;       \
  } while (0)

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" {

msa_status msa_index_scores(const msa_shape* shape, const void* idx_q, const void* idx_k,
                            float* block_scores, void* stream) {
  g_last_error[0] = 0;
  Dims d;
  MSA_TRY(make_dims(shape, &d));
  MSA_TRY(check_ptr(idx_q, "idx_q"));
  MSA_TRY(check_ptr(idx_k, "idx_k"));
  MSA_TRY(check_ptr(block_scores, "block_scores"));
  if (!d.decode && d.Hkv * d.Qt > 256 && d.dtype == MSA_F32)
    return fail(MSA_ERR_UNSUPPORTED, "fp32 index scores need n_heads_kv * q_tile <= 256");
  if (d.decode && d.Hkv != 1 && d.Hkv != 2 && d.Hkv != 4 && d.Hkv != 8)
    return fail(MSA_ERR_UNSUPPORTED, "decode index scan needs n_heads_kv in {1, 2, 4, 8}");
  if (!d.decode && d.dtype == MSA_BF16 && d.Hkv * d.Qt > 256)
    return fail(MSA_ERR_UNSUPPORTED, "index scores need n_heads_kv * q_tile <= 256");
  if (!d.decode && (size_t)d.Bk * d.dI * sizeof(float) > 200 * 1024)
    return fail(MSA_ERR_UNSUPPORTED, "index scores stage one key block (%d x %d fp32) in "
                "shared memory: at most 200 KiB", d.Bk, d.dI);
  cudaError_t e = launch_index_scores(d, idx_q, idx_k, block_scores, (cudaStream_t)stream,
                                      status_ptr());
  return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_index_scores launch");
}

msa_status msa_block_topk_shared(const msa_shape* shape, const float* block_scores,
                                 int32_t* sel, void* stream) {
  g_last_error[0] = 0;
  Dims d;
  MSA_TRY(make_dims(shape, &d));
  MSA_TRY(check_ptr(block_scores, "block_scores"));
  MSA_TRY(check_ptr(sel, "sel"));
  cudaError_t e = launch_block_topk(d, block_scores, sel, (cudaStream_t)stream, 1);
  return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_block_topk_shared launch");
}

msa_status msa_index_topk_fused(const msa_shape* shape, const void* idx_q, const void* idx_k,
                                float* block_scores, int32_t* sel, void* stream) {
  g_last_error[0] = 0;
  Dims d;
  MSA_TRY(make_dims(shape, &d));
  MSA_TRY(check_ptr(idx_q, "idx_q"));
  MSA_TRY(check_ptr(idx_k, "idx_k"));
  MSA_TRY(check_ptr(block_scores, "block_scores", true));
  MSA_TRY(check_ptr(sel, "sel"));
  if (!index_topk_fused_supported(d))
    return fail(MSA_ERR_UNSUPPORTED,
                "fused index + top-k runs bf16 prefill with index_dim 128, block 128, q_tile "
                "64, 4 KV heads and top_k <= 256");
  cudaError_t e = launch_index_scores_tc(d, idx_q, idx_k, block_scores, sel,
                                         (cudaStream_t)stream, status_ptr());
  return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_index_topk_fused launch");
}

msa_status msa_block_topk(const msa_shape* shape, const float* block_scores, int32_t* sel,
                          void* stream) {
  g_last_error[0] = 0;
  Dims d;
  MSA_TRY(make_dims(shape, &d));
  MSA_TRY(check_ptr(block_scores, "block_scores"));
  MSA_TRY(check_ptr(sel, "sel"));
  cudaError_t e = launch_block_topk(d, block_scores, sel, (cudaStream_t)stream);
  return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_block_topk launch");
}

msa_status msa_sparse_prefill(const msa_shape* shape, const void* q, const void* k,
                              const void* v, const int32_t* sel, void* out, float* lse,
                              void* workspace, size_t ws_bytes, void* stream) {
  g_last_error[0] = 0;
  (void)workspace;
  (void)ws_bytes;
  Dims d;
  MSA_TRY(make_dims(shape, &d));
  if (d.decode && d.Sk != 1)
    return fail(MSA_ERR_INVALID_ARG, "msa_sparse_prefill needs seq_q == seq_k; use msa_sparse_decode");
  MSA_TRY(check_ptr(q, "q"));
  MSA_TRY(check_ptr(k, "k"));
  MSA_TRY(check_ptr(v, "v"));
  MSA_TRY(check_ptr(sel, "sel"));
  MSA_TRY(check_ptr(out, "out"));
  MSA_TRY(check_ptr(lse, "lse", true));
  {
    const cudaError_t ve = launch_debug_validate(d, sel, (cudaStream_t)stream, status_ptr());
    if (ve != cudaSuccess) return cuda_fail(ve, "msa_sparse_prefill debug validation");
  }
  cudaError_t e = launch_sparse_prefill(d, q, k, v, sel, out, lse, (cudaStream_t)stream,
                                        status_ptr());
  return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_sparse_prefill launch");
}

msa_status msa_sparse_prefill_backward(const msa_shape* shape, const void* q, const void* k,
                                       const void* v, const int32_t* sel, const void* out,
                                       const float* lse, const void* dout, float* dq, float* dk,
                                       float* dv, void* workspace, size_t ws_bytes,
                                       void* stream) {
  g_last_error[0] = 0;
  Dims d;
  MSA_TRY(make_dims(shape, &d));
  if (d.decode && d.Sk != 1)
    return fail(MSA_ERR_INVALID_ARG, "msa_sparse_prefill_backward needs seq_q == seq_k");
  MSA_TRY(check_ptr(q, "q"));
  MSA_TRY(check_ptr(k, "k"));
  MSA_TRY(check_ptr(v, "v"));
  MSA_TRY(check_ptr(sel, "sel"));
  MSA_TRY(check_ptr(out, "out"));
  MSA_TRY(check_ptr(lse, "lse"));
  MSA_TRY(check_ptr(dout, "dout"));
  MSA_TRY(check_ptr(dq, "dq"));
  MSA_TRY(check_ptr(dk, "dk"));
  MSA_TRY(check_ptr(dv, "dv"));
  const size_t need = backward_workspace_bytes(d);
  if (need > 0) {
    MSA_TRY(check_ptr(workspace, "workspace"));
    if (ws_bytes < need)
      return fail(MSA_ERR_INVALID_ARG, "workspace of %zu bytes, need %zu", ws_bytes, need);
  }
  {
    const cudaError_t ve = launch_debug_validate(d, sel, (cudaStream_t)stream, status_ptr());
    if (ve != cudaSuccess) return cuda_fail(ve, "msa_sparse_prefill_backward debug validation");
  }
  cudaError_t e = launch_sparse_prefill_backward(d, q, k, v, sel, out, lse, dout, dq, dk, dv,
                                                 workspace, (cudaStream_t)stream, status_ptr());
  return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_sparse_prefill_backward launch");
}

msa_status msa_index_kl_loss(const msa_shape* shape, const void* q, const void* k,
                             const float* lse, const void* idx_q, const void* idx_k,
                             const int32_t* sel, float* loss, float* d_idx_q, float* d_idx_k,
                             void* workspace, size_t ws_bytes, void* stream) {
  g_last_error[0] = 0;
  Dims d;
  MSA_TRY(make_dims(shape, &d));
  if (d.decode && d.Sk != 1)
    return fail(MSA_ERR_INVALID_ARG, "msa_index_kl_loss needs seq_q == seq_k");
  if (d.G > 64) return fail(MSA_ERR_UNSUPPORTED, "index KL needs n_heads_q / n_heads_kv <= 64");
  MSA_TRY(check_ptr(q, "q"));
  MSA_TRY(check_ptr(k, "k"));
  MSA_TRY(check_ptr(lse, "lse"));
  MSA_TRY(check_ptr(idx_q, "idx_q"));
  MSA_TRY(check_ptr(idx_k, "idx_k"));
  MSA_TRY(check_ptr(sel, "sel"));
  MSA_TRY(check_ptr(loss, "loss"));
  MSA_TRY(check_ptr(d_idx_q, "d_idx_q"));
  MSA_TRY(check_ptr(d_idx_k, "d_idx_k"));
  const size_t need = index_kl_workspace_bytes(d);
  if (need > 0) {
    MSA_TRY(check_ptr(workspace, "workspace"));
    if (ws_bytes < need)
      return fail(MSA_ERR_INVALID_ARG, "workspace of %zu bytes, need %zu", ws_bytes, need);
  }
  {
    const cudaError_t ve = launch_debug_validate(d, sel, (cudaStream_t)stream, status_ptr());
    if (ve != cudaSuccess) return cuda_fail(ve, "msa_index_kl_loss debug validation");
  }
  cudaError_t e = launch_index_kl(d, q, k, lse, idx_q, idx_k, sel, loss, d_idx_q, d_idx_k,
                                  workspace, (cudaStream_t)stream, status_ptr());
  return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_index_kl_loss launch");
}

msa_status msa_sparse_decode(const msa_shape* shape, const void* q, const void* k_cache,
                             const void* v_cache, const int32_t* sel, void* out, float* lse,
                             void* workspace, size_t ws_bytes, void* stream) {
  g_last_error[0] = 0;
  Dims d;
  MSA_TRY(make_dims(shape, &d));
  if (!d.decode) return fail(MSA_ERR_INVALID_ARG, "msa_sparse_decode needs seq_q == q_tile == 1");
  if (d.G > 64) return fail(MSA_ERR_UNSUPPORTED, "decode needs n_heads_q / n_heads_kv <= 64");
  MSA_TRY(check_ptr(q, "q"));
  MSA_TRY(check_ptr(k_cache, "k_cache"));
  MSA_TRY(check_ptr(v_cache, "v_cache"));
  MSA_TRY(check_ptr(sel, "sel"));
  MSA_TRY(check_ptr(out, "out"));
  MSA_TRY(check_ptr(lse, "lse", true));
  MSA_TRY(check_ptr(workspace, "workspace"));
  const size_t need = decode_workspace_bytes(d);
  if (ws_bytes < need)
    return fail(MSA_ERR_INVALID_ARG, "workspace of %zu bytes is too small: need %zu", ws_bytes,
                need);
  {
    const cudaError_t ve = launch_debug_validate(d, sel, (cudaStream_t)stream, status_ptr());
    if (ve != cudaSuccess) return cuda_fail(ve, "msa_sparse_decode debug validation");
  }
  cudaError_t e = launch_sparse_decode(d, q, k_cache, v_cache, sel, out, lse,
                                       static_cast<float*>(workspace), (cudaStream_t)stream,
                                       status_ptr());
  return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_sparse_decode launch");
}

// ------------------------------------------------------------- paged / ragged decode

namespace {
msa_status make_paged_dims(const msa_shape* shape, const int32_t* seq_lens,
                           const int32_t* block_table, int32_t n_phys, Dims* d,
                           bool need_table) {
  MSA_TRY(make_dims(shape, d));
  if (!d->decode) return fail(MSA_ERR_INVALID_ARG, "paged decode needs seq_q == q_tile == 1");
  if (d->dtype != MSA_BF16 || d->d != 128 || d->dI != 128 || d->Bk != 128 || d->Hkv != 4 ||
      d->G > 16)
    return fail(MSA_ERR_UNSUPPORTED,
                "paged decode runs bf16, head_dim = index_dim = 128, block 128, 4 KV heads, "
                "at most 16 query heads per KV head");
  MSA_TRY(check_ptr(seq_lens, "seq_lens"));
  if (need_table) {
    MSA_TRY(check_ptr(block_table, "block_table"));
    if (n_phys < 1) return fail(MSA_ERR_INVALID_ARG, "n_phys must be >= 1");
  }
  d->seq_lens = seq_lens;
  d->block_table = need_table ? block_table : nullptr;
  d->n_phys = need_table ? n_phys : 0;
  return MSA_OK;
}
}  // namespace

msa_status msa_index_scores_paged(const msa_shape* shape, const int32_t* seq_lens,
                                  const int32_t* block_table, int32_t n_phys, const void* idx_q,
                                  const void* idx_k_pool, float* block_scores, void* stream) {
  g_last_error[0] = 0;
  Dims d;
  MSA_TRY(make_paged_dims(shape, seq_lens, block_table, n_phys, &d, true));
  MSA_TRY(check_ptr(idx_q, "idx_q"));
  MSA_TRY(check_ptr(idx_k_pool, "idx_k_pool"));
  MSA_TRY(check_ptr(block_scores, "block_scores"));
  {
    const cudaError_t ve = launch_debug_validate(d, nullptr, (cudaStream_t)stream, status_ptr());
    if (ve != cudaSuccess) return cuda_fail(ve, "msa_index_scores_paged debug validation");
  }
  cudaError_t e = launch_index_scores(d, idx_q, idx_k_pool, block_scores, (cudaStream_t)stream,
                                      status_ptr());
  return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_index_scores_paged launch");
}

msa_status msa_block_topk_ragged(const msa_shape* shape, const int32_t* seq_lens,
                                 const float* block_scores, int32_t* sel, void* stream) {
  g_last_error[0] = 0;
  Dims d;
  MSA_TRY(make_dims(shape, &d));
  if (!d.decode) return fail(MSA_ERR_INVALID_ARG, "ragged top-k needs seq_q == q_tile == 1");
  MSA_TRY(check_ptr(seq_lens, "seq_lens"));
  MSA_TRY(check_ptr(block_scores, "block_scores"));
  MSA_TRY(check_ptr(sel, "sel"));
  d.seq_lens = seq_lens;
  {
    const cudaError_t ve = launch_debug_validate(d, nullptr, (cudaStream_t)stream, status_ptr());
    if (ve != cudaSuccess) return cuda_fail(ve, "msa_block_topk_ragged debug validation");
  }
  cudaError_t e = launch_block_topk(d, block_scores, sel, (cudaStream_t)stream);
  return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_block_topk_ragged launch");
}

msa_status msa_sparse_decode_paged(const msa_shape* shape, const int32_t* seq_lens,
                                   const int32_t* block_table, int32_t n_phys, const void* q,
                                   const void* k_pool, const void* v_pool, const int32_t* sel,
                                   void* out, float* lse, void* workspace, size_t ws_bytes,
                                   void* stream) {
  g_last_error[0] = 0;
  Dims d;
  MSA_TRY(make_paged_dims(shape, seq_lens, block_table, n_phys, &d, true));
  MSA_TRY(check_ptr(q, "q"));
  MSA_TRY(check_ptr(k_pool, "k_pool"));
  MSA_TRY(check_ptr(v_pool, "v_pool"));
  MSA_TRY(check_ptr(sel, "sel"));
  MSA_TRY(check_ptr(out, "out"));
  MSA_TRY(check_ptr(lse, "lse", true));
  MSA_TRY(check_ptr(workspace, "workspace"));
  const size_t need = decode_workspace_bytes(d);
  if (ws_bytes < need)
    return fail(MSA_ERR_INVALID_ARG, "workspace of %zu bytes is too small: need %zu", ws_bytes,
                need);
  {
    const cudaError_t ve = launch_debug_validate(d, sel, (cudaStream_t)stream, status_ptr());
    if (ve != cudaSuccess) return cuda_fail(ve, "msa_sparse_decode_paged debug validation");
  }
  cudaError_t e = launch_sparse_decode(d, q, k_pool, v_pool, sel, out, lse,
                                       static_cast<float*>(workspace), (cudaStream_t)stream,
                                       status_ptr());
  return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_sparse_decode_paged launch");
}

size_t msa_workspace_bytes(const msa_shape* shape, int which) {
  Dims d;
  if (make_dims(shape, &d) != MSA_OK) return 0;
  if (which == 1 && d.decode) return decode_workspace_bytes(d);
  if (which == 2 && !d.decode) return backward_workspace_bytes(d);
  if (which == 3 && !d.decode) return index_kl_workspace_bytes(d);
  return 0;
}

msa_status msa_get_device_status(void* stream) {
  g_last_error[0] = 0;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "pending CUDA error");
  int code = 0;
  e = cudaMemcpyFromSymbol(&code, g_device_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "read device status");
  if (code != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
    if ((code & ~0xff) == kDebugCodeBase)
      return fail(MSA_ERR_BOUNDS, "a debug-build check found an index out of range (code %#x)",
                  code);
    return fail(MSA_ERR_TIMEOUT, "a kernel gave up a bounded wait (code %d)", code);
  }
  return MSA_OK;
}

const char* msa_status_string(msa_status status) {
  switch (status) {
    case MSA_OK: return "MSA_OK";
    case MSA_ERR_INVALID_ARG: return "MSA_ERR_INVALID_ARG: invalid argument";
    case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED: shape not supported";
    case MSA_ERR_CUDA: return "MSA_ERR_CUDA: CUDA error";
    case MSA_ERR_TIMEOUT: return "MSA_ERR_TIMEOUT: a kernel gave up a bounded wait";
    case MSA_ERR_BOUNDS: return "MSA_ERR_BOUNDS: a debug-build index check failed";
  }
  return "unknown msa_status";
}

const char* msa_last_error(void) { return g_last_error; }

msa_status msa_debug_set_fault(int32_t mode) {
  if (mode != 0 && mode != 1) return fail(MSA_ERR_INVALID_ARG, "fault mode must be 0 or 1");
  g_fault_mode = mode;
  return MSA_OK;
}

int32_t msa_abi_version(void) { return MSA_ABI_VERSION; }

int32_t msa_debug_build(void) { return kDebugChecks ? 1 : 0; }

}  // extern "C"

// -----------------------------------------------------------------------------------------
// Decode with library-held scratch, for callers that cannot allocate device memory where
// decode runs (for example a plugin whose host framework owns every device allocation and
// gives it no allocator, or a serving loop that must not allocate after start-up because
// cudaMalloc can stall the device and can fail under memory pressure).  The split-KV
// partial results go to a fixed array in device memory instead of a caller workspace.
// -----------------------------------------------------------------------------------------
#include <mutex>

namespace msa {
namespace {

// Largest split-KV scratch this entry point serves.  Every GPU that loads the library
// holds this much device memory until the process exits.
constexpr size_t kStaticScratchBytes = MSA_STATIC_DECODE_SCRATCH_BYTES;
static __device__ __align__(256) float g_static_scratch[kStaticScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device.  In host code the array's
// name only stands in for the symbol, so the address is looked up once per device (with
// that device current) and cached.
cudaError_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace msa

extern "C" msa_status msa_sparse_decode_static(const msa_shape* shape, const void* q,
                                               const void* k_cache, const void* v_cache,
                                               const int32_t* sel, void* out, float* lse,
                                               void* stream) {
  g_last_error[0] = 0;
  Dims d;
  MSA_TRY(make_dims(shape, &d));
  if (!d.decode) return fail(MSA_ERR_INVALID_ARG, "msa_sparse_decode_static needs seq_q == q_tile == 1");
  if (d.G > 64) return fail(MSA_ERR_UNSUPPORTED, "decode needs n_heads_q / n_heads_kv <= 64");
  MSA_TRY(check_ptr(q, "q"));
  MSA_TRY(check_ptr(k_cache, "k_cache"));
  MSA_TRY(check_ptr(v_cache, "v_cache"));
  MSA_TRY(check_ptr(sel, "sel"));
  MSA_TRY(check_ptr(out, "out"));
  MSA_TRY(check_ptr(lse, "lse", true));
  const size_t need = decode_workspace_bytes(d);
  if (need > kStaticScratchBytes)
    return fail(MSA_ERR_UNSUPPORTED,
                "this shape needs %zu bytes of decode scratch; the library's static array "
                "holds %zu (use msa_sparse_decode with a caller workspace)",
                need, kStaticScratchBytes);
  void* ws = nullptr;
  cudaError_t e = static_scratch_address(&ws);
  if (e != cudaSuccess) return cuda_fail(e, "msa_sparse_decode_static scratch address");
  // Every partial slot the merge reads is written by this call first, so the array's
  // previous contents never matter and nothing needs clearing.
  e = launch_debug_validate(d, sel, (cudaStream_t)stream, status_ptr());
  if (e != cudaSuccess) return cuda_fail(e, "msa_sparse_decode_static debug validation");
  e = launch_sparse_decode(d, q, k_cache, v_cache, sel, out, lse, static_cast<float*>(ws),
                           (cudaStream_t)stream, status_ptr());
  return e == cudaSuccess ? MSA_OK : cuda_fail(e, "msa_sparse_decode_static launch");
}
