/*
 * msa.h -- C ABI of the MiniMax Sparse Attention (MSA) hot path for GB300 (sm_103a).
 *
 * The method (from the talk pages on MSA):
 *   - an index branch runs lightweight causal full attention with one index query head
 *     per KV head against ONE shared index key head, and its scores are reduced to
 *     per-key-block scores ("Sparse Attention Cannot Be Directly Ported Across
 *     Architectures", disconfirmai.com, paragraph introducing MSA; "How MiniMax M3 was
 *     built", aietalks.com, section "MSA uses a lightweight index branch before sparse
 *     attention");
 *   - every KV head takes its own top-k of blocks, never merged across heads (same
 *     article, paragraph "MSA addresses these issues"; aietalks.com, section
 *     "Block-level retrieval makes sparse attention easier to run on GPUs");
 *   - the main GQA branch computes exact softmax attention over the selected blocks only
 *     (Chinese topic page on MSA, summary paragraph).
 * The pages fix no block size, k, pooling or tie-break; this library uses: scores are the
 * MAX over a query tile's tokens and a block's causally visible keys of
 * index_scale * <q_I, k_I>; the block holding the tile's last query (the "current block")
 * is always selected and counts towards top_k; the other top_k-1 are the highest scores,
 * ties to the lower block index, -0 == +0; the list is written ascending, padded with -1.
 *
 * Layouts (row-major, contiguous, element type = shape->dtype unless stated):
 *   q, out        [batch, seq_q, n_heads_q, head_dim]
 *   k, v          [batch, n_heads_kv, seq_k, head_dim]    (head-major: a block of one
 *                                                          KV head is one contiguous run)
 *   idx_q         [batch, seq_q, n_heads_kv, index_dim]   (index query head g serves KV head g)
 *   idx_k         [batch, seq_k, index_dim]               (the single index key head)
 *   block_scores  float32 [batch, n_heads_kv, n_rows, n_blocks]
 *   sel           int32   [batch, n_heads_kv, n_rows, top_k]
 *   lse           float32 [batch, n_heads_q, seq_q], natural log
 * with n_blocks = ceil(seq_k / block_size) and n_rows = ceil(seq_q / q_tile).
 *
 * Two modes, told apart by the shape:
 *   prefill  seq_q == seq_k == T, query i at position i, rows are tiles of q_tile queries
 *            (block_size % q_tile == 0);
 *   decode   seq_q == 1, q_tile == 1, seq_k == L (the cache includes the new token), the
 *            query at position L-1, one row per sequence (selection per token).
 * Query head h uses KV head h / (n_heads_q / n_heads_kv).
 *
 * Conventions:
 *   - Ownership: the caller owns every buffer.  Only msa_sparse_decode needs scratch, and
 *     the caller passes it (msa_workspace_bytes); no entry point here allocates memory.
 *   - Pointers are device pointers (cudaMalloc or equivalent), 16-byte aligned.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns after launching.  Argument checks happen before any launch; on
 *     failure nothing is launched and msa_last_error() describes the problem.
 *   - A kernel that gives up a bounded wait sets a device status word that
 *     msa_get_device_status() reports as MSA_ERR_TIMEOUT.
 *   - Inputs must be finite; NaN scores give an unspecified (but in-range) selection.
 *   - Calls on distinct streams may run concurrently; the device status word is shared.
 *   - The library looks up the device addresses of its own device variables (the status
 *     word, the static decode scratch) once per device and caches them.  cudaDeviceReset
 *     (or any other teardown of the primary context) leaves those addresses stale: using
 *     the library in the same process after a device reset is not supported.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MSA_ABI_VERSION 2

typedef enum msa_status {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, inconsistent or out-of-range shape */
  MSA_ERR_UNSUPPORTED = 2, /* valid shape that no kernel here handles (e.g. head_dim 96) */
  MSA_ERR_CUDA = 3,        /* a CUDA call or kernel launch failed */
  MSA_ERR_TIMEOUT = 4,     /* a kernel gave up a bounded wait (device status word) */
  MSA_ERR_BOUNDS = 5       /* debug builds only: a device-side index check failed (device
                            * status word; see msa_debug_build) */
} msa_status;

typedef enum msa_dtype { MSA_F32 = 0, MSA_BF16 = 1 } msa_dtype;

typedef struct msa_shape {
  int32_t batch;       /* B >= 1 */
  int32_t seq_q;       /* prefill: T; decode: 1 */
  int32_t seq_k;       /* prefill: T; decode: cache length L >= 1 */
  int32_t n_heads_q;   /* Hq, a multiple of n_heads_kv */
  int32_t n_heads_kv;  /* Hkv = number of index query heads; batch * Hkv <= 65535 */
  int32_t head_dim;    /* d: 64 or 128 */
  int32_t index_dim;   /* dI: 64 or 128 */
  int32_t block_size;  /* keys per block, >= 1; at most 32768 blocks per sequence */
  int32_t top_k;       /* blocks per KV head, current block included, >= 1 */
  int32_t q_tile;      /* queries sharing one selection: prefill divides block_size (at most
                        * 65535 tiles per sequence); decode 1 */
  int32_t dtype;       /* msa_dtype of q, k, v, idx_q, idx_k, out */
  float sm_scale;      /* softmax scale; 0 means 1/sqrt(head_dim) */
  float index_scale;   /* index logit scale; 0 means 1/sqrt(index_dim) */
} msa_shape;

/* Index branch: block_scores[b, g, m, blk] = max over the queries t of row m and the keys
 * j <= t of block blk of index_scale * <idx_q[b, t, g, :], idx_k[b, j, :]>; -inf for blocks
 * with no visible key.  Accumulation is fp32.  Prefill uses tcgen05 tensor cores for
 * bf16 with index_dim 128; decode is a streaming scan of the index-key cache. */
msa_status msa_index_scores(const msa_shape* shape, const void* idx_q, const void* idx_k,
                            float* block_scores, void* stream);

/* Per-KV-head block top-k of block_scores (layout above) into sel: the current block plus
 * the best top_k-1 of the earlier blocks by (score desc, index asc), ascending, -1 padded.
 * Bit-exact and deterministic.  Rows may hold up to 32768 candidate blocks. */
msa_status msa_block_topk(const msa_shape* shape, const float* block_scores, int32_t* sel,
                          void* stream);

/* Ablation, not MSA: the aggregated selection the pages contrast MSA with (DSA-style, one
 * token set shared by every KV head).  For each (sequence, row) the candidates' scores are
 * the fp32 sums of the KV heads' block scores, added in head order 0, 1, ...; one selection
 * by the same rule as msa_block_topk is written to every head's row of sel.  Used to
 * measure the head-diversity loss of sharing ("Sparse Attention Cannot Be Directly Ported
 * Across Architectures", paragraph on applying DSA to GQA). */
msa_status msa_block_topk_shared(const msa_shape* shape, const float* block_scores,
                                 int32_t* sel, void* stream);

/* msa_index_scores followed by msa_block_topk in one launch, without the block-score round
 * trip through HBM: the index kernel keeps each KV head's running best top_k-1 blocks as
 * the scores of successive blocks come out of the tensor cores, and writes sel directly
 * (same selection rule, bit-identical to the two calls).  block_scores may be NULL; when
 * given, it is filled as by msa_index_scores.  bf16 prefill with index_dim 128,
 * block_size 128, q_tile 64, 4 KV heads and top_k <= 256; other shapes get
 * MSA_ERR_UNSUPPORTED. */
msa_status msa_index_topk_fused(const msa_shape* shape, const void* idx_q, const void* idx_k,
                                float* block_scores, int32_t* sel, void* stream);

/* Main branch, prefill (seq_q == seq_k): for query t and head h (KV head g), attend over the
 * keys j <= t of the blocks listed in sel[b, g, t / q_tile, :] (entries -1 are skipped;
 * entries must be distinct).  Writes out (dtype) and, if lse != NULL, lse.  A row whose key
 * set is empty gets out = 0 and lse = -inf.  workspace may be NULL (ws_bytes 0). */
msa_status msa_sparse_prefill(const msa_shape* shape, const void* q, const void* k,
                              const void* v, const int32_t* sel, void* out, float* lse,
                              void* workspace, size_t ws_bytes, void* stream);

/* Training: gradients of msa_sparse_prefill for a loss L with dL/dout = dout.  Inputs are
 * the forward's q, k, v, sel, its out (dtype) and lse (natural log), and dout (dtype, same
 * layout as out).  Outputs, float32: dq [batch, seq_q, n_heads_q, head_dim] (written),
 * dk and dv [batch, n_heads_kv, seq_k, head_dim] (cleared on the stream, then accumulated:
 * a key block selected by several tiles collects all their contributions).  With p the
 * attention weights, D = dout . out, ds = p (dout . v - D): dq = sm_scale sum ds k,
 * dk += sm_scale ds q, dv += p dout.  bf16 shapes with head_dim 128, block 128, q_tile 64
 * run on the tensor cores (a query-tile pass for dq, a key-block pass for dk / dv) and need
 * a device workspace of msa_workspace_bytes(shape, 2) bytes (per-row D and a bitmap of
 * which tiles selected which blocks); other shapes run on CUDA cores and need none
 * (workspace may then be null).  dk / dv sums over several CTAs use fp32 atomics, so their
 * last bits can vary from run to run. */
msa_status msa_sparse_prefill_backward(const msa_shape* shape, const void* q, const void* k,
                                       const void* v, const int32_t* sel, const void* out,
                                       const float* lse, const void* dout, float* dq, float* dk,
                                       float* dv, void* workspace, size_t ws_bytes,
                                       void* stream);

/* Training the index branch (the pages: the index branch is trained with a KL loss to match
 * the main branch's attention).  The pages give no formula; this library's reading: for
 * token t and KV head g, over the keys J the main branch attends (selected blocks, j <= t),
 * the target is the main branch's attention distribution averaged over the group's query
 * heads (held constant; computed from q, k and the forward's lse), the index distribution
 * is the softmax over J of index_scale <idx_q[t,g], idx_k[j]>, and
 *   loss = sum over (t, g) of KL(target || index)          (natural log).
 * Outputs, float32: loss (one device scalar, cleared then accumulated), d_idx_q [batch,
 * seq_q, n_heads_kv, index_dim] (written), d_idx_k [batch, seq_k, index_dim] (cleared, then
 * accumulated over every tile and head): the gradients of loss.  Prefill shapes, at most
 * 64 query heads per KV head.  bf16 shapes with head_dim = index_dim = 128, block 128,
 * q_tile 64 and 2, 4, 8, 16 or 32 query heads per KV head run on the tensor cores (a
 * query-tile pass for the loss and d_idx_q, a key-block pass for d_idx_k) and need a
 * device workspace of msa_workspace_bytes(shape, 3) bytes; other shapes run on CUDA cores
 * in fp32 and need none.  d_idx_k and the loss are sums with fp32 atomics, so their last
 * bits can vary from run to run. */
msa_status msa_index_kl_loss(const msa_shape* shape, const void* q, const void* k,
                             const float* lse, const void* idx_q, const void* idx_k,
                             const int32_t* sel, float* loss, float* d_idx_q, float* d_idx_k,
                             void* workspace, size_t ws_bytes, void* stream);

/* Main branch, decode (seq_q == 1, q_tile == 1): the new token of every sequence attends
 * over the selected blocks of the cache (split over the blocks, partial results merged by
 * log-sum-exp).  workspace: device scratch of at least msa_workspace_bytes(shape, 1)
 * bytes, 16-byte aligned, owned by the caller; its contents on entry do not matter. */
msa_status msa_sparse_decode(const msa_shape* shape, const void* q, const void* k_cache,
                             const void* v_cache, const int32_t* sel, void* out, float* lse,
                             void* workspace, size_t ws_bytes, void* stream);

/* Decode for callers that cannot allocate device memory.  Some callers have no way to
 * call cudaMalloc where decode runs: a plugin whose host framework owns every device
 * allocation and hands it no allocator, or a serving loop that must not allocate after
 * start-up because cudaMalloc can stall the device and can fail under memory pressure.
 * This entry point computes exactly what msa_sparse_decode computes, with the same
 * arguments minus the workspace: the split-KV partial results go to a scratch array the
 * library keeps in device memory (MSA_STATIC_DECODE_SCRATCH_BYTES, held on every GPU that
 * loads the library until the process exits).  The talk pages have no counterpart to it.
 *   - A shape whose scratch (msa_workspace_bytes(shape, 1)) exceeds the array is rejected
 *     with MSA_ERR_UNSUPPORTED before anything runs; msa_last_error() names both sizes.
 *   - The first call on each device looks up the array's device address with that device
 *     current (cudaGetSymbolAddress) and caches it; make that first call before any stream
 *     capture.
 *   - Every call on a device uses the same array.  Calls that overlap on the GPU (other
 *     streams, other host threads) race on it and corrupt each other's results: serialise
 *     them.  Each call writes every scratch entry it reads, so leftovers of earlier calls do
 *     not matter and nothing needs clearing.
 *   - It calls no cudaMalloc, cudaFree or allocating library routine. */
#define MSA_STATIC_DECODE_SCRATCH_BYTES (8u << 20)
msa_status msa_sparse_decode_static(const msa_shape* shape, const void* q, const void* k_cache,
                                    const void* v_cache, const int32_t* sel, void* out,
                                    float* lse, void* stream);

/* Decode over a paged cache with a length per sequence (the serving form of decode).
 * shape: a decode shape (seq_q = q_tile = 1) whose seq_k is the capacity of the block table
 * (n_blocks = ceil(seq_k / block_size) entries per sequence); bf16, head_dim = index_dim =
 * 128, block_size 128, 4 KV heads, at most 16 query heads per KV head.
 *   seq_lens     int32 [batch], device: cache length L_b of sequence b, 1 <= L_b <= seq_k
 *                (the new token, at position L_b - 1, is already in the cache; 0 means an
 *                empty sequence: scores -inf, sel -1, out 0, lse -inf).
 *   block_table  int32 [batch, n_blocks], device: physical block holding logical block j of
 *                sequence b (entries past the sequence's last block are not read).
 *   n_phys       number of physical blocks in the pools.
 *   idx_k_pool   [n_phys, block_size, index_dim];  k_pool, v_pool [n_phys, n_heads_kv,
 *                block_size, head_dim]: one physical block holds all KV heads' keys of 128
 *                consecutive positions, each head's block contiguous.
 * Semantics are those of the contiguous decode on each sequence's logical cache.  Entries
 * of block_table outside [0, n_phys) read as zeros (no fault) and give meaningless output.
 * The three calls chain like the contiguous ones; msa_sparse_decode_paged takes the same
 * workspace as msa_sparse_decode (msa_workspace_bytes(shape, 1)). */
msa_status msa_index_scores_paged(const msa_shape* shape, const int32_t* seq_lens,
                                  const int32_t* block_table, int32_t n_phys, const void* idx_q,
                                  const void* idx_k_pool, float* block_scores, void* stream);
msa_status msa_block_topk_ragged(const msa_shape* shape, const int32_t* seq_lens,
                                 const float* block_scores, int32_t* sel, void* stream);
msa_status msa_sparse_decode_paged(const msa_shape* shape, const int32_t* seq_lens,
                                   const int32_t* block_table, int32_t n_phys, const void* q,
                                   const void* k_pool, const void* v_pool, const int32_t* sel,
                                   void* out, float* lse, void* workspace, size_t ws_bytes,
                                   void* stream);

/* Scratch bytes msa_sparse_prefill (which = 0), msa_sparse_decode (which = 1),
 * msa_sparse_prefill_backward (which = 2) or msa_index_kl_loss (which = 3) needs for this
 * shape; 0 when none.  Returns 0 for an invalid shape. */
size_t msa_workspace_bytes(const msa_shape* shape, int which);

/* Synchronises `stream`, then reports (and clears) the device status word and any pending
 * CUDA error: MSA_OK, MSA_ERR_TIMEOUT or MSA_ERR_CUDA. */
msa_status msa_get_device_status(void* stream);

/* Static description of a status code. */
const char* msa_status_string(msa_status status);

/* Human-readable detail of the last failure on the calling thread ("" if none). */
const char* msa_last_error(void);

/* Test hook for the failure path.  mode 1: every tensor-core sparse-prefill launch made
 * afterwards (from any thread) has its copy-issuing warp issue nothing, so the warps that
 * wait for the copies give up after their one-second bound, the kernel writes zeros and
 * -inf, and the next msa_get_device_status() reports MSA_ERR_TIMEOUT.  No copy or MMA is
 * ever in flight in this mode, and the CUDA context stays usable.  mode 0 (default):
 * normal operation.  Any other mode: MSA_ERR_INVALID_ARG. */
msa_status msa_debug_set_fault(int32_t mode);

/* MSA_ABI_VERSION of the loaded library. */
int32_t msa_abi_version(void);

/* 1 when the library was built with -DMSA_DEBUG, else 0.  A debug build checks on the
 * device, before the kernels of each call run, every selection entry it is given (-1 or a
 * block of the sequence: below ceil(seq_k / block_size), or below ceil(seq_lens[b] /
 * block_size) for a paged cache; no block twice in a row), every block-table entry of the
 * sequence's blocks (within [0, n_phys)) and every cache length (within [0, seq_k]); and,
 * inside the tensor-core kernels, the coordinates of their tensor copies and the indices of
 * their output stores.  A failed check records a code in the device status word, which
 * msa_get_device_status() reports as MSA_ERR_BOUNDS; no check traps, and an out-of-range
 * store is skipped.  Release builds carry none of these checks (they skip selection entries
 * outside [0, n_blocks) without reporting them). */
int32_t msa_debug_build(void);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
