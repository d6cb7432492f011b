/*
 * csgmv.h — C ABI of libcsgmv.so, the GB300 (sm_103a) chunked segmented-gather
 * matrix-vector (csgmv) multi-adapter LoRA delta path.
 *
 * The operations follow sglang's LoRA backend interface as printed in
 *   python/sglang/srt/lora/backend/base_backend.py   (class BaseLoRABackend)
 *   python/sglang/srt/lora/backend/chunked_backend.py (class ChunkedSgmvLoRABackend)
 *   python/sglang/srt/lora/lora_manager.py            (LoRAManager.prepare_lora_batch)
 *
 * Conventions for every call:
 *  - Pointers are DEVICE pointers owned by the caller unless marked "host".
 *    The library allocates nothing, frees nothing and never synchronizes; all
 *    work is enqueued on the given stream (NULL = legacy default stream), so
 *    every call can be captured in a CUDA graph.
 *  - bf16 tensors are passed as void* holding IEEE bfloat16 values; all
 *    tensors are dense row-major with the stated shapes; every device pointer
 *    must be 16-byte aligned.
 *  - Return value: CSGMV_OK (0) or a negative CSGMV_ERR_* code; then nothing
 *    was enqueued (except CSGMV_ERR_CUDA, when a launch itself failed).
 *    csgmv_last_error() gives a message for the calling thread.
 *  - Problems only the device can see (a slot index out of range, a rank
 *    above the buffer rank, a token id outside the vocabulary, a permutation
 *    entry out of range, a segment-capacity overflow, inconsistent request
 *    lengths) are OR-ed as CSGMV_STATUS_* bits into the batch info's device
 *    status word; the offending work item is skipped, nothing traps.
 */
#ifndef CSGMV_H
#define CSGMV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CSGMV_API __attribute__((visibility("default")))
#else
#define CSGMV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st *csgmv_stream_t;

enum {
    CSGMV_OK = 0,
    CSGMV_ERR_INVALID_ARG = -1, /* bad pointer, size, dtype or offsets (host check) */
    CSGMV_ERR_CAPACITY = -2,    /* batch exceeds the batch-info buffers (host check) */
    CSGMV_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed */
    CSGMV_ERR_TIMEOUT = -4,     /* reserved: no call here waits on another agent */
    CSGMV_ERR_DEVICE = -5,      /* reserved for callers that map the status word */
    CSGMV_ERR_UNSUPPORTED = -6  /* shape outside this build's limits (e.g. rank > 64) */
};

enum { CSGMV_DTYPE_BF16 = 0, CSGMV_DTYPE_F32 = 1 };

/* Bits of the device status word (csgmv_batch_info.status). */
enum {
    CSGMV_STATUS_BAD_ADAPTER = 1,     /* slot index outside [0, num_loras) */
    CSGMV_STATUS_BAD_RANK = 2,        /* slot rank outside [0, max_rank] */
    CSGMV_STATUS_BAD_TOKEN_ID = 4,    /* embedding id outside [0, vocab_size) */
    CSGMV_STATUS_BAD_PERMUTATION = 8, /* permutation entry outside [0, num_tokens) */
    CSGMV_STATUS_CAPACITY = 16,       /* segments exceed max_segments */
    CSGMV_STATUS_BAD_LENS = 32        /* negative length or lengths not summing to num_tokens */
};

/*
 * Batch info shared by every layer of one forward batch (sglang LoRABatchInfo;
 * chunked_backend.py init_cuda_graph_batch_info / prepare_lora_batch).
 * The caller allocates every device buffer once at the capacities below
 * (csgmv_batch_info_capacity gives the CUDA-graph capacities) and fills the
 * capacity fields; csgmv_build_batch_info fills the buffers and the host
 * mirror fields in place, so graphs captured over these pointers stay valid
 * across batches.
 *
 * Meaning (chunked_backend.py _get_permutation / _get_segments_info):
 *   permutation[p]     original token index at adapter-sorted position p
 *                      (stable: ties keep token order)
 *   seg_indptr[k]      first sorted position of segment k; segment k holds
 *                      positions [seg_indptr[k], seg_indptr[k+1]) that all use
 *                      slot weight_indices[k], at most chunk_size of them
 *   lora_ranks[a], scalings[a]   rank r_a and scaling of slot a (0 = no adapter)
 */
typedef struct csgmv_batch_info {
    int32_t *seg_indptr;         /* [max_segments + 1] */
    int32_t *weight_indices;     /* [max_segments] */
    int32_t *permutation;        /* [max_tokens] */
    int32_t *lora_ranks;         /* [max_loras] */
    float *scalings;             /* [max_loras] */
    int32_t *num_segments_dev;   /* [1] segments of the current batch */
    int32_t *max_len_dev;        /* [1] chunk size of the current batch */
    int32_t *req_seg_indptr;     /* [max_bs + 1] per-request token indptr, or NULL */
    int32_t *req_weight_indices; /* [max_bs] per-request slot, or NULL */
    int32_t *status;             /* [1] CSGMV_STATUS_* bits; reset by each build */
    /* capacities (set by the caller) */
    int32_t max_segments, max_tokens, max_loras, max_bs, max_rank;
    /* host mirror of the current batch (set by csgmv_build_batch_info) */
    int32_t num_tokens, chunk_size, bs, num_loras, use_cuda_graph;
    /* Optional (NULL for none): the token tiles of the current batch, for the
     * decode kernels of csgmv_qkv, so that no CTA rebuilds them from the
     * segments.  csgmv_build_batch_info writes [0] = tile count and [1..3] =
     * 0, then per tile {slot, first sorted position, tokens, 0}: every slot
     * run (a maximal stretch of segments on one slot) cut into
     * ceil(n / 64) tiles of balanced size, in segment order;
     * csgmv_build_lm_head_batch_info writes [0] = -1 (no tiles: the kernels
     * derive them from the segments).  csgmv_tile_table_ints() gives its
     * int32 length. */
    int32_t *tile_table;
} csgmv_batch_info;

/* int32 entries of csgmv_batch_info.tile_table for these capacities:
 * 4 * (max_loras + max_tokens / 64 + 2).  Host only; 0 for negative sizes. */
CSGMV_API int64_t csgmv_tile_table_ints(int max_loras, int max_tokens);

/* Message of the last failed call on this thread ("" if none). */
CSGMV_API const char *csgmv_last_error(void);

/* Library version string. */
CSGMV_API const char *csgmv_version(void);

/*
 * Chunk size for a batch of num_tokens tokens (chunked_backend.py
 * MIN_CHUNK_SIZE = 16 and _determine_chunk_size_for_tokens): 16 when
 * max_chunk_size <= 16; else min(max_chunk_size, 128 if num_tokens >= 256,
 * 32 if num_tokens >= 64, else 16).  Host only; never fails.
 */
CSGMV_API int csgmv_chunk_size(int num_tokens, int max_chunk_size);

/*
 * CUDA-graph capacities (chunked_backend.py init_cuda_graph_batch_info):
 * *max_segments = ceil(num_tokens_per_bs / 16) * max_bs and
 * *max_tokens = max_bs * num_tokens_per_bs (host pointers).  Returns
 * CSGMV_ERR_INVALID_ARG for negative sizes or int32 overflow.
 */
CSGMV_API int csgmv_batch_info_capacity(int max_bs, int num_tokens_per_bs, int32_t *max_segments,
                              int32_t *max_tokens);

/*
 * Build the batch info of one forward batch on the device (chunked_backend.py
 * prepare_lora_batch with _get_permutation and _get_segments_info;
 * lora_manager.py prepare_lora_batch for the slot ranks and scalings).
 *   req_lens[bs], req_adapter[bs]   device; tokens and slot of each request in
 *                                   token order (a decode request has 1 token)
 *   num_tokens                      host; sum of req_lens (checked on device)
 *   lora_ranks[num_loras], scalings[num_loras]  device; copied into the batch
 *                                   info (slots [num_loras, max_loras) get 0)
 *   max_chunk_size, chunk_size_override   chunk = override if > 0, else
 *                                   csgmv_chunk_size(num_tokens, max_chunk_size)
 *   use_cuda_graph                  1: pad weight_indices[n:max_segments] = 0 and
 *                                   seg_indptr[n+1:max_segments+1] = num_tokens
 * One single-CTA kernel; resets bi->status.  Host errors: bs > max_bs,
 * num_tokens > max_tokens, num_loras > max_loras, negative sizes, NULL buffers,
 * or a batch too large for one CTA's shared memory (CSGMV_ERR_UNSUPPORTED).
 * On a device-side error (status bits BAD_ADAPTER / BAD_LENS / BAD_RANK /
 * CAPACITY) the batch is left with zero segments, so later calls do nothing.
 */
CSGMV_API int csgmv_build_batch_info(csgmv_batch_info *bi, const int32_t *req_lens, const int32_t *req_adapter,
                           int bs, int num_tokens, const int32_t *lora_ranks, const float *scalings,
                           int num_loras, int max_chunk_size, int chunk_size_override,
                           int use_cuda_graph, csgmv_stream_t stream);

/*
 * Batch info of a pruned lm_head pass (chunked_backend.py
 * _prepare_lm_head_batch_info and _build_lm_head_batch_info): only
 * pruned_lens[i] tokens of request i go through lm_head, and they stay in
 * their original order, so the permutation is the identity.  Segments come
 * from merge_and_chunk_segments(weight_indices, pruned_lens, chunk), whose
 * body is not on the pages; read from its call sites: consecutive requests on
 * the same slot form one run (requests without pruned tokens are skipped, so
 * runs merge across them), and every run is cut into pieces of chunk tokens,
 * the last one shorter.  chunk = chunk_size_override if > 0, else
 * csgmv_chunk_size(num_tokens, max_chunk_size).
 *   pruned_lens[bs], req_adapter[bs]   device; pruned tokens and slot of each
 *                                      request, in request order
 *   num_tokens                         host; sum of pruned_lens
 *   lora_ranks, scalings, num_loras, use_cuda_graph   as csgmv_build_batch_info
 * The result drives csgmv_shrink / csgmv_expand / csgmv_qkv over the pruned
 * rows (x and base_output with num_tokens rows).  Runs here follow request
 * order, not slot order, so the batch info needs max_segments of up to
 * ceil(num_tokens / chunk) plus the number of requests with pruned tokens
 * (CSGMV_STATUS_CAPACITY otherwise).  req_seg_indptr and
 * req_weight_indices are not written.  One single-CTA kernel; errors as
 * csgmv_build_batch_info.
 */
CSGMV_API int csgmv_build_lm_head_batch_info(csgmv_batch_info *bi, const int32_t *pruned_lens,
                                   const int32_t *req_adapter, int bs, int num_tokens,
                                   const int32_t *lora_ranks, const float *scalings, int num_loras,
                                   int max_chunk_size, int chunk_size_override, int use_cuda_graph,
                                   csgmv_stream_t stream);

/*
 * Shrink (base_backend.py run_lora_a_sgemm; chunked_backend.py
 * run_lora_a_sgemm with num_slices): for token t on slot w with rank r,
 *     h[t][j*r + k] = sum_i x[t][i] * A[w][j*r + k][i]     (j < c, k < r)
 * and h[t][n] = 0 for c*r <= n < c*R (also for rank-0 tokens).
 *   x  bf16 (s, K), s = bi->num_tokens;  A  bf16 (max_loras, c*R, K), R = bi->max_rank
 *   h  (s, ldh) of h_dtype (CSGMV_DTYPE_BF16 rounds to nearest even,
 *      CSGMV_DTYPE_F32 keeps fp32), ldh >= c*R; only columns [0, c*R) are written
 *   num_slices c in {1, 2, 3}; K a multiple of 8; R in {8, 16, 32, 64}.
 * fp32 accumulation on the tensor cores.
 */
CSGMV_API int csgmv_shrink(const void *x, int64_t s, int64_t K, const void *A, int num_slices, void *h,
                 int h_dtype, int64_t ldh, const csgmv_batch_info *bi, csgmv_stream_t stream);

/*
 * Expand (base_backend.py run_lora_b_sgemm; chunked_backend.py
 * run_lora_b_sgemm / run_qkv_lora with slice_offsets, max_slice_size and
 * base_output): for token t on slot w with rank r and scaling sigma, slice j
 * and column n in [off[j], off[j+1]),
 *     out[t][n] = (accumulate ? out[t][n] : 0) + sigma * sum_{k<r} h[t][j*r+k] * B[w][n][k]
 * rounded once to bf16.  Columns outside [off[0], off[c]) are not touched;
 * with accumulate = 1 rows of rank-0 tokens are not touched either, with
 * accumulate = 0 they are set to 0 in the covered columns.
 *   h   (s, ldh) of h_dtype, as produced by csgmv_shrink
 *   B   bf16 (max_loras, N, R);  out  bf16 (s, N), in place when accumulate = 1
 *   slice_offsets  HOST int32[c+1], non-decreasing, multiples of 8, off[c] <= N
 *   max_slice_size >= the widest slice (sglang passes it to size the launch)
 * The fp32 h is applied as a bf16 hi + lo pair, so the product keeps ~16 bits.
 */
CSGMV_API int csgmv_expand(const void *h, int h_dtype, int64_t ldh, const void *B, int64_t N,
                 const int32_t *slice_offsets, int num_slices, int max_slice_size, void *out,
                 int accumulate, const csgmv_batch_info *bi, csgmv_stream_t stream);

/*
 * Fused shrink -> expand (chunked_backend.py run_qkv_lora and
 * run_gate_up_lora; c = 1 is the single-projection pair run_lora_a_sgemm +
 * run_lora_b_sgemm):
 *     base_output[t][n] += sigma_w * sum_k (sum_i x[t][i] A[w][j*r+k][i]) B[w][n][k]
 * for n in slice j = [off[j], off[j+1]).  h stays fp32, so the only rounding
 * to bf16 is the final store.  Shapes and limits as csgmv_shrink and
 * csgmv_expand; base_output is bf16 (s, N), updated in place.
 *   workspace, workspace_bytes   optional device scratch for h (NULL / 0 for
 *       none).  Without it h never leaves the chip (reduced across a
 *       thread-block cluster in distributed shared memory).  With room for
 *       a 256-byte header and one plane of fp32 h (num_tokens * num_slices *
 *       max_rank * 4 bytes; csgmv_qkv_workspace_bytes() covers every batch
 *       and the widest split of K), two kinds of call instead run the shrink and the expand
 *       as two kernels with h in the workspace, which is faster there:
 *       batches of long per-slot runs (128-token tiles, max_rank >= 16),
 *       decode batches (short per-slot runs onto fewer than 32768 columns,
 *       at most 2048 tokens, max_segments <= 512 and max_loras <= 256), and
 *       short per-slot runs with at least 32768 output columns (a
 *       vocabulary-wide lm_head).  The shrink may cut K into parts, one plane
 *       of partial sums each, that the expand adds in part order, so results
 *       do not depend on timing.  csgmv_qkv_path() tells which path a call
 *       takes.  Its contents on entry do
 *       not matter; on return they are unspecified.  It must be 16-byte
 *       aligned and must not overlap any other argument.
 */
CSGMV_API int csgmv_qkv(const void *x, int64_t K, const void *A, const void *B, int64_t N,
              const int32_t *slice_offsets, int num_slices, int max_slice_size, void *base_output,
              void *workspace, size_t workspace_bytes, const csgmv_batch_info *bi, csgmv_stream_t stream);

/*
 * Tuple-form B (base_backend.py run_qkv_lora: qkv_lora_b as a tuple of a q
 * buffer (1, num_lora, output_dim_q, r) and a combined kv buffer
 * (2, num_lora, output_dim_kv, r); run_gate_up_lora: gate_up_lora_b as a tuple
 * of two (num_lora, output_dim, r) buffers).  These are csgmv_expand and
 * csgmv_qkv with B given per slice instead of as one tensor:
 *   B_slices  HOST array of num_slices device pointers; B_slices[j] is bf16
 *             (max_loras, off[j+1] - off[j], R), row 0 being output column
 *             off[j].  For the qkv tuple: {q, kv, kv + max_loras * N_kv * R}.
 * Every slice offset must be a multiple of 64 (CSGMV_ERR_UNSUPPORTED
 * otherwise); everything else, results included, is as the single-tensor call.
 */
CSGMV_API int csgmv_expand_sliced(const void *h, int h_dtype, int64_t ldh, const void *const *B_slices, int64_t N,
                                  const int32_t *slice_offsets, int num_slices, int max_slice_size, void *out,
                                  int accumulate, const csgmv_batch_info *bi, csgmv_stream_t stream);
CSGMV_API int csgmv_qkv_sliced(const void *x, int64_t K, const void *A, const void *const *B_slices, int64_t N,
                               const int32_t *slice_offsets, int num_slices, int max_slice_size, void *base_output,
                               void *workspace, size_t workspace_bytes, const csgmv_batch_info *bi,
                               csgmv_stream_t stream);

/* Kernel paths of csgmv_qkv (csgmv_qkv_path). */
enum {
    CSGMV_PATH_FUSED = 0,       /* one kernel: h reduced across a thread-block cluster, never in memory */
    CSGMV_PATH_DECODE = 1,      /* decode batches: split-K shrink into fp32 planes, then the expand */
    CSGMV_PATH_SMALL_SPLIT = 2, /* short runs onto vocabulary-wide outputs: small-tile shrink, then expand */
    CSGMV_PATH_STREAM = 3       /* 128-token tiles: streaming tcgen05 shrink, then streaming expand */
};

/*
 * The path csgmv_qkv takes for the batch last built into bi, with these
 * shapes (as csgmv_qkv's K, N, slice_offsets, num_slices) and a workspace of
 * workspace_bytes (0 for none).  Host only: reads the capacity and host
 * mirror fields of bi, launches nothing, needs no GPU.  Returns a
 * CSGMV_PATH_* value (CSGMV_PATH_FUSED for an empty batch), or
 * CSGMV_ERR_INVALID_ARG / CSGMV_ERR_UNSUPPORTED as csgmv_qkv would for the
 * same shapes.  Paths other than CSGMV_PATH_FUSED launch two kernels.
 */
CSGMV_API int csgmv_qkv_path(const csgmv_batch_info *bi, int64_t K, int64_t N, const int32_t *slice_offsets,
                             int num_slices, size_t workspace_bytes);

/* Workspace bytes that let csgmv_qkv use its two-kernel paths for any batch
 * of this batch info, with h (fp32) held as partial sums over parts of K
 * (planes of max_tokens * num_slices * max_rank floats) after a 256-byte
 * header: 256 + P * max_tokens * num_slices * max_rank * 4 with P = 4, or
 * P = 32 * min(max_tokens, 2048) / max_tokens when that is more (room for the
 * decode kernels' 32 parts).  A smaller workspace of at least 256 +
 * num_tokens * num_slices * max_rank * 4 bytes also takes the paths, with
 * fewer parts. */
CSGMV_API size_t csgmv_qkv_workspace_bytes(const csgmv_batch_info *bi, int num_slices);

/*
 * csgmv_qkv for callers that cannot allocate device memory when they call it
 * (no counterpart on the pages: an addition of this library).  Some callers
 * cannot call cudaMalloc or a caching allocator at that point (for instance
 * code whose device memory is planned up front by an engine that owns every
 * buffer), so they cannot provide csgmv_qkv's workspace.  This entry point
 * takes the same arguments without one and uses a fixed 32 MiB array in the
 * library's own device memory as the h workspace; the library allocates
 * nothing and frees nothing here either.
 *   - Limit: when csgmv_qkv would take a two-kernel path, the batch's h,
 *     num_tokens * num_slices * max_rank * 4 bytes, and a 256-byte header
 *     must fit in 32 MiB, else CSGMV_ERR_CAPACITY (nothing is launched).  A
 *     batch whose h does not fit but which csgmv_qkv runs as one kernel
 *     (csgmv_qkv_path gives CSGMV_PATH_FUSED even with an unbounded
 *     workspace) runs that way, with no workspace.
 *   - Every GPU that loads the library holds the 32 MiB until the process
 *     exits.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before capturing the stream.
 *   - All calls share the one array: two calls that may run at the same time
 *     on the GPU (different streams, or unordered graph branches) race on it.
 *     Nothing in it has to start at zero; the shrink writes every h row the
 *     expand reads.
 */
CSGMV_API int csgmv_qkv_static_scratch(const void *x, int64_t K, const void *A, const void *B, int64_t N,
                             const int32_t *slice_offsets, int num_slices, int max_slice_size,
                             void *base_output, const csgmv_batch_info *bi, csgmv_stream_t stream);

/*
 * Embedding LoRA-A gather (base_backend.py run_lora_a_embedding;
 * chunked_backend.py run_lora_a_embedding, which takes no extra-token
 * embeddings): for token t on slot w with rank r,
 *     out[t][k] = A_emb[w][k][input_ids[t]]  for k < r,  0 for r <= k < rank.
 *   input_ids int32 (s,), s = bi->num_tokens;  A_emb bf16 (max_loras, rank, vocab_size)
 *   out bf16 (s, rank);  1 <= rank <= 1024.
 * An id outside [0, vocab_size) sets CSGMV_STATUS_BAD_TOKEN_ID and leaves
 * that row 0.  Bit-exact copy; no arithmetic.
 */
CSGMV_API int embedding_lora_a(const int32_t *input_ids, const void *A_emb, int64_t vocab_size, int rank,
                     void *out, const csgmv_batch_info *bi, csgmv_stream_t stream);

/*
 * Embedding LoRA-A gather with extra tokens (base_backend.py
 * run_lora_a_embedding with extra_embeddings: tokens with ids >= vocab_size
 * are extra tokens the adapter adds beyond the base vocabulary).  For token t
 * on slot w with rank r:
 *     out[t][k] = A_emb[w][k][id]                    0 <= id < vocab_size
 *     out[t][k] = extra_embeddings[w][id - vocab_size][k]
 *                                 vocab_size <= id < vocab_size + num_extra_tokens
 * for k < r, and 0 for r <= k < rank.
 *   extra_embeddings  bf16 (max_loras, num_extra_tokens, rank); may be NULL
 *                     when num_extra_tokens = 0 (then this is embedding_lora_a)
 *   other arguments as embedding_lora_a; out must be 16-byte aligned when rank
 *   is a multiple of 8.
 * An id outside [0, vocab_size + num_extra_tokens) sets
 * CSGMV_STATUS_BAD_TOKEN_ID and leaves that row 0.  Bit-exact copy.
 */
CSGMV_API int embedding_lora_a_extra(const int32_t *input_ids, const void *A_emb, int64_t vocab_size, int rank,
                                     const void *extra_embeddings, int64_t num_extra_tokens, void *out,
                                     const csgmv_batch_info *bi, csgmv_stream_t stream);

/*
 * embedding_lora_a_extra with A_emb stored transposed: A_emb_t bf16
 * (max_loras, vocab_size, rank), A_emb_t[w][id][k] = A_emb[w][k][id].  The
 * (max_loras, rank, vocab_size) layout of the pages puts each of a token's
 * rank values in its own 32-byte memory sector; here they are one
 * contiguous row, so the gather reads rank * 2 bytes per token instead of
 * rank sectors.  A caller transposes each adapter once when it loads it
 * (csgmv_transpose_embedding).  Results are identical to
 * embedding_lora_a_extra on the untransposed table.  An addition of this
 * library (the load-time layout is not on the pages).
 */
CSGMV_API int embedding_lora_a_transposed(const int32_t *input_ids, const void *A_emb_t, int64_t vocab_size,
                                          int rank, const void *extra_embeddings, int64_t num_extra_tokens,
                                          void *out, const csgmv_batch_info *bi, csgmv_stream_t stream);

/*
 * A_emb_t[w][v][k] = A_emb[w][k][v] for w < num_loras (both bf16, device):
 * the load-time layout of embedding_lora_a_transposed.  Asynchronous on
 * stream; the two buffers must not overlap.  1 <= rank <= 1024.
 */
CSGMV_API int csgmv_transpose_embedding(const void *A_emb, int64_t num_loras, int rank, int64_t vocab_size,
                                        void *A_emb_t, csgmv_stream_t stream);

/*
 * Extra-token embedding (base_backend.py run_extra_token_embedding): in the
 * (s, embed_dim) output of the base embedding, the row of every token t on
 * slot w with vocab_size <= id < vocab_size + num_extra_tokens becomes
 *     output[t][:] = extra_embeddings[w][id - vocab_size][:]
 * (the base vocabulary has no row for it); rows of ids below vocab_size are
 * not touched.
 *   input_ids         int32 (s,), s = bi->num_tokens (tokens mapped to slots
 *                     by the batch info)
 *   output            bf16 (s, embed_dim), updated in place
 *   extra_embeddings  bf16 (max_loras, num_extra_tokens, embed_dim)
 * Both bf16 tensors must be 16-byte aligned when embed_dim is a multiple of
 * 8.  An id outside [0, vocab_size + num_extra_tokens) sets
 * CSGMV_STATUS_BAD_TOKEN_ID and leaves the row untouched; num_extra_tokens = 0
 * does nothing.  Bit-exact copy.
 */
CSGMV_API int extra_token_embedding(const int32_t *input_ids, void *output, int64_t embed_dim,
                                    const void *extra_embeddings, int64_t num_extra_tokens, int64_t vocab_size,
                                    const csgmv_batch_info *bi, csgmv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CSGMV_H */
