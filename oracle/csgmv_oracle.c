/*
 * CPU oracle for the chunked segmented-gather (csgmv) multi-adapter LoRA path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this file.  Only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no header, helper or table with the CUDA
 * library: every conversion and index rule below is written out here again.
 *
 * Sources (sglang, as printed on the pages):
 *   [CB]  python/sglang/srt/lora/backend/chunked_backend.py,
 *         class ChunkedSgmvLoRABackend
 *   [BB]  python/sglang/srt/lora/backend/base_backend.py,
 *         class BaseLoRABackend (shape contracts of every run_* call)
 *   [LM]  python/sglang/srt/lora/lora_manager.py,
 *         LoRAManager.prepare_lora_batch (slot ranks / scalings)
 *
 * Everything is plain fp64 per-token loops.  The only library primitive used
 * is qsort, on (key, index) pairs, which makes it a stable sort.  OpenMP only
 * splits the independent per-token loops across host cores.
 *
 * Readings of points the pages leave open (each one is listed in the design
 * notes of the repository as well):
 *   - slice j of A[w] is rows [j*r_w, (j+1)*r_w) and slice j of h[t] is
 *     columns [j*r_w, (j+1)*r_w) ("packed" stride, r_w = rank of the slot);
 *     B[w] uses columns [0, r_w).  [BB] run_lora_a_sgemm / run_qkv_lora shapes.
 *   - h columns at and beyond c*r_w are 0; a rank-0 token has h == 0 and
 *     leaves the output exactly equal to base.
 *   - sigma (the slot's scaling) is applied in the expand.
 *   - permutation[p] is the original token index at sorted position p.
 *   - embedding output columns k >= r_w are 0; an id outside [0, V) is an
 *     error (extra tokens are not supported by the chunked backend, [CB]
 *     run_lora_a_embedding).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> double.  A bf16 value is the top 16 bits of an IEEE
 * binary32 value, so the widening is exact. */
static double oracle_bf16_to_f64(uint16_t v)
{
    uint32_t u = ((uint32_t)v) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------- *
 * Chunk size.  [CB] MIN_CHUNK_SIZE and _determine_chunk_size_for_tokens:
 * a maximum at or below the floor gives the floor; otherwise 128 from 256
 * tokens, 32 from 64 tokens, else 16, capped by the maximum.
 * ------------------------------------------------------------------------- */
#define ORACLE_MIN_CHUNK_SIZE 16

int oracle_chunk_size(int num_tokens, int max_chunk_size)
{
    int chunk;
    if (max_chunk_size <= ORACLE_MIN_CHUNK_SIZE)
        return ORACLE_MIN_CHUNK_SIZE;
    if (num_tokens >= 256)
        chunk = 128;
    else if (num_tokens >= 64)
        chunk = 32;
    else
        chunk = 16;
    return max_chunk_size < chunk ? max_chunk_size : chunk;
}

/* [CB] init_cuda_graph_batch_info: segment and token capacity of the
 * preallocated batch-info buffers. */
void oracle_capacity(int max_bs, int num_tokens_per_bs, int *max_segments, int *max_tokens)
{
    *max_segments = ((num_tokens_per_bs + ORACLE_MIN_CHUNK_SIZE - 1) / ORACLE_MIN_CHUNK_SIZE) * max_bs;
    *max_tokens = max_bs * num_tokens_per_bs;
}

/* Per-token adapter slot: the request's slot repeated once per token of the
 * request ([CB] _get_permutation, repeat_interleave of the request slots by
 * the sequence lengths).  Returns the token count. */
int oracle_token_adapter(const int32_t *req_lens, const int32_t *req_adapter, int bs, int32_t *token_adapter)
{
    int t = 0;
    for (int i = 0; i < bs; ++i)
        for (int j = 0; j < req_lens[i]; ++j)
            token_adapter[t++] = req_adapter[i];
    return t;
}

typedef struct {
    int32_t key;
    int32_t index;
} oracle_pair;

static int oracle_pair_cmp(const void *a, const void *b)
{
    const oracle_pair *x = (const oracle_pair *)a, *y = (const oracle_pair *)b;
    if (x->key != y->key) return x->key < y->key ? -1 : 1;
    if (x->index != y->index) return x->index < y->index ? -1 : 1;
    return 0;
}

/* ------------------------------------------------------------------------- *
 * Batch info.  [CB] prepare_lora_batch, _get_permutation, _get_segments_info
 * and _build_req_seg_indptr.
 *
 *   key[t]        = slot of token t (repeat_interleave)
 *   permutation   = stable argsort(key)
 *   reordered     = key[permutation]
 *   segments      = for each run of equal consecutive keys of length n, in
 *                   order: ceil(n/chunk) segments with that key, all of
 *                   length chunk except the last, n - (ceil(n/chunk)-1)*chunk
 *   seg_indptr    = [0, cumsum(seg_lens)]
 *   CUDA-graph mode ([CB] prepare_lora_batch, use_cuda_graph branch): slots
 *   [num_segments, max_segments) of weight_indices are 0 and entries
 *   [num_segments+1, max_segments+1) of seg_indptr are the token total.
 *   req_seg_indptr = [0, cumsum(req_lens)]; req_weight_indices = req slots.
 *
 * Returns 0, or -1 when the segments exceed max_segments.
 * ------------------------------------------------------------------------- */
int oracle_build_batch_info(const int32_t *req_lens, const int32_t *req_adapter, int bs, int chunk,
                            int use_cuda_graph, int max_segments,
                            int32_t *permutation, int32_t *weights_reordered,
                            int32_t *weight_indices, int32_t *seg_indptr, int32_t *num_segments,
                            int32_t *req_seg_indptr, int32_t *req_weight_indices)
{
    int s = 0;
    for (int i = 0; i < bs; ++i) s += req_lens[i];

    int32_t *key = (int32_t *)malloc(sizeof(int32_t) * (size_t)(s > 0 ? s : 1));
    oracle_pair *pairs = (oracle_pair *)malloc(sizeof(oracle_pair) * (size_t)(s > 0 ? s : 1));
    oracle_token_adapter(req_lens, req_adapter, bs, key);

    for (int t = 0; t < s; ++t) {
        pairs[t].key = key[t];
        pairs[t].index = t;
    }
    qsort(pairs, (size_t)s, sizeof(oracle_pair), oracle_pair_cmp);
    for (int p = 0; p < s; ++p) {
        permutation[p] = pairs[p].index;
        weights_reordered[p] = key[pairs[p].index];
    }

    /* unique_consecutive over the reordered keys, then chunk each group. */
    int nseg = 0, rc = 0;
    int cum = 0;
    seg_indptr[0] = 0;
    int p = 0;
    while (p < s) {
        int q = p;
        while (q < s && weights_reordered[q] == weights_reordered[p]) ++q;
        int group_len = q - p;
        int num_segs = (group_len + chunk - 1) / chunk;
        for (int k = 0; k < num_segs; ++k) {
            int len = (k < num_segs - 1) ? chunk : group_len - (num_segs - 1) * chunk;
            if (nseg >= max_segments) { rc = -1; break; }
            weight_indices[nseg] = weights_reordered[p];
            cum += len;
            seg_indptr[nseg + 1] = cum;
            ++nseg;
        }
        if (rc) break;
        p = q;
    }
    *num_segments = rc ? 0 : nseg;
    if (!rc && use_cuda_graph) {
        for (int k = nseg; k < max_segments; ++k) {
            weight_indices[k] = 0;
            seg_indptr[k + 1] = s;
        }
    }
    if (req_seg_indptr) {
        req_seg_indptr[0] = 0;
        for (int i = 0; i < bs; ++i) req_seg_indptr[i + 1] = req_seg_indptr[i] + req_lens[i];
    }
    if (req_weight_indices)
        for (int i = 0; i < bs; ++i) req_weight_indices[i] = req_adapter[i];

    free(key);
    free(pairs);
    return rc;
}

/* ------------------------------------------------------------------------- *
 * Pruned lm_head batch info.  [CB] _prepare_lm_head_batch_info and
 * _build_lm_head_batch_info: only pruned_lens[i] tokens of request i reach
 * lm_head, kept in their original order (identity permutation);
 * merge_and_chunk_segments(weight_indices, pruned_lens, chunk_size) gives the
 * segments.  Its body is not on the pages; read from its call sites:
 *   1. walk the requests in order, skipping those without pruned tokens, and
 *      merge each request into the previous run when both use the same slot;
 *   2. cut every run into pieces of chunk tokens, the last one shorter.
 * Returns 0, or -1 when the segments exceed max_segments (then 0 segments).
 * ------------------------------------------------------------------------- */
int oracle_build_lm_head_batch_info(const int32_t *pruned_lens, const int32_t *req_adapter, int bs, int chunk,
                                    int use_cuda_graph, int max_segments, int32_t *permutation,
                                    int32_t *weight_indices, int32_t *seg_indptr, int32_t *num_segments)
{
    /* step 1: runs of consecutive non-empty requests on one slot */
    int32_t *run_slot = (int32_t *)malloc(sizeof(int32_t) * (size_t)(bs > 0 ? bs : 1));
    int32_t *run_len = (int32_t *)malloc(sizeof(int32_t) * (size_t)(bs > 0 ? bs : 1));
    int nruns = 0, s = 0;
    for (int i = 0; i < bs; ++i) {
        if (pruned_lens[i] == 0) continue;
        if (nruns > 0 && run_slot[nruns - 1] == req_adapter[i]) {
            run_len[nruns - 1] += pruned_lens[i];
        } else {
            run_slot[nruns] = req_adapter[i];
            run_len[nruns] = pruned_lens[i];
            ++nruns;
        }
        s += pruned_lens[i];
    }
    /* step 2: chunks of every run */
    int nseg = 0, rc = 0, cum = 0;
    seg_indptr[0] = 0;
    for (int k = 0; k < nruns && !rc; ++k) {
        int left = run_len[k];
        while (left > 0) {
            int len = left < chunk ? left : chunk;
            if (nseg >= max_segments) { rc = -1; break; }
            weight_indices[nseg] = run_slot[k];
            cum += len;
            seg_indptr[nseg + 1] = cum;
            ++nseg;
            left -= len;
        }
    }
    for (int t = 0; t < s; ++t) permutation[t] = t;
    *num_segments = rc ? 0 : nseg;
    if (!rc && use_cuda_graph) {
        for (int k = nseg; k < max_segments; ++k) {  /* padding: zero-length segments at the end */
            weight_indices[k] = 0;
            seg_indptr[k + 1] = cum;
        }
    }
    free(run_slot);
    free(run_len);
    return rc;
}

/* ------------------------------------------------------------------------- *
 * Shrink.  [BB] run_lora_a_sgemm: x (s, K), A (L, c*R, K) -> h (s, c*R), and
 * [CB] run_lora_a_sgemm / run_qkv_lora / run_gate_up_lora (num_slices = c).
 * For token t with slot w and rank r:
 *     h[t][j*r + k] = sum_i x[t][i] * A[w][j*r + k][i],  j < c, k < r
 * and every other column of h[t] is 0.
 * token_adapter[t] is the slot of token t; a slot outside [0, L) is skipped
 * and counted in the return value.
 * ------------------------------------------------------------------------- */
int oracle_shrink(const uint16_t *x, int64_t s, int64_t K, const uint16_t *A, int L, int c, int R,
                  const int32_t *token_adapter, const int32_t *ranks, double *h)
{
    int bad = 0;
    const int64_t cR = (int64_t)c * R;
#pragma omp parallel for schedule(dynamic, 8) reduction(+ : bad)
    for (int64_t t = 0; t < s; ++t) {
        double *ht = h + t * cR;
        for (int64_t n = 0; n < cR; ++n) ht[n] = 0.0;
        int w = token_adapter[t];
        if (w < 0 || w >= L) { bad += 1; continue; }
        int r = ranks[w];
        const uint16_t *xt = x + t * K;
        const uint16_t *Aw = A + (int64_t)w * cR * K;
        for (int j = 0; j < c; ++j) {
            for (int k = 0; k < r; ++k) {
                const uint16_t *arow = Aw + ((int64_t)j * r + k) * K;
                double acc = 0.0;
                for (int64_t i = 0; i < K; ++i)
                    acc += oracle_bf16_to_f64(xt[i]) * oracle_bf16_to_f64(arow[i]);
                ht[(int64_t)j * r + k] = acc;
            }
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------- *
 * Expand.  [BB] run_lora_b_sgemm: h (s, r), B (L, N, R) -> (s, N), and
 * [CB] run_lora_b_sgemm / run_qkv_lora / run_gate_up_lora (slice_offsets,
 * base_output).  For token t with slot w, rank r and scaling sigma, and for
 * every slice j and output column n in [off[j], off[j+1]):
 *     y[t][n] = base[t][n] + sigma * sum_{k<r} h[t][j*r + k] * B[w][n][k]
 * with base taken as 0 when base is NULL (base_output=None).  Columns outside
 * [off[0], off[c]) keep the base value (or 0).  h is fp64 with row stride ldh.
 * ------------------------------------------------------------------------- */
int oracle_expand(const double *h, int64_t ldh, int64_t s, const uint16_t *B, int64_t N, int L, int R,
                  const int32_t *off, int c, const int32_t *token_adapter, const int32_t *ranks,
                  const float *scalings, const uint16_t *base, double *y)
{
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 8) reduction(+ : bad)
    for (int64_t t = 0; t < s; ++t) {
        double *yt = y + t * N;
        for (int64_t n = 0; n < N; ++n)
            yt[n] = base ? oracle_bf16_to_f64(base[t * N + n]) : 0.0;
        int w = token_adapter[t];
        if (w < 0 || w >= L) { bad += 1; continue; }
        int r = ranks[w];
        double sigma = (double)scalings[w];
        const double *ht = h + t * ldh;
        const uint16_t *Bw = B + (int64_t)w * N * R;
        for (int j = 0; j < c; ++j) {
            for (int64_t n = off[j]; n < off[j + 1]; ++n) {
                double acc = 0.0;
                for (int k = 0; k < r; ++k)
                    acc += ht[(int64_t)j * r + k] * oracle_bf16_to_f64(Bw[n * R + k]);
                yt[n] += sigma * acc;
            }
        }
    }
    return bad;
}

/* Fused shrink then expand with the intermediate kept in fp64: per token,
 * y[t] = base[t] + sigma_w * B_w (A_w x[t]) slice by slice. */
int oracle_fused(const uint16_t *x, int64_t s, int64_t K, const uint16_t *A, const uint16_t *B, int64_t N,
                 int L, int R, const int32_t *off, int c, const int32_t *token_adapter,
                 const int32_t *ranks, const float *scalings, const uint16_t *base, double *y)
{
    const int64_t cR = (int64_t)c * R;
    double *h = (double *)malloc(sizeof(double) * (size_t)(s > 0 ? s * cR : 1));
    int bad = oracle_shrink(x, s, K, A, L, c, R, token_adapter, ranks, h);
    oracle_expand(h, cR, s, B, N, L, R, off, c, token_adapter, ranks, scalings, base, y);
    free(h);
    return bad;
}

/* ------------------------------------------------------------------------- *
 * Expand with tuple-form B.  [BB] run_qkv_lora: qkv_lora_b may be a tuple of
 * a q buffer (1, L, N_q, R) and a combined kv buffer (2, L, N_kv, R); [BB]
 * run_gate_up_lora: a tuple of two (L, N_out, R) buffers.  Either way slice j
 * of the output has a B of its own, Bs[j] of shape (L, off[j+1] - off[j], R),
 * whose row 0 is output column off[j]:
 *     y[t][n] = base[t][n] + sigma * sum_{k<r} h[t][j*r + k] * Bs[j][w][n - off[j]][k]
 * for n in [off[j], off[j+1]).  Everything else as oracle_expand.
 * ------------------------------------------------------------------------- */
int oracle_expand_sliced(const double *h, int64_t ldh, int64_t s, const uint16_t *const *Bs, int64_t N, int L,
                         int R, const int32_t *off, int c, const int32_t *token_adapter, const int32_t *ranks,
                         const float *scalings, const uint16_t *base, double *y)
{
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 8) reduction(+ : bad)
    for (int64_t t = 0; t < s; ++t) {
        double *yt = y + t * N;
        for (int64_t n = 0; n < N; ++n)
            yt[n] = base ? oracle_bf16_to_f64(base[t * N + n]) : 0.0;
        int w = token_adapter[t];
        if (w < 0 || w >= L) { bad += 1; continue; }
        int r = ranks[w];
        double sigma = (double)scalings[w];
        const double *ht = h + t * ldh;
        for (int j = 0; j < c; ++j) {
            const int64_t width = (int64_t)off[j + 1] - off[j];
            const uint16_t *Bw = Bs[j] + (int64_t)w * width * R;
            for (int64_t n = off[j]; n < off[j + 1]; ++n) {
                double acc = 0.0;
                for (int k = 0; k < r; ++k)
                    acc += oracle_bf16_to_f64(Bw[(n - off[j]) * R + k]) * ht[(int64_t)j * r + k];
                yt[n] += acc * sigma;
            }
        }
    }
    return bad;
}

/* Fused shrink then expand with tuple-form B, h in fp64. */
int oracle_fused_sliced(const uint16_t *x, int64_t s, int64_t K, const uint16_t *A, const uint16_t *const *Bs,
                        int64_t N, int L, int R, const int32_t *off, int c, const int32_t *token_adapter,
                        const int32_t *ranks, const float *scalings, const uint16_t *base, double *y)
{
    const int64_t cR = (int64_t)c * R;
    double *h = (double *)malloc(sizeof(double) * (size_t)(s > 0 ? s * cR : 1));
    int bad = oracle_shrink(x, s, K, A, L, c, R, token_adapter, ranks, h);
    oracle_expand_sliced(h, cR, s, Bs, N, L, R, off, c, token_adapter, ranks, scalings, base, y);
    free(h);
    return bad;
}

/* ------------------------------------------------------------------------- *
 * Embedding LoRA-A gather.  [BB] run_lora_a_embedding: input_ids (s,),
 * weights (L, R, V) -> (s, R); [CB] run_lora_a_embedding (no extra tokens).
 *     out[t][k] = A_emb[w][k][ids[t]]  for k < r_w,  0 for r_w <= k < R.
 * An id outside [0, V) or a slot outside [0, L) leaves the row 0 and is
 * counted in the return value.
 * ------------------------------------------------------------------------- */
int oracle_embedding(const int32_t *ids, int64_t s, const uint16_t *A_emb, int L, int R, int64_t V,
                     const int32_t *token_adapter, const int32_t *ranks, uint16_t *out)
{
    int bad = 0;
    for (int64_t t = 0; t < s; ++t) {
        uint16_t *ot = out + t * R;
        for (int k = 0; k < R; ++k) ot[k] = 0;
        int w = token_adapter[t];
        int64_t id = ids[t];
        if (w < 0 || w >= L || id < 0 || id >= V) { ++bad; continue; }
        int r = ranks[w];
        for (int k = 0; k < r && k < R; ++k)
            ot[k] = A_emb[((int64_t)w * R + k) * V + id];
    }
    return bad;
}

/* ------------------------------------------------------------------------- *
 * Embedding LoRA-A gather with extra tokens.  [BB] run_lora_a_embedding:
 * tokens with ids >= vocab_size are extra tokens, whose LoRA-A rows come from
 * extra_embeddings (L, num_extra, R):
 *     out[t][k] = A_emb[w][k][id]          for 0 <= id < V,
 *     out[t][k] = extra[w][id - V][k]      for V <= id < V + num_extra,
 * for k < r_w, and 0 for r_w <= k < R (the rank rule of oracle_embedding).
 * Any other id, or a slot outside [0, L), leaves the row 0 and is counted.
 * ------------------------------------------------------------------------- */
int oracle_embedding_extra(const int32_t *ids, int64_t s, const uint16_t *A_emb, int L, int R, int64_t V,
                           const uint16_t *extra, int64_t num_extra, const int32_t *token_adapter,
                           const int32_t *ranks, uint16_t *out)
{
    int bad = 0;
    for (int64_t t = 0; t < s; ++t) {
        uint16_t *ot = out + t * R;
        for (int k = 0; k < R; ++k) ot[k] = 0;
        int w = token_adapter[t];
        int64_t id = ids[t];
        if (w < 0 || w >= L || id < 0 || id >= V + num_extra) { ++bad; continue; }
        const int rr = ranks[w] < R ? ranks[w] : R;
        for (int k = 0; k < rr; ++k) {
            if (id < V) ot[k] = A_emb[((int64_t)w * R + k) * V + id];
            else ot[k] = extra[((int64_t)w * num_extra + (id - V)) * R + k];
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------- *
 * Extra-token embedding.  [BB] run_extra_token_embedding: output (s, D) is
 * modified in place with extra_embeddings (L, num_extra, D): the row of every
 * token with V <= id < V + num_extra becomes extra[w][id - V][:] (the base
 * vocabulary has no embedding for it); rows of ids below V are untouched.  An
 * id outside [0, V + num_extra), or a slot outside [0, L), leaves the row
 * untouched and is counted.
 * ------------------------------------------------------------------------- */
int oracle_extra_token_embedding(const int32_t *ids, int64_t s, uint16_t *output, int64_t D,
                                 const uint16_t *extra, int L, int64_t num_extra, int64_t V,
                                 const int32_t *token_adapter)
{
    int bad = 0;
    for (int64_t t = 0; t < s; ++t) {
        int w = token_adapter[t];
        int64_t id = ids[t];
        if (w < 0 || w >= L || id < 0 || id >= V + num_extra) { ++bad; continue; }
        if (id < V) continue;
        for (int64_t d = 0; d < D; ++d)
            output[t * D + d] = extra[((int64_t)w * num_extra + (id - V)) * D + d];
    }
    return bad;
}
