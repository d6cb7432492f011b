// C ABI of libcsgmv.so (declared in include/csgmv.h): argument checks on the
// host, then one kernel launch per call on the caller's stream.  Nothing here
// allocates, frees or synchronizes.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "csgmv_internal.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(CSGMV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace csgmv {
int set_error(int code, const char *msg) {
    g_last_error = msg;
    return code;
}
}  // namespace csgmv

namespace {

bool overlaps(const void *a, size_t abytes, const void *b, size_t bbytes) {
    if (!a || !b || abytes == 0 || bbytes == 0) return false;
    uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// The LoRA kernels take every control-flow decision from the batch info, so
// an output that overlaps it would be a contract violation the kernel cannot
// survive; refuse it up front.
bool overlaps_batch_info(const csgmv_batch_info *bi, const void *out, size_t bytes) {
    return overlaps(out, bytes, bi->seg_indptr, 4 * ((size_t)bi->max_segments + 1)) ||
           overlaps(out, bytes, bi->weight_indices, 4 * (size_t)bi->max_segments) ||
           overlaps(out, bytes, bi->permutation, 4 * (size_t)bi->max_tokens) ||
           overlaps(out, bytes, bi->lora_ranks, 4 * (size_t)bi->max_loras) ||
           overlaps(out, bytes, bi->scalings, 4 * (size_t)bi->max_loras) ||
           overlaps(out, bytes, bi->num_segments_dev, 4) || overlaps(out, bytes, bi->max_len_dev, 4) ||
           overlaps(out, bytes, bi->status, 4) ||
           (bi->tile_table &&
            overlaps(out, bytes, bi->tile_table, 4 * (size_t)csgmv_tile_table_ints(bi->max_loras, bi->max_tokens)));
}

int check_bi(const csgmv_batch_info *bi, bool built) {
    if (!bi) return fail(CSGMV_ERR_INVALID_ARG, "batch info is NULL");
    if (!bi->seg_indptr || !bi->weight_indices || !bi->permutation || !bi->lora_ranks || !bi->scalings ||
        !bi->num_segments_dev || !bi->max_len_dev || !bi->status)
        return fail(CSGMV_ERR_INVALID_ARG, "batch info has a NULL device buffer");
    if (bi->max_segments < 0 || bi->max_tokens < 0 || bi->max_loras <= 0 || bi->max_bs < 0 || bi->max_rank < 0)
        return fail(CSGMV_ERR_INVALID_ARG, "batch info capacities must be non-negative (max_loras > 0)");
    if (built && (bi->num_tokens < 0 || bi->num_tokens > bi->max_tokens))
        return fail(CSGMV_ERR_INVALID_ARG, "batch info was not built (num_tokens %d, max_tokens %d)",
                    bi->num_tokens, bi->max_tokens);
    return CSGMV_OK;
}

int check_offsets(const int32_t *off, int c, int64_t N, int max_slice_size) {
    if (!off) return fail(CSGMV_ERR_INVALID_ARG, "slice_offsets is NULL");
    if (c < 1 || c > csgmv::kMaxSlices) return fail(CSGMV_ERR_INVALID_ARG, "num_slices %d not in {1,2,3}", c);
    int widest = 0;
    for (int j = 0; j <= c; ++j) {
        if (off[j] < 0 || off[j] % 8 != 0)
            return fail(CSGMV_ERR_INVALID_ARG, "slice_offsets[%d] = %d must be a non-negative multiple of 8", j, off[j]);
        if (j > 0) {
            if (off[j] < off[j - 1])
                return fail(CSGMV_ERR_INVALID_ARG, "slice_offsets must be non-decreasing");
            widest = off[j] - off[j - 1] > widest ? off[j] - off[j - 1] : widest;
        }
    }
    if (off[c] > N) return fail(CSGMV_ERR_INVALID_ARG, "slice_offsets[%d] = %d exceeds N = %lld", c, off[c], (long long)N);
    if (max_slice_size < widest)
        return fail(CSGMV_ERR_INVALID_ARG, "max_slice_size %d is below the widest slice %d", max_slice_size, widest);
    return CSGMV_OK;
}

int check_rank(const csgmv_batch_info *bi) {
    if (bi->max_rank > csgmv::kMaxRank)
        return fail(CSGMV_ERR_UNSUPPORTED, "max_rank %d exceeds %d", bi->max_rank, csgmv::kMaxRank);
    if (bi->max_rank != 8 && bi->max_rank != 16 && bi->max_rank != 32 && bi->max_rank != 64)
        return fail(CSGMV_ERR_UNSUPPORTED, "max_rank %d must be 8, 16, 32 or 64 (B rows of 16..128 bytes, swizzled)",
                    bi->max_rank);
    return CSGMV_OK;
}

// B as one (max_loras, N, R) tensor: every slice reads rows w * N + n of it.
void single_b(csgmv::LoraParams &p) {
    for (int j = 0; j < csgmv::kMaxSlices; ++j) {
        p.Bs[j] = p.B;
        p.b_rows[j] = (int)p.N;
        p.b_row0[j] = j < p.c ? p.off[j] : 0;
    }
}

void fill_common(csgmv::LoraParams &p, const csgmv_batch_info *bi) {
    p.h_parts = 1;
    p.h_plane = 0;
    p.h_parts_dev = nullptr;
    p.seg_indptr = bi->seg_indptr;
    p.weight_indices = bi->weight_indices;
    p.permutation = bi->permutation;
    p.lora_ranks = bi->lora_ranks;
    p.scalings = bi->scalings;
    p.num_segments_dev = bi->num_segments_dev;
    p.max_len_dev = bi->max_len_dev;
    p.tile_table = bi->tile_table;
    p.status = bi->status;
    p.num_tokens = bi->num_tokens;
    p.max_loras = bi->max_loras;
    p.R = bi->max_rank;
}

// B as one (max_loras, N, R) tensor, or as one (max_loras, off[j+1] - off[j], R)
// tensor per slice (tuple form; slice offsets multiples of 64).
int check_b(const void *B, const void *const *B_slices, const int32_t *off, int c) {
    if (!B_slices) {
        if (!B) return fail(CSGMV_ERR_INVALID_ARG, "B is NULL");
        if (!aligned16(B)) return fail(CSGMV_ERR_INVALID_ARG, "B must be 16-byte aligned");
        return CSGMV_OK;
    }
    for (int j = 0; j < c; ++j) {
        if (!B_slices[j]) return fail(CSGMV_ERR_INVALID_ARG, "B_slices[%d] is NULL", j);
        if (!aligned16(B_slices[j])) return fail(CSGMV_ERR_INVALID_ARG, "B_slices[%d] must be 16-byte aligned", j);
    }
    for (int j = 0; j <= c; ++j)
        if (off[j] % 64)
            return fail(CSGMV_ERR_UNSUPPORTED, "with separate slice tensors, slice_offsets[%d] = %d must be a multiple of 64",
                        j, off[j]);
    return CSGMV_OK;
}

void set_b(csgmv::LoraParams &p, const void *const *B_slices) {
    if (!B_slices) {
        single_b(p);
        p.b_tuple = 0;
        return;
    }
    p.B = nullptr;
    for (int j = 0; j < csgmv::kMaxSlices; ++j) {
        const int jj = j < p.c ? j : 0;
        p.Bs[j] = static_cast<const uint16_t *>(B_slices[jj]);
        p.b_rows[j] = p.off[jj + 1] - p.off[jj];
        p.b_row0[j] = 0;
    }
    p.b_tuple = 1;
}

int expand_impl(const void *h, int h_dtype, int64_t ldh, const void *B, const void *const *B_slices, int64_t N,
                const int32_t *slice_offsets, int num_slices, int max_slice_size, void *out, int accumulate,
                const csgmv_batch_info *bi, csgmv_stream_t stream) {
    int rc = check_bi(bi, true);
    if (rc) return rc;
    if ((rc = check_rank(bi))) return rc;
    if ((rc = check_offsets(slice_offsets, num_slices, N, max_slice_size))) return rc;
    if (N <= 0 || N % 8 != 0 || N > INT32_MAX) return fail(CSGMV_ERR_INVALID_ARG, "N %lld must be a positive multiple of 8", (long long)N);
    if (h_dtype != CSGMV_DTYPE_BF16 && h_dtype != CSGMV_DTYPE_F32) return fail(CSGMV_ERR_INVALID_ARG, "bad h_dtype");
    if (ldh < (int64_t)num_slices * bi->max_rank) return fail(CSGMV_ERR_INVALID_ARG, "ldh below c*R");
    const int64_t s = bi->num_tokens;
    if (s == 0) return CSGMV_OK;
    if (!h || !out) return fail(CSGMV_ERR_INVALID_ARG, "NULL tensor");
    if (!aligned16(out)) return fail(CSGMV_ERR_INVALID_ARG, "out must be 16-byte aligned");
    if ((rc = check_b(B, B_slices, slice_offsets, num_slices))) return rc;
    if (overlaps_batch_info(bi, out, (size_t)s * N * 2)) return fail(CSGMV_ERR_INVALID_ARG, "out overlaps the batch info");
    csgmv::LoraParams p = {};
    fill_common(p, bi);
    p.B = static_cast<const uint16_t *>(B);
    p.y = static_cast<uint16_t *>(out);
    p.h = const_cast<void *>(h);
    p.h_f32 = h_dtype == CSGMV_DTYPE_F32;
    p.ldh = ldh;
    p.N = N;
    p.c = num_slices;
    for (int j = 0; j <= num_slices; ++j) p.off[j] = slice_offsets[j];
    set_b(p, B_slices);
    p.accumulate = accumulate ? 1 : 0;
    cudaError_t e = csgmv::launch_lora(csgmv::kModeExpand, p, *bi, reinterpret_cast<cudaStream_t>(stream), nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "csgmv_expand launch");
    return CSGMV_OK;
}

int qkv_impl(const void *x, int64_t K, const void *A, const void *B, const void *const *B_slices, int64_t N,
             const int32_t *slice_offsets, int num_slices, int max_slice_size, void *base_output, void *workspace,
             size_t workspace_bytes, const csgmv_batch_info *bi, csgmv_stream_t stream) {
    int rc = check_bi(bi, true);
    if (rc) return rc;
    if ((rc = check_rank(bi))) return rc;
    if ((rc = check_offsets(slice_offsets, num_slices, N, max_slice_size))) return rc;
    if (K <= 0 || K % 8 != 0 || K > INT32_MAX) return fail(CSGMV_ERR_INVALID_ARG, "K %lld must be a positive multiple of 8", (long long)K);
    if (N <= 0 || N % 8 != 0 || N > INT32_MAX) return fail(CSGMV_ERR_INVALID_ARG, "N %lld must be a positive multiple of 8", (long long)N);
    const int64_t s = bi->num_tokens;
    if (s == 0) return CSGMV_OK;
    if (!x || !A || !base_output) return fail(CSGMV_ERR_INVALID_ARG, "NULL tensor");
    if (!aligned16(x) || !aligned16(A) || !aligned16(base_output))
        return fail(CSGMV_ERR_INVALID_ARG, "x / A / base_output must be 16-byte aligned");
    if ((rc = check_b(B, B_slices, slice_offsets, num_slices))) return rc;
    if (overlaps_batch_info(bi, base_output, (size_t)s * N * 2))
        return fail(CSGMV_ERR_INVALID_ARG, "base_output overlaps the batch info");
    csgmv::LoraParams p = {};
    fill_common(p, bi);
    p.x = static_cast<const uint16_t *>(x);
    p.A = static_cast<const uint16_t *>(A);
    p.B = static_cast<const uint16_t *>(B);
    p.y = static_cast<uint16_t *>(base_output);
    p.K = K;
    p.N = N;
    p.c = num_slices;
    for (int j = 0; j <= num_slices; ++j) p.off[j] = slice_offsets[j];
    set_b(p, B_slices);
    p.accumulate = 1;
    const size_t hbytes = (size_t)s * num_slices * bi->max_rank * 4;
    const int path = csgmv::qkv_path(p, *bi, workspace ? workspace_bytes : 0);
    if (path != CSGMV_PATH_FUSED) {
        // the header and the planes of h the call may write (parts of K, hbytes each)
        const size_t ws_used =
            std::min(workspace_bytes, csgmv::kWsHeader + (size_t)csgmv::qkv_max_parts(p, *bi) * hbytes);
        if (!aligned16(workspace)) return fail(CSGMV_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
        if (overlaps_batch_info(bi, workspace, ws_used) ||
            overlaps(workspace, ws_used, base_output, (size_t)s * N * 2))
            return fail(CSGMV_ERR_INVALID_ARG, "workspace overlaps the batch info or base_output");
        // shrink into the workspace (fp32 h, columns [0, c*R), one plane per
        // part of K), then expand onto base_output
        csgmv::LoraParams ps = p;
        ps.B = nullptr;
        ps.y = nullptr;
        ps.N = 0;
        ps.h = workspace;
        ps.h_f32 = 1;
        ps.ldh = (int64_t)num_slices * bi->max_rank;
        ps.accumulate = 0;
        csgmv::LoraParams pe = p;
        pe.x = nullptr;
        pe.A = nullptr;
        pe.K = 0;
        pe.h = workspace;
        pe.h_f32 = 1;
        pe.ldh = ps.ldh;
        cudaError_t e =
            csgmv::launch_qkv_split(ps, pe, *bi, reinterpret_cast<cudaStream_t>(stream), workspace, ws_used, path);
        if (e != cudaSuccess) return cuda_fail(e, "csgmv_qkv shrink / expand launch");
        return CSGMV_OK;
    }
    cudaError_t e = csgmv::launch_lora(csgmv::kModeFused, p, *bi, reinterpret_cast<cudaStream_t>(stream), nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "csgmv_qkv launch");
    return CSGMV_OK;
}

int embedding_impl(const int32_t *input_ids, const void *A_emb, int transposed, int64_t vocab_size, int rank,
                   const void *extra_embeddings, int64_t num_extra_tokens, void *out, const csgmv_batch_info *bi,
                   csgmv_stream_t stream);

}  // namespace

extern "C" {

const char *csgmv_last_error(void) { return g_last_error.c_str(); }

const char *csgmv_version(void) { return "csgmv-gb300 0.1 (sm_103a)"; }

int csgmv_chunk_size(int num_tokens, int max_chunk_size) {
    if (max_chunk_size <= csgmv::kMinChunkSize) return csgmv::kMinChunkSize;
    int chunk = num_tokens >= 256 ? 128 : (num_tokens >= 64 ? 32 : 16);
    return max_chunk_size < chunk ? max_chunk_size : chunk;
}

int csgmv_batch_info_capacity(int max_bs, int num_tokens_per_bs, int32_t *max_segments, int32_t *max_tokens) {
    if (max_bs < 0 || num_tokens_per_bs < 0 || !max_segments || !max_tokens)
        return fail(CSGMV_ERR_INVALID_ARG, "capacity: negative size or NULL output");
    int64_t segs = (int64_t)((num_tokens_per_bs + csgmv::kMinChunkSize - 1) / csgmv::kMinChunkSize) * max_bs;
    int64_t toks = (int64_t)max_bs * num_tokens_per_bs;
    if (segs > INT32_MAX || toks > INT32_MAX) return fail(CSGMV_ERR_INVALID_ARG, "capacity overflows int32");
    *max_segments = (int32_t)segs;
    *max_tokens = (int32_t)toks;
    return CSGMV_OK;
}

int csgmv_build_batch_info(csgmv_batch_info *bi, const int32_t *req_lens, const int32_t *req_adapter, int bs,
                           int num_tokens, const int32_t *lora_ranks, const float *scalings, int num_loras,
                           int max_chunk_size, int chunk_size_override, int use_cuda_graph,
                           csgmv_stream_t stream) {
    int rc = check_bi(bi, false);
    if (rc) return rc;
    if (bs < 0 || num_tokens < 0 || num_loras < 0)
        return fail(CSGMV_ERR_INVALID_ARG, "negative bs / num_tokens / num_loras");
    if (bs > 0 && (!req_lens || !req_adapter))
        return fail(CSGMV_ERR_INVALID_ARG, "req_lens / req_adapter is NULL");
    if (num_loras > 0 && (!lora_ranks || !scalings))
        return fail(CSGMV_ERR_INVALID_ARG, "lora_ranks / scalings is NULL");
    if (bs > bi->max_bs) return fail(CSGMV_ERR_CAPACITY, "bs %d exceeds max_bs %d", bs, bi->max_bs);
    if (num_tokens > bi->max_tokens)
        return fail(CSGMV_ERR_CAPACITY, "num_tokens %d exceeds max_tokens %d", num_tokens, bi->max_tokens);
    if (num_loras > bi->max_loras)
        return fail(CSGMV_ERR_CAPACITY, "num_loras %d exceeds max_loras %d", num_loras, bi->max_loras);
    if (chunk_size_override < 0) return fail(CSGMV_ERR_INVALID_ARG, "negative chunk_size_override");
    if (csgmv::build_smem_bytes(bs, bi->max_loras) > 227 * 1024)
        return fail(CSGMV_ERR_UNSUPPORTED, "bs %d with max_loras %d exceeds the single-CTA builder", bs,
                    bi->max_loras);
    const int chunk = chunk_size_override > 0 ? chunk_size_override : csgmv_chunk_size(num_tokens, max_chunk_size);
    csgmv::BuildParams p;
    p.req_lens = req_lens;
    p.req_adapter = req_adapter;
    p.ranks_in = lora_ranks;
    p.scalings_in = scalings;
    p.bs = bs;
    p.num_tokens = num_tokens;
    p.num_loras = num_loras;
    p.chunk = chunk;
    p.use_graph = use_cuda_graph ? 1 : 0;
    cudaError_t e = csgmv::launch_build(p, *bi, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "csgmv_build_batch_info launch");
    bi->num_tokens = num_tokens;
    bi->chunk_size = chunk;
    bi->bs = bs;
    bi->num_loras = num_loras;
    bi->use_cuda_graph = p.use_graph;
    return CSGMV_OK;
}

int csgmv_build_lm_head_batch_info(csgmv_batch_info *bi, const int32_t *pruned_lens, const int32_t *req_adapter,
                                   int bs, int num_tokens, const int32_t *lora_ranks, const float *scalings,
                                   int num_loras, int max_chunk_size, int chunk_size_override, int use_cuda_graph,
                                   csgmv_stream_t stream) {
    int rc = check_bi(bi, false);
    if (rc) return rc;
    if (bs < 0 || num_tokens < 0 || num_loras < 0)
        return fail(CSGMV_ERR_INVALID_ARG, "negative bs / num_tokens / num_loras");
    if (bs > 0 && (!pruned_lens || !req_adapter))
        return fail(CSGMV_ERR_INVALID_ARG, "pruned_lens / req_adapter is NULL");
    if (num_loras > 0 && (!lora_ranks || !scalings))
        return fail(CSGMV_ERR_INVALID_ARG, "lora_ranks / scalings is NULL");
    if (bs > bi->max_bs) return fail(CSGMV_ERR_CAPACITY, "bs %d exceeds max_bs %d", bs, bi->max_bs);
    if (num_tokens > bi->max_tokens)
        return fail(CSGMV_ERR_CAPACITY, "num_tokens %d exceeds max_tokens %d", num_tokens, bi->max_tokens);
    if (num_loras > bi->max_loras)
        return fail(CSGMV_ERR_CAPACITY, "num_loras %d exceeds max_loras %d", num_loras, bi->max_loras);
    if (chunk_size_override < 0) return fail(CSGMV_ERR_INVALID_ARG, "negative chunk_size_override");
    if (csgmv::build_lm_head_smem_bytes(bs) > 227 * 1024)
        return fail(CSGMV_ERR_UNSUPPORTED, "bs %d exceeds the single-CTA builder", bs);
    const int chunk = chunk_size_override > 0 ? chunk_size_override : csgmv_chunk_size(num_tokens, max_chunk_size);
    csgmv::BuildParams p;
    p.req_lens = pruned_lens;
    p.req_adapter = req_adapter;
    p.ranks_in = lora_ranks;
    p.scalings_in = scalings;
    p.bs = bs;
    p.num_tokens = num_tokens;
    p.num_loras = num_loras;
    p.chunk = chunk;
    p.use_graph = use_cuda_graph ? 1 : 0;
    cudaError_t e = csgmv::launch_build_lm_head(p, *bi, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "csgmv_build_lm_head_batch_info launch");
    bi->num_tokens = num_tokens;
    bi->chunk_size = chunk;
    bi->bs = bs;
    bi->num_loras = num_loras;
    bi->use_cuda_graph = p.use_graph;
    return CSGMV_OK;
}

int csgmv_shrink(const void *x, int64_t s, int64_t K, const void *A, int num_slices, void *h, int h_dtype,
                 int64_t ldh, const csgmv_batch_info *bi, csgmv_stream_t stream) {
    int rc = check_bi(bi, true);
    if (rc) return rc;
    if ((rc = check_rank(bi))) return rc;
    if (num_slices < 1 || num_slices > csgmv::kMaxSlices)
        return fail(CSGMV_ERR_INVALID_ARG, "num_slices %d not in {1,2,3}", num_slices);
    if (s != bi->num_tokens) return fail(CSGMV_ERR_INVALID_ARG, "s %lld != batch num_tokens %d", (long long)s, bi->num_tokens);
    if (K <= 0 || K % 8 != 0 || K > INT32_MAX) return fail(CSGMV_ERR_INVALID_ARG, "K %lld must be a positive multiple of 8", (long long)K);
    if (h_dtype != CSGMV_DTYPE_BF16 && h_dtype != CSGMV_DTYPE_F32) return fail(CSGMV_ERR_INVALID_ARG, "bad h_dtype");
    if (ldh < (int64_t)num_slices * bi->max_rank) return fail(CSGMV_ERR_INVALID_ARG, "ldh below c*R");
    if (s == 0) return CSGMV_OK;
    if (!x || !A || !h) return fail(CSGMV_ERR_INVALID_ARG, "NULL tensor");
    if (!aligned16(x) || !aligned16(A)) return fail(CSGMV_ERR_INVALID_ARG, "x / A must be 16-byte aligned");
    const size_t hbytes = (size_t)s * ldh * (h_dtype == CSGMV_DTYPE_F32 ? 4 : 2);
    if (overlaps_batch_info(bi, h, hbytes)) return fail(CSGMV_ERR_INVALID_ARG, "h overlaps the batch info");
    csgmv::LoraParams p = {};
    fill_common(p, bi);
    p.x = static_cast<const uint16_t *>(x);
    p.A = static_cast<const uint16_t *>(A);
    p.h = h;
    p.h_f32 = h_dtype == CSGMV_DTYPE_F32;
    p.ldh = ldh;
    p.K = K;
    p.c = num_slices;
    p.N = 0;
    p.accumulate = 0;
    cudaError_t e = csgmv::launch_lora(csgmv::kModeShrink, p, *bi, reinterpret_cast<cudaStream_t>(stream), nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "csgmv_shrink launch");
    return CSGMV_OK;
}

int csgmv_expand(const void *h, int h_dtype, int64_t ldh, const void *B, int64_t N, const int32_t *slice_offsets,
                 int num_slices, int max_slice_size, void *out, int accumulate, const csgmv_batch_info *bi,
                 csgmv_stream_t stream) {
    return expand_impl(h, h_dtype, ldh, B, nullptr, N, slice_offsets, num_slices, max_slice_size, out, accumulate,
                       bi, stream);
}

int csgmv_expand_sliced(const void *h, int h_dtype, int64_t ldh, const void *const *B_slices, int64_t N,
                        const int32_t *slice_offsets, int num_slices, int max_slice_size, void *out, int accumulate,
                        const csgmv_batch_info *bi, csgmv_stream_t stream) {
    if (!B_slices) return fail(CSGMV_ERR_INVALID_ARG, "B_slices is NULL");
    return expand_impl(h, h_dtype, ldh, nullptr, B_slices, N, slice_offsets, num_slices, max_slice_size, out,
                       accumulate, bi, stream);
}

int64_t csgmv_tile_table_ints(int max_loras, int max_tokens) {
    if (max_loras < 0 || max_tokens < 0) return 0;
    return 4 * ((int64_t)max_loras + max_tokens / csgmv::kDecTM + 2);
}

int csgmv_qkv_path(const csgmv_batch_info *bi, int64_t K, int64_t N, const int32_t *slice_offsets, int num_slices,
                   size_t workspace_bytes) {
    int rc = check_bi(bi, true);
    if (rc) return rc;
    if ((rc = check_rank(bi))) return rc;
    int widest = 0;
    if (slice_offsets && num_slices >= 1 && num_slices <= csgmv::kMaxSlices)
        for (int j = 0; j < num_slices; ++j) widest = std::max(widest, slice_offsets[j + 1] - slice_offsets[j]);
    if ((rc = check_offsets(slice_offsets, num_slices, N, widest))) return rc;
    if (K <= 0 || K % 8 != 0 || K > INT32_MAX) return fail(CSGMV_ERR_INVALID_ARG, "K %lld must be a positive multiple of 8", (long long)K);
    if (N <= 0 || N % 8 != 0 || N > INT32_MAX) return fail(CSGMV_ERR_INVALID_ARG, "N %lld must be a positive multiple of 8", (long long)N);
    csgmv::LoraParams p = {};
    fill_common(p, bi);
    p.K = K;
    p.N = N;
    p.c = num_slices;
    for (int j = 0; j <= num_slices; ++j) p.off[j] = slice_offsets[j];
    p.accumulate = 1;
    return csgmv::qkv_path(p, *bi, workspace_bytes);
}

size_t csgmv_qkv_workspace_bytes(const csgmv_batch_info *bi, int num_slices) {
    if (!bi || bi->max_tokens < 0 || bi->max_rank < 0 || num_slices < 1 || num_slices > csgmv::kMaxSlices) return 0;
    // up to kMaxKParts planes of every token, or kDecMaxParts planes of a
    // batch small enough for the decode kernels
    const size_t T = (size_t)bi->max_tokens;
    const size_t rows = std::max((size_t)csgmv::kMaxKParts * T,
                                 (size_t)csgmv::kDecMaxParts * std::min(T, (size_t)csgmv::kDecPermCap));
    return csgmv::kWsHeader + rows * num_slices * bi->max_rank * 4;
}

int csgmv_qkv(const void *x, int64_t K, const void *A, const void *B, int64_t N, const int32_t *slice_offsets,
              int num_slices, int max_slice_size, void *base_output, void *workspace, size_t workspace_bytes,
              const csgmv_batch_info *bi, csgmv_stream_t stream) {
    return qkv_impl(x, K, A, B, nullptr, N, slice_offsets, num_slices, max_slice_size, base_output, workspace,
                    workspace_bytes, bi, stream);
}

int csgmv_qkv_sliced(const void *x, int64_t K, const void *A, const void *const *B_slices, int64_t N,
                     const int32_t *slice_offsets, int num_slices, int max_slice_size, void *base_output,
                     void *workspace, size_t workspace_bytes, const csgmv_batch_info *bi, csgmv_stream_t stream) {
    if (!B_slices) return fail(CSGMV_ERR_INVALID_ARG, "B_slices is NULL");
    return qkv_impl(x, K, A, nullptr, B_slices, N, slice_offsets, num_slices, max_slice_size, base_output, workspace,
                    workspace_bytes, bi, stream);
}

int embedding_lora_a(const int32_t *input_ids, const void *A_emb, int64_t vocab_size, int rank, void *out,
                     const csgmv_batch_info *bi, csgmv_stream_t stream) {
    return embedding_lora_a_extra(input_ids, A_emb, vocab_size, rank, nullptr, 0, out, bi, stream);
}

int embedding_lora_a_extra(const int32_t *input_ids, const void *A_emb, int64_t vocab_size, int rank,
                           const void *extra_embeddings, int64_t num_extra_tokens, void *out,
                           const csgmv_batch_info *bi, csgmv_stream_t stream) {
    return embedding_impl(input_ids, A_emb, 0, vocab_size, rank, extra_embeddings, num_extra_tokens, out, bi, stream);
}

int embedding_lora_a_transposed(const int32_t *input_ids, const void *A_emb_t, int64_t vocab_size, int rank,
                                const void *extra_embeddings, int64_t num_extra_tokens, void *out,
                                const csgmv_batch_info *bi, csgmv_stream_t stream) {
    return embedding_impl(input_ids, A_emb_t, 1, vocab_size, rank, extra_embeddings, num_extra_tokens, out, bi,
                          stream);
}

int csgmv_transpose_embedding(const void *A_emb, int64_t num_loras, int rank, int64_t vocab_size, void *A_emb_t,
                              csgmv_stream_t stream) {
    if (num_loras < 0 || rank < 1 || rank > 1024 || vocab_size <= 0)
        return fail(CSGMV_ERR_INVALID_ARG, "num_loras >= 0, 1 <= rank <= 1024 and vocab_size > 0 required");
    if (num_loras == 0) return CSGMV_OK;
    if (!A_emb || !A_emb_t) return fail(CSGMV_ERR_INVALID_ARG, "NULL tensor");
    const size_t bytes = (size_t)num_loras * rank * vocab_size * 2;
    if (overlaps(A_emb, bytes, A_emb_t, bytes)) return fail(CSGMV_ERR_INVALID_ARG, "A_emb_t overlaps A_emb");
    cudaError_t e = csgmv::launch_transpose_embedding(static_cast<const uint16_t *>(A_emb), num_loras, rank,
                                                      vocab_size, static_cast<uint16_t *>(A_emb_t),
                                                      reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "csgmv_transpose_embedding launch");
    return CSGMV_OK;
}

}  // extern "C"

namespace {

int embedding_impl(const int32_t *input_ids, const void *A_emb, int transposed, int64_t vocab_size, int rank,
                   const void *extra_embeddings, int64_t num_extra_tokens, void *out, const csgmv_batch_info *bi,
                   csgmv_stream_t stream) {
    int rc = check_bi(bi, true);
    if (rc) return rc;
    if (rank < 1 || rank > 1024) return fail(CSGMV_ERR_UNSUPPORTED, "rank %d not in [1, 1024]", rank);
    if (vocab_size <= 0) return fail(CSGMV_ERR_INVALID_ARG, "vocab_size must be positive");
    if (num_extra_tokens < 0) return fail(CSGMV_ERR_INVALID_ARG, "num_extra_tokens must be non-negative");
    if (num_extra_tokens > 0 && !extra_embeddings)
        return fail(CSGMV_ERR_INVALID_ARG, "extra_embeddings is NULL with num_extra_tokens > 0");
    if (vocab_size + num_extra_tokens > INT32_MAX)
        return fail(CSGMV_ERR_INVALID_ARG, "vocab_size + num_extra_tokens exceeds int32 token ids");
    const int64_t s = bi->num_tokens;
    if (s == 0) return CSGMV_OK;
    if (!input_ids || !A_emb || !out) return fail(CSGMV_ERR_INVALID_ARG, "NULL tensor");
    if (rank % 8 == 0 && !aligned16(out)) return fail(CSGMV_ERR_INVALID_ARG, "out must be 16-byte aligned");
    if (overlaps_batch_info(bi, out, (size_t)s * rank * 2)) return fail(CSGMV_ERR_INVALID_ARG, "out overlaps the batch info");
    csgmv::EmbeddingParams p;
    p.ids = input_ids;
    p.A = static_cast<const uint16_t *>(A_emb);
    p.transposed = transposed;
    p.extra = num_extra_tokens > 0 ? static_cast<const uint16_t *>(extra_embeddings) : nullptr;
    p.out = static_cast<uint16_t *>(out);
    p.V = vocab_size;
    p.E = num_extra_tokens > 0 ? num_extra_tokens : 0;
    p.R = rank;
    p.num_tokens = bi->num_tokens;
    p.max_loras = bi->max_loras;
    cudaError_t e = csgmv::launch_embedding(p, *bi, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "embedding_lora_a launch");
    return CSGMV_OK;
}

}  // namespace

extern "C" {

int extra_token_embedding(const int32_t *input_ids, void *output, int64_t embed_dim, const void *extra_embeddings,
                          int64_t num_extra_tokens, int64_t vocab_size, const csgmv_batch_info *bi,
                          csgmv_stream_t stream) {
    int rc = check_bi(bi, true);
    if (rc) return rc;
    if (embed_dim <= 0) return fail(CSGMV_ERR_INVALID_ARG, "embed_dim must be positive");
    if (vocab_size <= 0) return fail(CSGMV_ERR_INVALID_ARG, "vocab_size must be positive");
    if (num_extra_tokens < 0) return fail(CSGMV_ERR_INVALID_ARG, "num_extra_tokens must be non-negative");
    if (vocab_size + num_extra_tokens > INT32_MAX)
        return fail(CSGMV_ERR_INVALID_ARG, "vocab_size + num_extra_tokens exceeds int32 token ids");
    const int64_t s = bi->num_tokens;
    if (s == 0 || num_extra_tokens == 0) return CSGMV_OK;
    if (!input_ids || !output || !extra_embeddings) return fail(CSGMV_ERR_INVALID_ARG, "NULL tensor");
    if (embed_dim % 8 == 0 && (!aligned16(output) || !aligned16(extra_embeddings)))
        return fail(CSGMV_ERR_INVALID_ARG, "output / extra_embeddings must be 16-byte aligned");
    if (overlaps_batch_info(bi, output, (size_t)s * embed_dim * 2))
        return fail(CSGMV_ERR_INVALID_ARG, "output overlaps the batch info");
    csgmv::ExtraTokenParams p;
    p.ids = input_ids;
    p.extra = static_cast<const uint16_t *>(extra_embeddings);
    p.out = static_cast<uint16_t *>(output);
    p.V = vocab_size;
    p.E = num_extra_tokens;
    p.D = embed_dim;
    p.num_tokens = bi->num_tokens;
    p.max_loras = bi->max_loras;
    cudaError_t e = csgmv::launch_extra_token(p, *bi, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "extra_token_embedding launch");
    return CSGMV_OK;
}

}  // extern "C"
