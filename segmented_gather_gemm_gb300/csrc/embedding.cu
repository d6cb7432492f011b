// Embedding LoRA-A gather (sglang base_backend.py run_lora_a_embedding;
// chunked_backend.py run_lora_a_embedding, no extra-token embeddings):
//     out[t][k] = A_emb[w(t)][k][ids[t]]   k < r_w,   0 for r_w <= k < R.
// A_emb is (L, R, V), so the R values of one token are V elements apart: each
// is its own 32-byte sector and the gather is bound by sector count and
// latency, not by bytes.  Blocks own (segment, token-slice) pairs so the slot
// is read once per segment; each warp takes one token row at a time with one
// lane per rank column (so the output row is one coalesced store), and every
// lane issues its loads for four tokens before storing, to keep several
// sectors in flight per lane.
#include "csgmv_internal.h"

namespace csgmv {
namespace {

constexpr int kEmbThreads = 256;
constexpr int kTokPerIter = 8;  // token rows per block iteration (32 lanes each)
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kEmbThreads)
embedding_lora_a_kernel(EmbeddingParams p, const int32_t *__restrict__ seg_indptr,
                        const int32_t *__restrict__ weight_indices, const int32_t *__restrict__ permutation,
                        const int32_t *__restrict__ ranks, const int32_t *__restrict__ nseg_dev,
                        int32_t *status) {
    griddep_wait();  // the batch info may come from the kernel launched just before
    const int nseg = *nseg_dev;
    const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
    for (int seg = blockIdx.x; seg < nseg; seg += gridDim.x) {
        const int w = weight_indices[seg];
        const int p0 = max(seg_indptr[seg], 0), p1 = min(seg_indptr[seg + 1], p.num_tokens);
        int r = 0;
        const bool wok = w >= 0 && w < p.max_loras;
        if (!wok) {
            if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(status, CSGMV_STATUS_BAD_ADAPTER);
        } else {
            r = ranks[w];
            if (r < 0 || r > p.R) {
                if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(status, CSGMV_STATUS_BAD_RANK);
                r = 0;
            }
        }
        const uint16_t *Aw = p.A + (int64_t)(wok ? w : 0) * p.R * p.V;
        const int step = gridDim.y * kTokPerIter;
        for (int pb = p0 + blockIdx.y * kTokPerIter * kUnroll; pb < p1; pb += step * kUnroll) {
            int t[kUnroll];
            int64_t id[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                int pos = pb + u * kTokPerIter + ty;
                t[u] = -1;
                id[u] = -1;
                if (pos < p1) {
                    int tt = permutation[pos];
                    if (tt < 0 || tt >= p.num_tokens) {
                        if (tx == 0) atomicOr(status, CSGMV_STATUS_BAD_PERMUTATION);
                    } else {
                        t[u] = tt;
                        int64_t v = p.ids[tt];
                        if (v < 0 || v >= p.V) {
                            if (tx == 0) atomicOr(status, CSGMV_STATUS_BAD_TOKEN_ID);
                        } else {
                            id[u] = v;
                        }
                    }
                }
            }
            for (int k0 = 0; k0 < p.R; k0 += 32) {
                const int k = k0 + tx;
                uint16_t v[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u)
                    v[u] = (id[u] >= 0 && k < r) ? __ldg(Aw + (int64_t)k * p.V + id[u]) : (uint16_t)0;
#pragma unroll
                for (int u = 0; u < kUnroll; ++u)
                    if (t[u] >= 0 && k < p.R) p.out[(int64_t)t[u] * p.R + k] = v[u];
            }
        }
    }
}

}  // namespace

cudaError_t launch_embedding(const EmbeddingParams &p, const csgmv_batch_info &bi, cudaStream_t stream) {
    // One block row per segment slot, and enough token slices to cover a
    // segment of chunk_size tokens.
    const int chunk = bi.chunk_size > 0 ? bi.chunk_size : kMinChunkSize;
    int gy = (chunk + kTokPerIter * kUnroll - 1) / (kTokPerIter * kUnroll);
    gy = gy < 1 ? 1 : (gy > 64 ? 64 : gy);
    const int gx = bi.max_segments < 1 ? 1 : bi.max_segments;
    dim3 grid(gx, gy, 1);
    // programmatic dependent launch: the blocks start while the batch-info
    // builder before it finishes, and wait for it on the device
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kEmbThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, embedding_lora_a_kernel, p, (const int32_t *)bi.seg_indptr,
                                       (const int32_t *)bi.weight_indices, (const int32_t *)bi.permutation,
                                       (const int32_t *)bi.lora_ranks, (const int32_t *)bi.num_segments_dev,
                                       (int32_t *)bi.status);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace csgmv
