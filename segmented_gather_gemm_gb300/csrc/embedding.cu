// Embedding LoRA-A gather and extra-token embedding (sglang base_backend.py
// run_lora_a_embedding with optional extra_embeddings, and
// run_extra_token_embedding; chunked_backend.py run_lora_a_embedding):
//     out[t][k] = A_emb[w(t)][k][id]            0 <= id < V,      k < r_w
//     out[t][k] = extra[w(t)][id - V][k]        V <= id < V + E,  k < r_w
//     out[t][k] = 0                             r_w <= k < R
// A_emb is (L, R, V), so the R values of one token are V elements apart:
// each is its own 32-byte sector, and the gather is bound by the number of
// sectors in flight and by the chain of dependent loads (segment -> token ->
// id -> table), not by bytes.  Blocks own (segment, token-slice) pairs so the
// slot is read once per segment.
#include <algorithm>

#include "csgmv_internal.h"

namespace csgmv {
namespace {

// A_emb[w][k][id]: (L, R, V), or (L, V, R) for the transposed layout.
__device__ __forceinline__ uint16_t emb_at(const EmbeddingParams &p, int w, int k, int64_t id) {
    return p.transposed ? __ldg(p.A + ((int64_t)w * p.V + id) * p.R + k) : __ldg(p.A + ((int64_t)w * p.R + k) * p.V + id);
}

constexpr int kEmbThreads = 128;
constexpr int kEmbWarps = kEmbThreads / 32;

struct SegInfo {
    int w, r, p0, p1;
    bool ok;
};

// Segment seg of the batch info, its slot and rank (errors reported by one thread).
__device__ __forceinline__ SegInfo seg_info(int seg, int num_tokens, int max_loras, int R,
                                            const int32_t *seg_indptr, const int32_t *weight_indices,
                                            const int32_t *ranks, int32_t *status, bool report) {
    SegInfo g;
    g.w = weight_indices[seg];
    g.p0 = max(seg_indptr[seg], 0);
    g.p1 = min(seg_indptr[seg + 1], num_tokens);
    g.ok = g.w >= 0 && g.w < max_loras;
    g.r = 0;
    if (!g.ok) {
        if (report) atomicOr(status, CSGMV_STATUS_BAD_ADAPTER);
        return g;
    }
    g.r = ranks[g.w];
    if (g.r < 0 || g.r > R) {
        if (report) atomicOr(status, CSGMV_STATUS_BAD_RANK);
        g.r = 0;
    }
    return g;
}

// One token row per warp at a time, one lane per rank column (the output row
// is one coalesced store); every lane issues its loads for kUnroll tokens
// before it stores, to keep that many sectors in flight per lane.
constexpr int kTokPerIter = kEmbWarps;  // token rows per block iteration
constexpr int kUnroll = 8;

__global__ void __launch_bounds__(kEmbThreads)
embedding_lora_a_kernel(EmbeddingParams p, const int32_t *__restrict__ seg_indptr,
                        const int32_t *__restrict__ weight_indices, const int32_t *__restrict__ permutation,
                        const int32_t *__restrict__ ranks, const int32_t *__restrict__ nseg_dev, int32_t *status) {
    griddep_wait();  // the batch info may come from the kernel launched just before
    const int nseg = *nseg_dev;
    const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
    for (int seg = blockIdx.x; seg < nseg; seg += gridDim.x) {
        const SegInfo g = seg_info(seg, p.num_tokens, p.max_loras, p.R, seg_indptr, weight_indices, ranks, status,
                                   threadIdx.x == 0 && blockIdx.y == 0);
        const uint16_t *Ew = p.extra ? p.extra + (int64_t)(g.ok ? g.w : 0) * p.E * p.R : nullptr;
        const int step = gridDim.y * kTokPerIter;
        for (int pb = g.p0 + blockIdx.y * kTokPerIter * kUnroll; pb < g.p1; pb += step * kUnroll) {
            int t[kUnroll];
            int64_t id[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int pos = pb + u * kTokPerIter + ty;
                t[u] = -1;
                id[u] = -1;
                if (pos < g.p1) {
                    const int tt = permutation[pos];
                    if (tt < 0 || tt >= p.num_tokens) {
                        if (tx == 0) atomicOr(status, CSGMV_STATUS_BAD_PERMUTATION);
                    } else {
                        t[u] = tt;
                        const int64_t v = p.ids[tt];
                        if (v < 0 || v >= p.V + p.E) {
                            if (tx == 0) atomicOr(status, CSGMV_STATUS_BAD_TOKEN_ID);
                        } else if (g.ok) {
                            id[u] = v;
                        }
                    }
                }
            }
            for (int k0 = 0; k0 < p.R; k0 += 32) {
                const int k = k0 + tx;
                uint16_t v[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    v[u] = 0;
                    if (id[u] >= 0 && k < g.r)
                        v[u] = id[u] < p.V ? emb_at(p, g.ok ? g.w : 0, k, id[u]) : __ldg(Ew + (id[u] - p.V) * p.R + k);
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u)
                    if (t[u] >= 0 && k < p.R) p.out[(int64_t)t[u] * p.R + k] = v[u];
            }
        }
    }
}

// Token-major gather for batch infos with per-request fields (every batch
// info from either builder, when the caller allocated those fields): the
// token's slot is its request's, so a block of kTokPerBlock consecutive
// tokens loads, in one round, their ids together with the request starts,
// request slots and slot ranks; lanes 0..7 of each warp find their token's
// request by binary search in shared memory, and then every lane gathers its
// rank column of the warp's eight tokens.  Two dependent rounds of memory
// (ids, then the table) instead of five (segments, token, id, table).
constexpr int kTokThreads = 256;
constexpr int kTokWarps = kTokThreads / 32;
constexpr int kTokPerWarp = 8;
constexpr int kTokPerBlock = kTokWarps * kTokPerWarp;

__global__ void __launch_bounds__(kTokThreads)
embedding_token_kernel(EmbeddingParams p, const int32_t *__restrict__ req_start_g, const int32_t *__restrict__ req_slot_g,
                       int bs, const int32_t *__restrict__ ranks, int nl, const int32_t *__restrict__ nseg_dev,
                       int32_t *status) {
    extern __shared__ int sm_tok[];
    int *st = sm_tok;        // [bs + 1] first token of request i
    int *sl = st + bs + 1;   // [bs] slot of request i
    int *rk = sl + bs;       // [nl] slot ranks
    griddep_wait();  // the batch info may come from the kernel launched just before
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i <= bs; i += kTokThreads) {
        st[i] = req_start_g[i];
        if (i < bs) sl[i] = req_slot_g[i];
    }
    for (int a = tid; a < nl; a += kTokThreads) rk[a] = ranks[a];
    const int nseg = *nseg_dev;
    const int t0 = blockIdx.x * kTokPerBlock + warp * kTokPerWarp;
    // lane u < 8 owns token t0 + u: its id, then its slot and rank
    const int tu = t0 + lane;
    int64_t my_id = -1;
    if (lane < kTokPerWarp && tu < p.num_tokens) my_id = p.ids[tu];
    __syncthreads();
    if (nseg <= 0) return;  // the build failed (or the batch is empty): nothing is written, as in the segment kernel
    int my_w = -1, my_r = 0;
    if (lane < kTokPerWarp && tu < p.num_tokens) {
        int lo = 0, hi = bs;  // last request with start <= tu
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (st[mid] <= tu) lo = mid; else hi = mid;
        }
        const int w = sl[lo];
        if (w < 0 || w >= p.max_loras || w >= nl) {
            atomicOr(status, CSGMV_STATUS_BAD_ADAPTER);
        } else {
            const int r = rk[w];
            if (r < 0 || r > p.R) atomicOr(status, CSGMV_STATUS_BAD_RANK);
            else { my_w = w; my_r = r; }
        }
        if (my_id < 0 || my_id >= p.V + p.E) {
            atomicOr(status, CSGMV_STATUS_BAD_TOKEN_ID);
            my_id = -1;
        }
        if (my_w < 0) my_id = -1;
    }
    int64_t id[kTokPerWarp];
    int w[kTokPerWarp], r[kTokPerWarp];
#pragma unroll
    for (int u = 0; u < kTokPerWarp; ++u) {
        id[u] = __shfl_sync(0xffffffffu, my_id, u);
        w[u] = __shfl_sync(0xffffffffu, my_w, u);
        r[u] = __shfl_sync(0xffffffffu, my_r, u);
    }
    for (int k0 = 0; k0 < p.R; k0 += 32) {
        const int k = k0 + lane;
        uint16_t v[kTokPerWarp];
#pragma unroll
        for (int u = 0; u < kTokPerWarp; ++u) {
            v[u] = 0;
            if (id[u] >= 0 && k < r[u])
                v[u] = id[u] < p.V ? emb_at(p, w[u], k, id[u])
                                   : __ldg(p.extra + ((int64_t)w[u] * p.E + (id[u] - p.V)) * p.R + k);
        }
#pragma unroll
        for (int u = 0; u < kTokPerWarp; ++u)
            if (t0 + u < p.num_tokens && k < p.R) p.out[(int64_t)(t0 + u) * p.R + k] = v[u];
    }
}

constexpr int kTokReqCap = 4096;  // requests whose table fits the token-major kernel's shared memory
constexpr int kTokLoraCap = 4096;

// Rows of extra tokens of an (s, D) output become extra[w][id - V][:].  Each
// lane checks one token of the warp's slice; the warp then copies the rows of
// the lanes that hold an extra token, one row at a time, 16 bytes per lane.
__global__ void __launch_bounds__(kEmbThreads)
extra_token_kernel(ExtraTokenParams p, const int32_t *__restrict__ seg_indptr,
                   const int32_t *__restrict__ weight_indices, const int32_t *__restrict__ permutation,
                   const int32_t *__restrict__ nseg_dev, int32_t *status, int spp) {
    griddep_wait();
    const int nseg = *nseg_dev;
    const int lane = threadIdx.x & 31;
    const int64_t nitems = (int64_t)max(nseg, 0) * spp;
    const int64_t wstride = (int64_t)gridDim.x * kEmbWarps;
    const bool vec = (p.D & 7) == 0;
    for (int64_t it = (int64_t)blockIdx.x * kEmbWarps + (threadIdx.x >> 5); it < nitems; it += wstride) {
        const int seg = (int)(it / spp), sl = (int)(it % spp);
        const int w = weight_indices[seg];
        const int p0 = max(seg_indptr[seg], 0), p1 = min(seg_indptr[seg + 1], p.num_tokens);
        if (p0 + 32 * sl >= p1) continue;
        const bool wok = w >= 0 && w < p.max_loras;
        if (!wok && sl == 0 && lane == 0) atomicOr(status, CSGMV_STATUS_BAD_ADAPTER);
        const int pos = p0 + 32 * sl + lane;
        int t = -1;
        int64_t e = -1;
        if (pos < p1) {
            const int tt = permutation[pos];
            if (tt < 0 || tt >= p.num_tokens) {
                atomicOr(status, CSGMV_STATUS_BAD_PERMUTATION);
            } else {
                const int64_t v = p.ids[tt];
                if (v < 0 || v >= p.V + p.E) atomicOr(status, CSGMV_STATUS_BAD_TOKEN_ID);
                else if (v >= p.V && wok) { t = tt; e = v - p.V; }
            }
        }
        uint32_t todo = __ballot_sync(0xffffffffu, t >= 0);
        while (todo) {
            const int src = __ffs(todo) - 1;
            todo &= todo - 1;
            const int tt = __shfl_sync(0xffffffffu, t, src);
            const int64_t ee = __shfl_sync(0xffffffffu, e, src);
            const uint16_t *from = p.extra + ((int64_t)w * p.E + ee) * p.D;
            uint16_t *to = p.out + (int64_t)tt * p.D;
            if (vec) {
                for (int64_t d = 8 * lane; d < p.D; d += 256)
                    *reinterpret_cast<uint4 *>(to + d) = __ldg(reinterpret_cast<const uint4 *>(from + d));
            } else {
                for (int64_t d = lane; d < p.D; d += 32) to[d] = __ldg(from + d);
            }
        }
    }
}

// out[w][v][k] = A[w][k][v]: 32 x 32 tiles through shared memory (the +1
// column keeps the transposed reads free of bank conflicts); grid (V / 32,
// R / 32, L) rounded up.
__global__ void __launch_bounds__(256) transpose_embedding_kernel(const uint16_t *__restrict__ A, int R, int64_t V,
                                                                  uint16_t *__restrict__ out) {
    __shared__ uint16_t tile[32][33];
    const int64_t v0 = (int64_t)blockIdx.x * 32;
    const int k0 = blockIdx.y * 32;
    const int64_t w = blockIdx.z;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 rows of 32
    for (int i = ty; i < 32; i += 8) {
        const int k = k0 + i;
        const int64_t v = v0 + tx;
        if (k < R && v < V) tile[i][tx] = A[(w * R + k) * V + v];
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int64_t v = v0 + i;
        const int k = k0 + tx;
        if (k < R && v < V) out[(w * V + v) * R + k] = tile[tx][i];
    }
}

// Grid for warps walking (segment, 32-token slice) items: enough blocks for
// the largest batch the batch info holds, at most eight per SM.
int item_grid(const csgmv_batch_info &bi, int spp) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t items = (int64_t)std::max(bi.max_segments, 1) * spp;
    const int64_t blocks = (items + kEmbWarps - 1) / kEmbWarps;
    return (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)sms * 8));
}

cudaLaunchConfig_t item_config(const csgmv_batch_info &bi, int spp, cudaStream_t stream, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(item_grid(bi, spp), 1, 1);
    cfg.blockDim = dim3(kEmbThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    // programmatic dependent launch: the blocks start while the batch-info
    // builder before them finishes, and wait for it on the device
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

}  // namespace

cudaError_t launch_embedding(const EmbeddingParams &p, const csgmv_batch_info &bi, cudaStream_t stream) {
    if (bi.req_seg_indptr && bi.req_weight_indices && bi.bs >= 1 && bi.bs <= kTokReqCap &&
        bi.max_loras <= kTokLoraCap && p.num_tokens > 0) {
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = item_config(bi, 1, stream, attr);
        cfg.gridDim = dim3((p.num_tokens + kTokPerBlock - 1) / kTokPerBlock, 1, 1);
        cfg.blockDim = dim3(kTokThreads, 1, 1);
        cfg.dynamicSmemBytes = sizeof(int) * (2 * (size_t)bi.bs + 1 + (size_t)bi.max_loras);
        cudaError_t e = cudaLaunchKernelEx(&cfg, embedding_token_kernel, p, (const int32_t *)bi.req_seg_indptr,
                                           (const int32_t *)bi.req_weight_indices, (int)bi.bs,
                                           (const int32_t *)bi.lora_ranks, (int)bi.max_loras,
                                           (const int32_t *)bi.num_segments_dev, (int32_t *)bi.status);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    // One block row per segment slot, and enough token slices to cover a
    // segment of chunk_size tokens.
    const int chunk = bi.chunk_size > 0 ? bi.chunk_size : kMinChunkSize;
    int gy = (chunk + kTokPerIter * kUnroll - 1) / (kTokPerIter * kUnroll);
    gy = gy < 1 ? 1 : (gy > 64 ? 64 : gy);
    const int gx = bi.max_segments < 1 ? 1 : bi.max_segments;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = item_config(bi, 1, stream, attr);
    cfg.gridDim = dim3(gx, gy, 1);
    cudaError_t e = cudaLaunchKernelEx(&cfg, embedding_lora_a_kernel, p, (const int32_t *)bi.seg_indptr,
                                       (const int32_t *)bi.weight_indices, (const int32_t *)bi.permutation,
                                       (const int32_t *)bi.lora_ranks, (const int32_t *)bi.num_segments_dev,
                                       (int32_t *)bi.status);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_transpose_embedding(const uint16_t *A, int64_t L, int R, int64_t V, uint16_t *out,
                                       cudaStream_t stream) {
    if (L <= 0 || R <= 0 || V <= 0) return cudaSuccess;
    const dim3 grid((unsigned)((V + 31) / 32), (unsigned)((R + 31) / 32), (unsigned)L);
    transpose_embedding_kernel<<<grid, 256, 0, stream>>>(A, R, V, out);
    return cudaGetLastError();
}

cudaError_t launch_extra_token(const ExtraTokenParams &p, const csgmv_batch_info &bi, cudaStream_t stream) {
    const int chunk = bi.chunk_size > 0 ? bi.chunk_size : kMinChunkSize;
    const int spp = (chunk + 31) / 32;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = item_config(bi, spp, stream, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, extra_token_kernel, p, (const int32_t *)bi.seg_indptr,
                                       (const int32_t *)bi.weight_indices, (const int32_t *)bi.permutation,
                                       (const int32_t *)bi.num_segments_dev, (int32_t *)bi.status, spp);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace csgmv
