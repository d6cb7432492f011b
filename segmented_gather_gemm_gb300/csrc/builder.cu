// Device batch-info builder: sglang chunked_backend.py prepare_lora_batch,
// _get_permutation (stable sort of tokens by slot) and _get_segments_info
// (ceil(n / chunk) segments per slot run), plus _build_req_seg_indptr and the
// CUDA-graph padding of the prepare_lora_batch use_cuda_graph branch.
//
// One CTA of 1024 threads does the whole batch, so the call is one launch,
// needs no global scratch and can sit inside a CUDA graph.  The stable sort is
// a counting sort over slots at request granularity: a request's tokens are
// contiguous in token order and stay contiguous in sorted order, so each
// request only needs its destination offset
//     dest[i] = (tokens of slots < a_i) + (tokens of earlier requests on a_i).
#include <mutex>
#include <set>
#include <utility>

#include "csgmv_internal.h"

namespace csgmv {
namespace {

constexpr int kBuildThreads = 1024;
constexpr int kWarps = kBuildThreads / 32;

// Exclusive block-wide scan of v; returns the prefix and writes the block
// total to *total.  `warp_sums` is kWarps ints of shared memory.
__device__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    int prefix = (warp > 0 ? warp_sums[warp - 1] : 0) + inc - v;
    *total = warp_sums[kWarps - 1];
    __syncthreads();
    return prefix;
}

// Exclusive block-wide scans of three values at once (one set of barriers
// for all three); block totals in t[0..2].  `ws` is 3 * kWarps ints.
__device__ void block_exclusive_scan3(const int (&v)[3], int (&pre)[3], int (&t)[3], int *ws) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc[3] = {v[0], v[1], v[2]};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int c = 0; c < 3; ++c) {
            const int n = __shfl_up_sync(0xffffffffu, inc[c], o);
            if (lane >= o) inc[c] += n;
        }
    }
    if (lane == 31)
#pragma unroll
        for (int c = 0; c < 3; ++c) ws[c * kWarps + warp] = inc[c];
    __syncthreads();
    if (warp < 3) {
        int w = ws[warp * kWarps + lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        ws[warp * kWarps + lane] = w;
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 3; ++c) {
        pre[c] = (warp > 0 ? ws[c * kWarps + warp - 1] : 0) + inc[c] - v[c];
        t[c] = ws[c * kWarps + kWarps - 1];
    }
    __syncthreads();
}

// For this lane: the sum of l over the lanes below it that carry the same
// key, and (last) whether no lane above it does.  Lanes with equal keys are
// found with one match; their lengths are read from `lens` (32 ints of
// shared memory for this warp), so the cost follows the group size rather
// than the warp width.  Every lane of the warp calls it.
__device__ __forceinline__ int same_key_prefix(int key, int l, int *lens, bool &last) {
    const int lane = threadIdx.x & 31;
    lens[lane] = l;
    __syncwarp();
    const unsigned m = __match_any_sync(0xffffffffu, key);
    const unsigned above = lane == 31 ? 0u : (0xffffffffu << (lane + 1));
    last = (m & above) == 0u;
    unsigned below = m & ((1u << lane) - 1u);
    int pre = 0;
    while (below) {
        pre += lens[__ffs(below) - 1];
        below &= below - 1u;
    }
    __syncwarp();
    return pre;
}

// Largest i in [0, n) with a[i] <= key (a non-decreasing, a[0] <= key).
__device__ int last_not_greater(const int *a, int n, int key) {
    int lo = 0, hi = n;  // answer in [lo, hi)
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (a[mid] <= key) lo = mid; else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(kBuildThreads, 1)
build_batch_info_kernel(BuildParams p, csgmv_batch_info bi) {
    extern __shared__ int sm[];
    // The LoRA kernel that consumes this batch info may start launching now
    // (programmatic dependent launch); it waits for this kernel to finish
    // before it reads anything.
    griddep_launch_dependents();
    const int L = bi.max_loras;
    int *cnt = sm;                      // [L]   tokens per slot
    int *tokbase = cnt + L;             // [L]   first sorted position of slot a
    int *segbase = tokbase + L;         // [L+1] first segment of slot a
    int *run = segbase + L + 1;         // [L]   running sorted position of slot a
    int *req_start = run + L;           // [bs+1] first token of request i
    int *req_dest = req_start + p.bs + 1;  // [bs] first sorted position of request i
    int *warp_sums = req_dest + p.bs;   // [32]
    int *flags = warp_sums + kWarps;    // [0] error bits, [1] nseg

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int chunk = p.chunk;
    int *wsum = flags + 2;  // [kWarps][L] per-warp token totals of each slot
    int *tilebase = wsum + kWarps * L;  // [L] first decode tile of slot a
    int *ws3 = tilebase + L;            // [3][kWarps] scan scratch
    int *lens_w = ws3 + 3 * kWarps + 32 * warp;  // [kWarps][32] request lengths of each warp
    // Up to 1024 requests (one per thread) take one pass: each thread loads its
    // request once and keeps it in registers for the counts, the offsets and
    // its destination.
    const bool one_tile = p.bs <= kBuildThreads;
    int my_a = -1, my_l = 0;
    if (one_tile && tid < p.bs) {
        my_a = p.req_adapter[tid];
        my_l = p.req_lens[tid];
    }
    if (tid == 0) { flags[0] = 0; flags[1] = 0; }
    for (int a = tid; a < L; a += kBuildThreads) cnt[a] = 0;
    if (one_tile)
        for (int x = tid; x < kWarps * L; x += kBuildThreads) wsum[x] = 0;
    __syncthreads();

    // Slot table (lora_manager.py prepare_lora_batch: lora_ranks / scalings per slot).
    for (int a = tid; a < L; a += kBuildThreads) {
        int r = 0;
        float sc = 0.f;
        if (a < p.num_loras) {
            r = p.ranks_in[a];
            sc = p.scalings_in[a];
            if (r < 0 || r > bi.max_rank) { atomicOr(&flags[0], CSGMV_STATUS_BAD_RANK); r = 0; }
        }
        bi.lora_ranks[a] = r;
        bi.scalings[a] = sc;
    }

    // Per-slot token counts and validation.
    int my_pre = 0;  // one pass: tokens of earlier requests of this warp on the same slot
    if (one_tile) {
        const bool valid = tid < p.bs;
        if (valid) {
            if (my_a < 0 || my_a >= p.num_loras) atomicOr(&flags[0], CSGMV_STATUS_BAD_ADAPTER);
            else if (my_l < 0) atomicOr(&flags[0], CSGMV_STATUS_BAD_LENS);
            else atomicAdd(&cnt[my_a], my_l);
        }
        bool last;
        my_pre = same_key_prefix(my_a, my_l, lens_w, last);
        if (valid && last && my_a >= 0 && my_a < L) wsum[warp * L + my_a] = my_pre + my_l;
    } else {
        for (int i = tid; i < p.bs; i += kBuildThreads) {
            int a = p.req_adapter[i], l = p.req_lens[i];
            if (a < 0 || a >= p.num_loras) atomicOr(&flags[0], CSGMV_STATUS_BAD_ADAPTER);
            else if (l < 0) atomicOr(&flags[0], CSGMV_STATUS_BAD_LENS);
            else atomicAdd(&cnt[a], l);
        }
    }

    // req_start = [0, cumsum(lens)] (chunked_backend.py _build_req_seg_indptr).
    int carry = 0;
    if (one_tile) {
        int tot;
        const int pre = block_exclusive_scan(tid < p.bs ? max(my_l, 0) : 0, warp_sums, &tot);
        if (tid < p.bs) req_start[tid] = pre;
        carry = tot;
    } else {
        for (int i0 = 0; i0 < p.bs; i0 += kBuildThreads) {
            int i = i0 + tid;
            int l = (i < p.bs) ? max(p.req_lens[i], 0) : 0;
            int tot;
            int pre = block_exclusive_scan(l, warp_sums, &tot);
            if (i < p.bs) req_start[i] = carry + pre;
            carry += tot;
        }
    }
    if (tid == 0) {
        req_start[p.bs] = carry;
        if (carry != p.num_tokens) atomicOr(&flags[0], CSGMV_STATUS_BAD_LENS);
    }
    __syncthreads();

    // Sorted-order base of each slot, its first segment and its first decode
    // tile (csgmv_batch_info.tile_table: ceil(n / kDecTM) tiles per slot).
    int tcarry = 0, scarry = 0, dcarry = 0;
    for (int a0 = 0; a0 < L; a0 += kBuildThreads) {
        int a = a0 + tid;
        const int n = (a < L) ? cnt[a] : 0;
        const int v[3] = {n, (n + chunk - 1) / chunk, (n + kDecTM - 1) / kDecTM};
        int pre[3], tot[3];
        block_exclusive_scan3(v, pre, tot, ws3);
        if (a < L) {
            tokbase[a] = tcarry + pre[0];
            run[a] = tcarry + pre[0];
            segbase[a] = scarry + pre[1];
            tilebase[a] = dcarry + pre[2];
        }
        tcarry += tot[0];
        scarry += tot[1];
        dcarry += tot[2];
    }
    if (tid == 0) {
        segbase[L] = scarry;
        flags[1] = scarry;
        if (scarry > bi.max_segments) atomicOr(&flags[0], CSGMV_STATUS_CAPACITY);
    }
    __syncthreads();

    const int err = flags[0];
    const int nseg = err ? 0 : flags[1];
    if (err) {
        if (tid == 0) {
            *bi.num_segments_dev = 0;
            *bi.max_len_dev = chunk;
            bi.seg_indptr[0] = 0;
            if (bi.tile_table) bi.tile_table[0] = 0;
            *bi.status = err;
        }
        return;
    }

    // Destination of every request: stable within a slot, so earlier requests
    // on the same slot come first.  Per 1024-request tile: lanes of a warp
    // with the same slot add up their predecessors' lengths, the last such
    // lane posts the warp's total for the slot, and one warp per slot scans
    // the warp totals into running offsets.
    auto slot_scan = [&]() {
        for (int b = warp; b < L; b += kWarps) {  // one warp per slot: scan over the 32 warps
            const int v = wsum[lane * L + b];
            int inc = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += n;
            }
            const int base = run[b];
            wsum[lane * L + b] = base + inc - v;
            __syncwarp();
            if (lane == 31) run[b] = base + inc;
        }
    };
    if (one_tile) {
        slot_scan();  // the warp totals were posted in the counting pass
        __syncthreads();
        if (tid < p.bs) req_dest[tid] = wsum[warp * L + my_a] + my_pre;
    } else {
        for (int i0 = 0; i0 < p.bs; i0 += kBuildThreads) {
            int i = i0 + tid;
            bool valid = i < p.bs;
            int a = valid ? p.req_adapter[i] : -1;
            int l = valid ? p.req_lens[i] : 0;
            bool last;
            const int pre = same_key_prefix(a, l, lens_w, last);
            for (int x = tid; x < kWarps * L; x += kBuildThreads) wsum[x] = 0;
            __syncthreads();
            if (valid && last) wsum[warp * L + a] = pre + l;
            __syncthreads();
            slot_scan();
            __syncthreads();
            if (valid) req_dest[i] = wsum[warp * L + a] + pre;
            __syncthreads();  // wsum is reused by the next tile
        }
    }
    __syncthreads();

    // Segments (chunked_backend.py _get_segments_info): slot runs in ascending
    // slot order, each cut into ceil(n / chunk) pieces of chunk tokens, the
    // last one shorter.
    if (tid == 0) bi.seg_indptr[0] = 0;
    for (int k = tid; k < nseg; k += kBuildThreads) {
        int a = last_not_greater(segbase, L, k);
        int j = k - segbase[a];
        bi.weight_indices[k] = a;
        bi.seg_indptr[k + 1] = tokbase[a] + min((j + 1) * chunk, cnt[a]);
    }
    if (p.use_graph) {
        for (int k = nseg + tid; k < bi.max_segments; k += kBuildThreads) {
            bi.weight_indices[k] = 0;
            bi.seg_indptr[k + 1] = p.num_tokens;
        }
    }

    // permutation[dest of token t] = t: one warp per request, whose tokens
    // stay consecutive in sorted order.
    for (int i = warp; i < p.bs; i += kWarps) {
        const int s0 = req_start[i], n = req_start[i + 1] - s0, d0 = req_dest[i];
        for (int j = lane; j < n; j += 32) bi.permutation[d0 + j] = s0 + j;
    }

    // Decode tiles (csgmv_batch_info.tile_table): slots in ascending order are
    // the slot runs; slot a's cnt[a] tokens become ceil(cnt[a] / kDecTM)
    // tiles of balanced size.
    if (bi.tile_table) {
        int *rec = bi.tile_table + 4;
        for (int t = tid; t < dcarry; t += kBuildThreads) {
            const int a = last_not_greater(tilebase, L, t);  // the last slot whose tiles start at or before t
            const int n = cnt[a];
            const int nt = (n + kDecTM - 1) / kDecTM;
            const int i = t - tilebase[a];
            const int lo = i * n / nt, hi = (i + 1) * n / nt;
            rec[4 * t] = a;
            rec[4 * t + 1] = tokbase[a] + lo;
            rec[4 * t + 2] = hi - lo;
            rec[4 * t + 3] = 0;
        }
        if (tid < 4) bi.tile_table[tid] = tid == 0 ? dcarry : 0;
    }

    // Per-request fields (chunked_backend.py _build_req_seg_indptr, req_weight_indices).
    if (bi.req_seg_indptr)
        for (int i = tid; i <= p.bs; i += kBuildThreads) bi.req_seg_indptr[i] = req_start[i];
    if (bi.req_weight_indices)
        for (int i = tid; i < p.bs; i += kBuildThreads) bi.req_weight_indices[i] = p.req_adapter[i];

    if (tid == 0) {
        *bi.num_segments_dev = nseg;
        *bi.max_len_dev = chunk;
        *bi.status = 0;
    }
}

// Inclusive block-wide maximum scan of v; the block maximum goes to *total.
__device__ int block_inclusive_max_scan(int v, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc = max(inc, n);
    }
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w = max(w, n);
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const int r = warp > 0 ? max(warp_sums[warp - 1], inc) : inc;
    *total = warp_sums[kWarps - 1];
    __syncthreads();
    return r;
}

// Batch info of a pruned lm_head pass (chunked_backend.py
// _prepare_lm_head_batch_info / _build_lm_head_batch_info): the pruned tokens
// stay in their original order (identity permutation); a token starts a run
// when its slot differs from the previous pruned token's, and a segment at
// every chunk-th token of a run.  Requests without pruned tokens contribute
// no token, so runs merge across them.  Tiles of 1024 tokens; the current
// run's start and the segment count carry from tile to tile.
__global__ void __launch_bounds__(kBuildThreads, 1)
build_lm_head_kernel(BuildParams p, csgmv_batch_info bi) {
    extern __shared__ int sm[];
    griddep_launch_dependents();  // as in build_batch_info_kernel
    const int L = bi.max_loras;
    int *req_start = sm;                   // [bs+1] first pruned token of request i
    int *warp_sums = req_start + p.bs + 1;  // [32]
    int *flags = warp_sums + kWarps;       // [0] error bits
    const int tid = threadIdx.x;
    const int chunk = p.chunk;
    if (tid == 0) flags[0] = 0;
    __syncthreads();

    // Slot table (lora_manager.py prepare_lora_batch: lora_ranks / scalings per slot).
    for (int a = tid; a < L; a += kBuildThreads) {
        int r = 0;
        float sc = 0.f;
        if (a < p.num_loras) {
            r = p.ranks_in[a];
            sc = p.scalings_in[a];
            if (r < 0 || r > bi.max_rank) { atomicOr(&flags[0], CSGMV_STATUS_BAD_RANK); r = 0; }
        }
        bi.lora_ranks[a] = r;
        bi.scalings[a] = sc;
    }
    // First pruned token of every request, and validation.
    int carry = 0;
    for (int i0 = 0; i0 < p.bs; i0 += kBuildThreads) {
        const int i = i0 + tid;
        int l = 0;
        if (i < p.bs) {
            l = p.req_lens[i];
            const int a = p.req_adapter[i];
            if (a < 0 || a >= p.num_loras) atomicOr(&flags[0], CSGMV_STATUS_BAD_ADAPTER);
            if (l < 0) { atomicOr(&flags[0], CSGMV_STATUS_BAD_LENS); l = 0; }
        }
        int tot;
        const int pre = block_exclusive_scan(l, warp_sums, &tot);
        if (i < p.bs) req_start[i] = carry + pre;
        carry += tot;
    }
    if (tid == 0) {
        req_start[p.bs] = carry;
        if (carry != p.num_tokens) atomicOr(&flags[0], CSGMV_STATUS_BAD_LENS);
    }
    __syncthreads();
    const int err = flags[0];
    // no tile table: the decode kernels derive tiles from the segments
    if (tid == 0 && bi.tile_table) bi.tile_table[0] = -1;
    // per-request fields: first pruned token and slot of every request
    if (!err) {
        if (bi.req_seg_indptr)
            for (int i = tid; i <= p.bs; i += kBuildThreads) bi.req_seg_indptr[i] = req_start[i];
        if (bi.req_weight_indices)
            for (int i = tid; i < p.bs; i += kBuildThreads) bi.req_weight_indices[i] = p.req_adapter[i];
    }
    if (err) {
        if (tid == 0) {
            *bi.num_segments_dev = 0;
            *bi.max_len_dev = chunk;
            bi.seg_indptr[0] = 0;
            *bi.status = err;
        }
        return;
    }

    const int s = p.num_tokens;
    auto slot_of = [&](int t) { return p.req_adapter[last_not_greater(req_start, p.bs + 1, t)]; };
    int run_carry = 0, seg_carry = 0;
    for (int t0 = 0; t0 < s; t0 += kBuildThreads) {
        const int t = t0 + tid;
        const bool valid = t < s;
        const int a = valid ? slot_of(t) : -1;
        const bool run_start = valid && (t == 0 || slot_of(t - 1) != a);
        int rmax;
        int rs = block_inclusive_max_scan(run_start ? t : -1, warp_sums, &rmax);
        rs = max(rs, run_carry);
        const int seg_start = valid && ((t - rs) % chunk == 0);
        int nnew;
        const int seg = seg_carry + block_exclusive_scan(seg_start, warp_sums, &nnew);
        if (seg_start && seg < bi.max_segments) {
            bi.weight_indices[seg] = a;
            bi.seg_indptr[seg] = t;
        }
        if (valid) bi.permutation[t] = t;
        run_carry = max(run_carry, rmax);
        seg_carry += nnew;
    }
    const int nseg = seg_carry;
    if (nseg > bi.max_segments) {
        if (tid == 0) {
            *bi.num_segments_dev = 0;
            *bi.max_len_dev = chunk;
            bi.seg_indptr[0] = 0;
            *bi.status = CSGMV_STATUS_CAPACITY;
        }
        return;
    }
    if (tid == 0) bi.seg_indptr[nseg] = s;
    if (p.use_graph) {
        for (int k = nseg + tid; k < bi.max_segments; k += kBuildThreads) {
            bi.weight_indices[k] = 0;
            bi.seg_indptr[k + 1] = s;
        }
    }
    if (tid == 0) {
        *bi.num_segments_dev = nseg;
        *bi.max_len_dev = chunk;
        *bi.status = 0;
    }
}

// Lets `fn` take up to 227 KB of dynamic shared memory on the current
// device.  The attribute belongs to the kernel on each device, so it is set
// once per (kernel, device), under a lock for callers on several threads.
cudaError_t allow_large_smem(const void *fn) {
    static std::mutex mu;
    static std::set<std::pair<const void *, int>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    if (done.count({fn, dev})) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    done.insert({fn, dev});
    return cudaSuccess;
}

}  // namespace

size_t build_lm_head_smem_bytes(int bs) { return sizeof(int) * ((size_t)bs + 1 + kWarps + 2); }

cudaError_t launch_build_lm_head(const BuildParams &p, const csgmv_batch_info &bi, cudaStream_t stream) {
    size_t smem = build_lm_head_smem_bytes(p.bs);
    cudaError_t e = allow_large_smem(reinterpret_cast<const void *>(build_lm_head_kernel));
    if (e != cudaSuccess) return e;
    build_lm_head_kernel<<<1, kBuildThreads, smem, stream>>>(p, bi);
    return cudaGetLastError();
}

size_t build_smem_bytes(int bs, int max_loras) {
    return sizeof(int) * ((size_t)5 * max_loras + 1 + 2 * (size_t)bs + 1 + kWarps + 2 + (size_t)kWarps * max_loras +
                          3 * kWarps + 32 * kWarps);
}

cudaError_t launch_build(const BuildParams &p, const csgmv_batch_info &bi, cudaStream_t stream) {
    size_t smem = build_smem_bytes(p.bs, bi.max_loras);
    cudaError_t e = allow_large_smem(reinterpret_cast<const void *>(build_batch_info_kernel));
    if (e != cudaSuccess) return e;
    build_batch_info_kernel<<<1, kBuildThreads, smem, stream>>>(p, bi);
    return cudaGetLastError();
}

}  // namespace csgmv
