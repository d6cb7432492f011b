// Decode-shaped csgmv_qkv through the h workspace: the split-K shrink and the
// expand described in lora_decode.cuh.
#include "lora_decode.cuh"

namespace csgmv {
namespace {

struct DecTab {
    int *ip, *sw, *rk, *perm, *run_w, *run_p0, *run_n, *run_t0, *scratch, *rec;
    float *sc;
};

__device__ __forceinline__ DecTab dec_tab(unsigned char *base) {
    int *t = reinterpret_cast<int *>(base);
    DecTab T;
    T.ip = t + kDecTabIp;
    T.sw = t + kDecTabSw;
    T.rk = t + kDecTabRk;
    T.sc = reinterpret_cast<float *>(t + kDecTabSc);
    T.perm = t + kDecTabPerm;
    T.run_w = t + kDecTabRunW;
    T.run_p0 = t + kDecTabRunP0;
    T.run_n = t + kDecTabRunN;
    T.run_t0 = t + kDecTabRunT0;
    T.scratch = t + kDecTabScratch;
    T.rec = t + kDecTabRec;
    return T;
}

__device__ __forceinline__ unsigned char *align_1024(unsigned char *p) {
    return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ int warp_inclusive_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Tile table of the batch (chunked_backend.py _get_segments_info order: slot
// runs in segment order).  A slot run is a maximal stretch of consecutive
// segments on one slot; a run of n tokens becomes ceil(n / kDecTM) tiles of
// balanced size.  Every word is loaded in one round, bounded by the
// capacities rather than by the counts that come with them: the batch info's
// tile table (its count and first kDecRecCap records), and the segments,
// slot ranks and scalings and the permutation.  When the builder wrote the
// table (count >= 0), that is all; otherwise one warp builds the runs from
// the segments with shuffles while the others wait.  Returns the tile count
// and the run count (-1: tiles come from the builder's records); every
// thread of the block calls it, and it ends with a block barrier.
template <int NT>
__device__ int dec_build(const DecodeParams &k, const DecTab &T, int *nruns_out) {
    const LoraParams &p = k.p;
    const int tid = threadIdx.x;
    const int ms = min(k.max_segments, kDecSegCap);
    const int nl = min(p.max_loras, kDecLoraCap);
    const int nperm = min(p.num_tokens, kDecPermCap);
    const int nrec = p.tile_table ? 4 * min(k.tile_cap, kDecRecCap) : 0;
    // a fixed number of words per thread, all loaded into registers before
    // the first of them is stored, so that the loads overlap
    constexpr int NIP = (kDecSegCap + NT) / NT, NL = (kDecLoraCap + NT - 1) / NT;
    constexpr int NP = (kDecPermCap + NT - 1) / NT, NR = (4 * kDecRecCap + NT - 1) / NT;
    int vip[NIP], vsw[NIP], vrk[NL], vp[NP], vrec[NR];
    float vsc[NL];
    const int nseg_raw = *p.num_segments_dev;
    const int built = p.tile_table ? p.tile_table[0] : -1;
#pragma unroll
    for (int i = 0; i < NIP; ++i) {
        const int s = tid + i * NT;
        vip[i] = s <= ms ? p.seg_indptr[s] : 0;
        vsw[i] = s < ms ? p.weight_indices[s] : 0;
    }
#pragma unroll
    for (int i = 0; i < NL; ++i) {
        const int a = tid + i * NT;
        vrk[i] = a < nl ? p.lora_ranks[a] : 0;
        vsc[i] = a < nl ? p.scalings[a] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < NP; ++i) vp[i] = tid + i * NT < nperm ? p.permutation[tid + i * NT] : 0;
#pragma unroll
    for (int i = 0; i < NR; ++i) vrec[i] = tid + i * NT < nrec ? p.tile_table[4 + tid + i * NT] : 0;
#pragma unroll
    for (int i = 0; i < NIP; ++i) {
        const int s = tid + i * NT;
        if (s <= ms) T.ip[s] = vip[i];
        if (s < ms) T.sw[s] = vsw[i];
    }
#pragma unroll
    for (int i = 0; i < NL; ++i)
        if (tid + i * NT < nl) {
            T.rk[tid + i * NT] = vrk[i];
            T.sc[tid + i * NT] = vsc[i];
        }
#pragma unroll
    for (int i = 0; i < NP; ++i)
        if (tid + i * NT < nperm) T.perm[tid + i * NT] = vp[i];
#pragma unroll
    for (int i = 0; i < NR; ++i)
        if (tid + i * NT < nrec) T.rec[tid + i * NT] = vrec[i];
    __syncthreads();
    if (built >= 0) {
        *nruns_out = -1;
        return min(built, k.tile_cap);
    }

    if (tid < 32) {
        const int lane = tid;
        const int nseg = max(0, min(nseg_raw, ms));
        // lane `lane` takes segments [s0, s1)
        const int per = (nseg + 31) >> 5;
        const int s0 = min(nseg, lane * per), s1 = min(nseg, s0 + per);
        int starts = 0;
        for (int s = s0; s < s1; ++s) starts += s == 0 || T.sw[s] != T.sw[s - 1];
        const int inc = warp_inclusive_scan(starts);
        const int nruns = __shfl_sync(0xffffffffu, inc, 31);
        int cur = inc - starts - 1;  // run holding the segment before s0
        for (int s = s0; s < s1; ++s) {
            if (s == 0 || T.sw[s] != T.sw[s - 1]) {
                ++cur;
                T.run_w[cur] = T.sw[s];
                T.run_p0[cur] = T.ip[s];
            }
            if (s == nseg - 1 || T.sw[s + 1] != T.sw[s]) T.run_n[cur] = T.ip[s + 1];  // the run's end for now
        }
        __syncwarp();
        // lane `lane` takes runs [r0, r1): lengths (clamped) and tiles
        const int perr = (nruns + 31) >> 5;
        const int r0 = min(nruns, lane * perr), r1 = min(nruns, r0 + perr);
        int tiles = 0;
        for (int r = r0; r < r1; ++r) {
            const int a = max(0, min(T.run_p0[r], p.num_tokens));
            const int b = max(a, min(T.run_n[r], p.num_tokens));
            T.run_p0[r] = a;
            T.run_n[r] = b - a;
            tiles += (b - a + kDecTM - 1) / kDecTM;
        }
        const int tinc = warp_inclusive_scan(tiles);
        int t0 = tinc - tiles;
        for (int r = r0; r < r1; ++r) {
            T.run_t0[r] = t0;
            t0 += (T.run_n[r] + kDecTM - 1) / kDecTM;
        }
        if (lane == 31) {
            T.run_t0[nruns] = tinc;
            T.scratch[0] = tinc;
            T.scratch[1] = nruns;
        }
    }
    __syncthreads();
    *nruns_out = T.scratch[1];
    return T.scratch[0];
}

// Slot, first sorted position and size of tile `tile`.
__device__ __forceinline__ void dec_tile(const DecodeParams &k, const DecTab &T, int nruns, int tile, int &w, int &p0,
                                         int &M) {
    if (nruns < 0) {  // the builder's records
        const int *rec = tile < kDecRecCap ? T.rec + 4 * tile : k.p.tile_table + 4 + 4 * tile;
        w = rec[0];
        p0 = max(0, min(rec[1], k.p.num_tokens));
        M = max(0, min(rec[2], min(kDecTM, k.p.num_tokens - p0)));
        return;
    }
    int lo = 0, hi = nruns;  // last run with run_t0 <= tile (runs without tiles are skipped)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (T.run_t0[mid] <= tile) lo = mid; else hi = mid;
    }
    const int nt = T.run_t0[lo + 1] - T.run_t0[lo];
    const int i = tile - T.run_t0[lo];
    const int n = T.run_n[lo];
    const int a = i * n / nt, b = (i + 1) * n / nt;  // n <= kDecPermCap, i < 64
    w = T.run_w[lo];
    p0 = T.run_p0[lo] + a;
    M = b - a;
}

// Rank of slot w, or -1 for an invalid slot or rank (reported once per unit).
__device__ __forceinline__ int dec_rank(const DecodeParams &k, const DecTab &T, int w, bool report) {
    if (w < 0 || w >= k.p.max_loras || w >= kDecLoraCap) {
        if (report) atomicOr(k.p.status, CSGMV_STATUS_BAD_ADAPTER);
        return -1;
    }
    const int r = T.rk[w];
    if (r < 0 || r > k.p.R) {
        if (report) atomicOr(k.p.status, CSGMV_STATUS_BAD_RANK);
        return -1;
    }
    return r;
}

// Token of sorted position pos, or -1 (reported) when the entry is out of range.
__device__ __forceinline__ int dec_token(const DecodeParams &k, const DecTab &T, int pos) {
    const int t = T.perm[pos];
    if (t < 0 || t >= k.p.num_tokens) {
        atomicOr(k.p.status, CSGMV_STATUS_BAD_PERMUTATION);
        return -1;
    }
    return t;
}

// Parts of K per tile: about one shrink unit per CTA of the shrink launch,
// at most kDecPartsTarget, one part per K chunk and one per plane the
// workspace holds.
__device__ __forceinline__ int dec_parts(const DecodeParams &k, int ntiles) {
    const int P = ntiles > 0 ? k.shrink_grid / ntiles : 1;
    return max(1, min(min(P, kDecPartsTarget), min(k.nkc, k.p.h_parts)));
}

// Row m of a tile is copied by lane 1 + m / W of warp m % W (W warps; lane 0
// of each warp issues the TMA boxes), so that no lane issues more than
// kDecTM / W copies and rows go out from every warp at once.
template <int W>
__device__ __forceinline__ int dec_row_of_thread(int lane, int warp) {
    return lane >= 1 && lane <= kDecTM / W ? (lane - 1) * W + warp : -1;
}

}  // namespace

// ------------------------------------------------------------------------------------ shrink
// The shrink's products of one pass: NMT 16-row tiles of x times NJ n8
// column tiles of h (this warp's: columns (warp + 8 i) * 8), over nch 64-wide
// K chunks.  x rows at xm[mt] (the lane's ldmatrix row, 16-row tile mt); the
// A box of chunk ci at a_base + ci * abox (128-byte rows, 128-byte swizzle),
// the lane's ldmatrix row of column tile i at b_off[i] and its 16-byte chunk
// of k16 step ks at cofs[ks].
template <int NMT, int NJ>
__device__ __forceinline__ void shrink_mma(float (&acc)[4][3][4], uint32_t a_base, uint32_t abox,
                                           const uint32_t (&xm)[4], int nch, const uint32_t (&b_off)[3],
                                           const uint32_t (&cofs)[4]) {
    for (int ci = 0; ci < nch; ++ci) {
        const uint32_t ab = a_base + ci * abox;
        const uint32_t xc = ci * 128;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t b[NJ][2];
#pragma unroll
            for (int i = 0; i < NJ; ++i) ldsm_x2(b[i][0], b[i][1], ab + b_off[i] + cofs[ks]);
#pragma unroll
            for (int mt = 0; mt < NMT; ++mt) {
                uint32_t a[4];
                ldsm_x4(a, xm[mt] + xc + ks * 32);
#pragma unroll
                for (int i = 0; i < NJ; ++i) mma_bf16_16816(acc[mt][i], a, b[i][0], b[i][1]);
            }
        }
    }
}

template <int NMT>
__device__ __forceinline__ void shrink_mma_nj(int nj, float (&acc)[4][3][4], uint32_t a_base, uint32_t abox,
                                              const uint32_t (&xm)[4], int nch, const uint32_t (&b_off)[3],
                                              const uint32_t (&cofs)[4]) {
    if (nj == 1) shrink_mma<NMT, 1>(acc, a_base, abox, xm, nch, b_off, cofs);
    else if (nj == 2) shrink_mma<NMT, 2>(acc, a_base, abox, xm, nch, b_off, cofs);
    else if (nj == 3) shrink_mma<NMT, 3>(acc, a_base, abox, xm, nch, b_off, cofs);
}

__global__ void __launch_bounds__(kDecThreads, 2) lora_decode_shrink_kernel(const __grid_constant__ DecodeParams k) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = align_1024(smem_raw);
    const LoraParams &p = k.p;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + k.o_bar);
    const DecTab T = dec_tab(smem + k.o_tab);
    unsigned char *as = smem + k.o_a;  // [kc_max][a_rows][128 B] A boxes, 128-byte swizzle
    unsigned char *xs = smem + k.o_x;  // [kDecTM][xpitch] x rows
    if (tid == 0) {
        mbar_init(full, kDecThreads);
        fence_mbar_init();
        prefetch_tmap(&k.tmA);
    }
    griddep_wait();  // the batch info and the planes' last reader come before this kernel
    // the expand may launch now: every word it reads before its own wait is final
    griddep_launch_dependents();
    int nruns;
    const int ntiles = dec_build<kDecThreads>(k, T, &nruns);
    const int P = dec_parts(k, ntiles);
    const int units = ntiles * P;  // <= kDecPermCap * kDecMaxParts
    const uint32_t abox = (uint32_t)k.a_rows * 128;
    const int my_row = dec_row_of_thread<kDecWarps>(lane, warp);
    // per-lane shared-memory addresses of the ldmatrix rows
    const uint32_t as_u = smem_u32(as);
    uint32_t cofs[4], xm[4];
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) cofs[ks] = (uint32_t)(((2 * ks + ((lane >> 3) & 1)) ^ (lane & 7)) << 4);
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
        xm[mt] = smem_u32(xs) + (uint32_t)((mt * 16 + (lane & 15)) * k.xpitch + 16 * (lane >> 4));
    uint32_t b_off[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) b_off[i] = (uint32_t)((warp + kDecWarps * i) * 8 * 128 + (lane & 7) * 128);
    uint32_t phase = 0;

    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int tile = u / P, part = u - (u / P) * P;
        int w, p0, M;
        dec_tile(k, T, nruns, tile, w, p0, M);
        const int r = dec_rank(k, T, w, tid == 0 && part == 0);
        if (r <= 0 || M <= 0) continue;  // rank 0: the expand leaves these rows alone
        const int nt8 = ((p.c * r + 7) & ~7) / 8;                    // n8 column tiles of h
        const int nj = warp < nt8 ? (nt8 - warp + kDecWarps - 1) / kDecWarps : 0;  // this warp's
        const int nmt = (M + 15) / 16;
        const int kc0 = part * k.nkc / P, kc1 = (part + 1) * k.nkc / P;
        const int t_row = my_row >= 0 && my_row < M ? dec_token(k, T, p0 + my_row) : -1;

        float acc[4][3][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int i = 0; i < 3; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][i][e] = 0.f;

        for (int c0 = kc0; c0 < kc1; c0 += k.kc_max) {
            const int nch = min(k.kc_max, kc1 - c0);
            const int xcols = (int)(min((int64_t)(c0 + nch) * 64, p.K) - (int64_t)c0 * 64);
            fence_proxy_async_smem();  // generic reads of the last pass before the copies overwrite them
            __syncthreads();
            uint32_t bytes = 0;
            if (lane == 0)
                for (int ci = warp; ci < nch; ci += kDecWarps) bytes += abox;
            if (my_row >= 0) {
                // columns past K in a partial last chunk meet the zero-filled
                // A columns: zero them, since stale values could be NaN
                __nv_bfloat16 *row = reinterpret_cast<__nv_bfloat16 *>(xs + my_row * k.xpitch);
                for (int col = xcols; col < nch * 64; ++col) row[col] = __float2bfloat16_rn(0.f);
                if (t_row >= 0) bytes += (uint32_t)xcols * 2;
            }
            mbar_arrive_expect_tx(full, bytes);
            if (lane == 0)
                for (int ci = warp; ci < nch; ci += kDecWarps)
                    tma_load_2d(as + ci * abox, &k.tmA, (c0 + ci) * 64, w * p.c * p.R, full);
            if (t_row >= 0)
                bulk_g2s(xs + my_row * k.xpitch, p.x + (int64_t)t_row * p.K + (int64_t)c0 * 64, (uint32_t)xcols * 2,
                         full);
            mbar_wait(full, phase, p.status, kStatusTimeout);
            phase ^= 1;
            switch (nmt) {  // warp-uniform: one specialised loop per tile count
                case 1: shrink_mma_nj<1>(nj, acc, as_u, abox, xm, nch, b_off, cofs); break;
                case 2: shrink_mma_nj<2>(nj, acc, as_u, abox, xm, nch, b_off, cofs); break;
                case 3: shrink_mma_nj<3>(nj, acc, as_u, abox, xm, nch, b_off, cofs); break;
                default: shrink_mma_nj<4>(nj, acc, as_u, abox, xm, nch, b_off, cofs); break;
            }
        }

        // partial sums over this part of K into plane `part`, rows p0 + m
        float *plane = reinterpret_cast<float *>(p.h) + (int64_t)part * p.h_plane;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                if (mt < nmt && i < nj) {
                    const int row = mt * 16 + (lane >> 2), col = (warp + kDecWarps * i) * 8 + 2 * (lane & 3);
                    if (row < M)
                        *reinterpret_cast<float2 *>(plane + (int64_t)(p0 + row) * p.ldh + col) =
                            make_float2(acc[mt][i][0], acc[mt][i][1]);
                    if (row + 8 < M)
                        *reinterpret_cast<float2 *>(plane + (int64_t)(p0 + row + 8) * p.ldh + col) =
                            make_float2(acc[mt][i][2], acc[mt][i][3]);
                }
            }
        }
    }
}

// ------------------------------------------------------------------------------------ expand
// Column parts of one tile: slice j's 64-column blocks (counted from off[j])
// go to cum[j + 1] - cum[j] parts, about Q * (its blocks) / (all blocks) and
// at least enough for bmax blocks a part, so that no unit spans two slices.
// cum[c] is the tile's unit count.
__device__ __forceinline__ void dec_col_parts(const LoraParams &p, int Q, int bmax, int (&cum)[kMaxSlices + 1]) {
    int b[kMaxSlices], B = 0;
#pragma unroll
    for (int j = 0; j < kMaxSlices; ++j) {
        b[j] = j < p.c ? (p.off[j + 1] - p.off[j] + 63) / 64 : 0;
        B += b[j];
    }
    cum[0] = 0;
    int acc = 0;
#pragma unroll
    for (int j = 0; j < kMaxSlices; ++j) {
        acc += b[j];
        const int want = B > 0 ? (int)(((int64_t)Q * acc + B / 2) / B) : 0;
        const int parts = b[j] > 0 ? max((b[j] + bmax - 1) / bmax, max(1, want - cum[j])) : 0;
        cum[j + 1] = cum[j] + parts;
    }
}

// Slice of output column col (slice offsets are multiples of 8, so an n8
// column tile lies in one slice).
__device__ __forceinline__ int slice_of(const LoraParams &p, int col) {
    return (p.c > 1 && col >= p.off[1]) + (p.c > 2 && col >= p.off[2]);
}

template <int RMAX>
__global__ void __launch_bounds__(kDecExpThreads, 2) lora_decode_expand_kernel(const __grid_constant__ DecodeParams k) {
    constexpr int KS = RMAX / 16;  // k16 steps at most
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = align_1024(smem_raw);
    const LoraParams &p = k.p;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + k.o_bar);
    const DecTab T = dec_tab(smem + k.o_tab);
    unsigned char *ys = smem + k.o_y;  // [kDecTM][ypitch] base rows, then y in place
    __nv_bfloat16 *bs = reinterpret_cast<__nv_bfloat16 *>(smem + k.o_b);  // [cols_max][R] B rows (TMA boxes)
    // h as mma A fragments: [slice][16-row tile][k16 step][hi, lo][lane][4 registers]
    uint32_t *hf = reinterpret_cast<uint32_t *>(smem + k.o_h);
    if (tid == 0) {
        mbar_init(full, kDecExpThreads);
        fence_mbar_init();
        prefetch_tmap(&k.tmB);
        if (p.b_tuple)
            for (int j = 0; j < kMaxSlices; ++j) prefetch_tmap(&k.tmBs[j]);
    }
    // The batch info, B and the base rows are read before griddep_wait.
    // This kernel follows its shrink in the stream, and the shrink lets it
    // launch only after every shrink CTA has passed its own griddep_wait, so
    // the builder and every earlier kernel that wrote those words (an earlier
    // call's expand included) are complete.  Only the planes come from the
    // shrink itself.
    int nruns;
    const int ntiles = dec_build<kDecExpThreads>(k, T, &nruns);
    const int P = dec_parts(k, ntiles);
    const int ncols = p.off[p.c] - p.off[0];
    const int nblk = (ncols + 63) / 64;
    const int bmax = k.cols_max / 64;
    const int qmin = (nblk + bmax - 1) / bmax;
    const int Qw = max(qmin, min(nblk, ntiles > 0 ? (int)gridDim.x / ntiles : 1));
    int cum[kMaxSlices + 1];
    dec_col_parts(p, Qw, bmax, cum);
    const int Q = cum[p.c];  // units per tile
    const int units = ntiles * Q;
    const int my_row = dec_row_of_thread<kDecExpWarps>(lane, warp);
    const int pcB = p.R / 8, shB = pc_shift_of(pcB);
    const uint32_t ys_u = smem_u32(ys), bs_u = smem_u32(bs), hf_u = smem_u32(hf);
    const int pstep = (int)p.h_plane;  // floats per plane: num_tokens * ldh <= kDecPermCap * 192
    bool waited = false;
    uint32_t phase = 0;

    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int tile = u / Q, q = u - (u / Q) * Q;
        int w, p0, M;
        dec_tile(k, T, nruns, tile, w, p0, M);
        const int r = dec_rank(k, T, w, false);  // the shrink reports bad slots and ranks
        if (r <= 0 || M <= 0) continue;          // accumulate: rank 0 leaves y as it is
        int js = 0;
        while (js + 1 < p.c && q >= cum[js + 1]) ++js;
        const int bj = (p.off[js + 1] - p.off[js] + 63) / 64, parts = cum[js + 1] - cum[js], iq = q - cum[js];
        const int n0 = p.off[js] + 64 * (iq * bj / parts);
        const int n1 = min(p.off[js + 1], p.off[js] + 64 * ((iq + 1) * bj / parts));
        if (n1 <= n0) continue;
        const int nu = n1 - n0;
        const int nbox = (nu + 63) / 64;
        const int t_row = my_row >= 0 && my_row < M ? T.perm[p0 + my_row] : -1;
        const bool row_ok = t_row >= 0 && t_row < p.num_tokens;

        fence_proxy_async_smem();  // generic accesses of the last unit before the copies overwrite them
        __syncthreads();
        uint32_t bytes = 0;
        if (lane == 0)
            for (int bx = warp; bx < nbox; bx += kDecExpWarps) bytes += 64u * p.R * 2;
        if (row_ok) bytes += (uint32_t)nu * 2;
        mbar_arrive_expect_tx(full, bytes);
        if (lane == 0)
            for (int bx = warp; bx < nbox; bx += kDecExpWarps) {
                const int col = n0 + 64 * bx;
                if (!p.b_tuple) {
                    tma_load_2d(bs + bx * 64 * p.R, &k.tmB, 0, w * (int)p.N + col, full);
                } else {
                    const int j = slice_of(p, col);
                    tma_load_2d(bs + bx * 64 * p.R, &k.tmBs[j], 0, w * p.b_rows[j] + p.b_row0[j] + (col - p.off[j]),
                                full);
                }
            }
        if (row_ok) bulk_g2s(ys + my_row * k.ypitch, p.y + (int64_t)t_row * p.N + n0, (uint32_t)nu * 2, full);
        if (!waited) {
            griddep_wait();  // the shrink's planes are complete from here on
            waited = true;
        }

        // h of the slices [jl, jh] this unit spans, the planes summed in part
        // order, written as bf16 hi / lo A fragments: element (m, kk) of a
        // slice goes to lane (m % 8) * 4 + (kk % 8) / 2, register
        // (m / 8) % 2 + 2 * ((kk % 16) / 8) of 16-row tile m / 16, k16 step
        // kk / 16.  Each thread takes kDecExpItems (row, column) items per
        // round with the loads of all of them in flight at once; even lanes
        // pair their column with the next lane's (kcols is even, so those are
        // neighbours in a row).
        const int jl = slice_of(p, n0), jh = slice_of(p, n1 - 1);
        const int nmt = (M + 15) / 16;
        const int ksteps = (r + 15) / 16;
        const int rows = nmt * 16, kcols = 16 * ksteps;
        const int per_slice = rows * kcols;
        const int items = (jh - jl + 1) * per_slice;
        const float *planes = reinterpret_cast<const float *>(p.h);
        for (int base = 0; base < items; base += kDecExpItems * kDecExpThreads) {
            const float *src[kDecExpItems];
            int jm[kDecExpItems], mm[kDecExpItems], kk2[kDecExpItems];
            bool live[kDecExpItems];
#pragma unroll
            for (int h = 0; h < kDecExpItems; ++h) {
                const int it = base + h * kDecExpThreads + tid;
                const int js = it / per_slice, rem = it - js * per_slice;
                jm[h] = jl + js;
                mm[h] = rem / kcols;
                kk2[h] = rem - mm[h] * kcols;
                live[h] = it < items && mm[h] < M && kk2[h] < r;
                src[h] = planes + (p0 + mm[h]) * (int)p.ldh + jm[h] * r + kk2[h];
            }
            float v[kDecExpItems];
#pragma unroll
            for (int h = 0; h < kDecExpItems; ++h) v[h] = 0.f;
#pragma unroll
            for (int b0 = 0; b0 < kDecMaxParts; b0 += 16) {
                if (b0 < P) {
                    float a[kDecExpItems][16];
#pragma unroll
                    for (int h = 0; h < kDecExpItems; ++h)
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (live[h] && b0 + i < P) a[h][i] = src[h][(b0 + i) * pstep];
#pragma unroll
                    for (int h = 0; h < kDecExpItems; ++h)
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (live[h] && b0 + i < P) v[h] = (b0 + i == 0) ? a[h][i] : v[h] + a[h][i];
                }
            }
#pragma unroll
            for (int h = 0; h < kDecExpItems; ++h) {
                const float v1 = __shfl_down_sync(0xffffffffu, v[h], 1);
                const int it = base + h * kDecExpThreads + tid;
                if (!(lane & 1) && it < items) {
                    uint32_t hi, lo;
                    split_pair(v[h], v1, hi, lo);
                    const int m = mm[h], cp = kk2[h] >> 1;
                    const int fl = (m & 7) * 4 + (cp & 3), reg = ((m >> 3) & 1) + 2 * ((cp >> 2) & 1);
                    uint32_t *f = hf + ((((jm[h] * 4 + (m >> 4)) * KS + (cp >> 3)) * 2) * 32 + fl) * 4 + reg;
                    f[0] = hi;
                    f[128] = lo;
                }
            }
        }
        mbar_wait(full, phase, p.status, kStatusTimeout);
        phase ^= 1;
        // B columns [r, 16 * ceil(r / 16)) are adapter padding (R = 8: [r, 8)):
        // zero them so that padding never reaches the output, even NaN
        const bool r_ragged = p.R == 8 ? (r < 8) : (r % 16 != 0);
        if (r_ragged) {
            const int rpad = p.R == 8 ? 8 : (r + 15) / 16 * 16;
            const int npad = rpad - r;
            for (int idx = tid; idx < nbox * 64 * npad; idx += kDecExpThreads) {
                const int n = idx / npad, kk = r + idx % npad;
                bs[swz(n, kk >> 3, pcB, shB) + (kk & 7)] = __float2bfloat16_rn(0.f);
            }
        }
        __syncthreads();  // h fragments written, B padding zeroed

        // warp `warp` takes 16-column pairs warp, warp + 8, ...: per 16-row
        // tile, the pair's B fragments (ldmatrix x4, both n8 halves), h
        // fragments of each half's slice, hi and lo MMAs, then
        // y = base + sigma * acc stored from registers
        const float sigma = T.sc[w];
        const int npairs = (nu + 15) / 16;
        const uint32_t hf_lane = hf_u + (uint32_t)lane * 16;
        for (int pc = warp; pc < npairs; pc += kDecExpWarps) {
            const int lc = 16 * pc;  // local column of the pair
            const bool has1 = lc + 8 < nu;
            const int j0 = slice_of(p, n0 + lc), j1 = has1 ? slice_of(p, n0 + lc + 8) : j0;
            uint32_t baddr[KS];
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                if (RMAX == 16 && p.R == 8) {
                    baddr[ks] = bs_u + (uint32_t)((lc + 8 * ((lane >> 3) & 1) + (lane & 7)) * 16);
                } else {
                    const int nrow = lc + 8 * (lane >> 4) + (lane & 7);
                    const int ch = 2 * ks + ((lane >> 3) & 1);
                    baddr[ks] = bs_u + (uint32_t)swz(nrow, ch, pcB, shB) * 2;
                }
            }
            for (int mt = 0; mt < nmt; ++mt) {
                float acc[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[h][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    if (ks < ksteps) {
                        uint32_t bf[4];
                        if (RMAX == 16 && p.R == 8) {
                            ldsm_x2(bf[0], bf[2], baddr[ks]);
                            bf[1] = 0u;
                            bf[3] = 0u;
                        } else {
                            ldsm_x4(bf, baddr[ks]);
                        }
                        const uint32_t f0 = hf_lane + (uint32_t)(((j0 * 4 + mt) * KS + ks) * 2 * 512);
                        const uint4 h0 = lds_v4(f0), l0 = lds_v4(f0 + 512);
                        const uint32_t ah[4] = {h0.x, h0.y, h0.z, h0.w}, al[4] = {l0.x, l0.y, l0.z, l0.w};
                        mma_bf16_16816(acc[0], ah, bf[0], bf[1]);
                        mma_bf16_16816(acc[0], al, bf[0], bf[1]);
                        if (has1) {
                            if (j1 == j0) {
                                mma_bf16_16816(acc[1], ah, bf[2], bf[3]);
                                mma_bf16_16816(acc[1], al, bf[2], bf[3]);
                            } else {
                                const uint32_t f1 = hf_lane + (uint32_t)(((j1 * 4 + mt) * KS + ks) * 2 * 512);
                                const uint4 h1 = lds_v4(f1), l1 = lds_v4(f1 + 512);
                                const uint32_t bh[4] = {h1.x, h1.y, h1.z, h1.w}, bl[4] = {l1.x, l1.y, l1.z, l1.w};
                                mma_bf16_16816(acc[1], bh, bf[2], bf[3]);
                                mma_bf16_16816(acc[1], bl, bf[2], bf[3]);
                            }
                        }
                    }
                }
                // y = base + sigma * acc, stored from registers (a quad of
                // lanes writes 16 consecutive bytes of a row)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int row = mt * 16 + (lane >> 2) + 8 * rr;
                    if (row >= M) continue;
                    const int t = T.perm[p0 + row];
                    if (t < 0 || t >= p.num_tokens) continue;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h == 1 && !has1) continue;
                        const int col = lc + 8 * h + 2 * (lane & 3);
                        const float2 bv = unpack_bf16x2(lds_b32(ys_u + (uint32_t)(row * k.ypitch + col * 2)));
                        *reinterpret_cast<uint32_t *>(p.y + (int64_t)t * p.N + n0 + col) =
                            pack_bf16x2(bv.x + sigma * acc[h][2 * rr], bv.y + sigma * acc[h][2 * rr + 1]);
                    }
                }
            }
        }
    }
}

const void *lora_kernel_decode(int which, int rmax) {
    if (which == 0) return reinterpret_cast<const void *>(lora_decode_shrink_kernel);
    if (rmax == 16) return reinterpret_cast<const void *>(lora_decode_expand_kernel<16>);
    if (rmax == 32) return reinterpret_cast<const void *>(lora_decode_expand_kernel<32>);
    if (rmax == 64) return reinterpret_cast<const void *>(lora_decode_expand_kernel<64>);
    return nullptr;
}

}  // namespace csgmv
