// The streaming tcgen05 shrink kernel for 128-token tiles (see lora_stream.cuh).
#include "lora_stream.cuh"

namespace csgmv {

namespace {

struct ShBars {
    uint64_t *full, *empty;           // [S]
    uint64_t *acc_full, *acc_empty;   // [2]
    uint64_t *tok_full, *tok_empty;   // [2]
    uint32_t *tmem_slot;
    int *tok;   // [2][128]
    int *flag;  // [2] the tile's rows are consecutive tokens
};

__device__ __forceinline__ ShBars sh_bars(const ShrinkParams &k, unsigned char *smem) {
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + k.o_bar);
    ShBars w;
    w.full = b;
    w.empty = b + k.S;
    w.acc_full = b + 2 * k.S;
    w.acc_empty = w.acc_full + 2;
    w.tok_full = w.acc_empty + 2;
    w.tok_empty = w.tok_full + 2;
    w.tmem_slot = reinterpret_cast<uint32_t *>(w.tok_empty + 2);
    w.tok = reinterpret_cast<int *>(smem + k.o_tok);
    w.flag = w.tok + 256;
    return w;
}

constexpr int kShAccCols = 256;  // TMEM columns per accumulator (c * R <= 192)

// Unit u of the walk: part u / ntiles of K (so that the CTAs working at one
// time share the A columns of one part) of token tile u % ntiles.  False when
// the unit has no tensor-core work (rank 0, an invalid slot or rank).
struct ShWalk {
    int ntiles, P, kc_per;  // tiles, parts of K, 64-wide K chunks per part
};

__device__ __forceinline__ bool sh_unit(const ShrinkParams &k, const int *tables, int nruns, const ShWalk &wk,
                                        int64_t u, bool report, Unit &T, int &r, int &part, int &c0, int &c1) {
    part = (int)(u / wk.ntiles);
    const int tile = (int)(u % wk.ntiles);
    T = tile_of<128>(tables, k.runcap, nruns, tile);
    r = unit_rank(k.p, T, report && part == 0);
    const int nkc = (int)((k.p.K + 63) / 64);
    c0 = part * wk.kc_per;
    c1 = min(nkc, c0 + wk.kc_per);
    return r > 0 && c1 > c0;
}

// Parts of K for ntiles tiles on `grid` CTAs: the best-filled last wave, at
// least four K chunks a part, at most max_parts.  The same on every thread.
__device__ __forceinline__ ShWalk sh_walk(int ntiles, int nkc, int max_parts, int grid) {
    ShWalk wk;
    wk.ntiles = ntiles;
    wk.P = 1;
    float best = 0.f;
    for (int P = 1; P <= max(1, max_parts); ++P) {
        const int kc = (nkc + P - 1) / P;
        if ((nkc + kc - 1) / kc != P || (P > 1 && kc < 4)) continue;
        const long long units = (long long)ntiles * P;
        const long long waves = (units + grid - 1) / grid;
        const float fill = (float)units / (float)(waves * grid);
        if (fill > best + 0.02f) {
            best = fill;
            wk.P = P;
        }
    }
    wk.kc_per = (nkc + wk.P - 1) / wk.P;
    return wk;
}

// A box of a whole stage (3-D view): the smallest of 16, 32 or 64 rows that
// covers the slot's 16 * n16 rows when that is below the full round16(c*R)
// rows (tmA3s[level]), else the full box (level -1).  The chunks of the stage
// then sit `a_stride` bytes apart.  Producer and MMA issuer both use it.
__device__ __forceinline__ int sh_a3_level(const ShrinkParams &k, int n16) {
    const int rows = n16 <= 1 ? 16 : (n16 <= 2 ? 32 : (n16 <= 4 ? 64 : (1 << 30)));
    if (rows >= k.a_bytes / 128) return -1;
    return rows == 16 ? 0 : (rows == 32 ? 1 : 2);
}
__device__ __forceinline__ int sh_a_stride(const ShrinkParams &k, int level) {
    return level < 0 ? k.a_bytes : (16 << level) * 128;
}

// ------------------------------------------------------------------------------------- producer
__device__ void sh_producer(const ShrinkParams &k, unsigned char *smem, const int *tables, int nruns, const ShWalk &wk,
                            int64_t nunits) {
    const LoraParams &p = k.p;
    const int lane = threadIdx.x & 31;
    const ShBars W = sh_bars(k, smem);
    const int cR = p.c * p.R;
    uint32_t it = 0, uc = 0;
    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
        Unit T;
        int r, part, c0, c1;
        if (!sh_unit(k, tables, nruns, wk, u, lane == 0, T, r, part, c0, c1)) continue;
        const int b = uc & 1;
        mbar_wait(&W.tok_empty[b], ((uc >> 1) & 1) ^ 1, p.status, kStatusTimeout);
        int *tok = W.tok + b * 128;
        for (int m = lane; m < 128; m += 32) {
            int t = -1;
            if (m < T.M) {
                t = p.permutation[T.p0 + m];
                if (t < 0 || t >= p.num_tokens) {
                    if (part == 0) atomicOr(p.status, CSGMV_STATUS_BAD_PERMUTATION);
                    t = -1;
                }
            }
            tok[m] = t;
        }
        __syncwarp();
        const int t0 = tok[0];
        bool mine = true;
        for (int m = lane; m < T.M; m += 32) mine = mine && tok[m] == t0 + m;
        const bool contig = __all_sync(0xffffffffu, mine) && t0 >= 0;
        if (lane == 0) {
            W.flag[b] = contig ? 1 : 0;
            mbar_arrive(&W.tok_full[b]);
        }
        const int tfill = t0 >= 0 ? t0 : 0;
        auto grow = [&](int mm) {
            const int t = mm < T.M ? tok[mm] : -1;
            return t >= 0 ? t : tfill;
        };
        const int n16 = (p.c * r + 15) / 16;  // 16-row boxes of A: rows [0, round16(c*r)) of the slot
        // a partial tile's x rows as one box of 64, 32, 16 or 8 rows (the
        // rest of the 128-row operand is stale and only feeds unused rows)
        const int xb = T.M > 64 ? -1 : (T.M > 32 ? 0 : (T.M > 16 ? 1 : (T.M > 8 ? 2 : 3)));
        const CUtensorMap *xmap = xb < 0 ? &k.tmX : &k.tmXp[xb];
        const uint32_t xbytes = contig ? (xb < 0 ? 128u : 64u >> xb) * 128u : 128u * 128u;
        for (int ci = c0; ci < c1; ci += k.chunks, ++it) {
            const int s = it % k.S;
            const int nch = min(k.chunks, c1 - ci);  // chunks in this stage
            // a whole stage of whole chunks: x (a full contiguous tile) and A
            // each as one 3-D box over the stage's chunks; A then brings
            // round16(c*R) rows (rows past the rank feed no output column)
            const bool full3 = k.use3d && nch == k.chunks;
            const bool x3 = full3 && contig && xb < 0;
            const int alev = sh_a3_level(k, n16);
            const uint32_t sbytes =
                (uint32_t)nch * (xbytes + (full3 ? (uint32_t)sh_a_stride(k, alev) : (uint32_t)n16 * 16 * 128));
            mbar_wait(&W.empty[s], ((it / k.S) & 1) ^ 1, p.status, kStatusTimeout);
            unsigned char *st = smem + k.o_ring + s * k.stage_bytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(&W.full[s], sbytes);
                if (x3) {
                    tma_load_3d(st, &k.tmX3, 0, t0, ci, &W.full[s]);
                } else if (contig) {
                    for (int j = 0; j < nch; ++j) tma_load_2d(st + j * 128 * 128, xmap, (ci + j) * 64, t0, &W.full[s]);
                }
                if (full3) {
                    tma_load_3d(st + k.a_off, alev < 0 ? &k.tmA3 : &k.tmA3s[alev], 0, T.w * cR, ci, &W.full[s]);
                } else {
                    // A rows [0, 16 * n16) of each chunk as boxes of 64, then 32, then 16 rows
                    for (int j = 0; j < nch; ++j)
                        for (int i = 0; i < n16;) {
                            const int nb = n16 - i >= 4 ? 4 : (n16 - i >= 2 ? 2 : 1);
                            const CUtensorMap *am = nb == 4 ? &k.tmA64 : (nb == 2 ? &k.tmA32 : &k.tmA);
                            tma_load_2d(st + k.a_off + j * k.a_bytes + i * 16 * 128, am, (ci + j) * 64, T.w * cR + 16 * i,
                                        &W.full[s]);
                            i += nb;
                        }
                }
            }
            if (!contig) {
                // lane l: tile rows 4l .. 4l+3 in one gather; rows past the tile
                // (or of an invalid token) read a valid row that is never used
                __syncwarp();  // after the byte count is posted
                const int m = 4 * lane;
                for (int j = 0; j < nch; ++j)
                    tma_gather4(st + j * 128 * 128 + m * 128, &k.tmXg, (ci + j) * 64, grow(m), grow(m + 1), grow(m + 2),
                                grow(m + 3), &W.full[s]);
            }
        }
        ++uc;
    }
}

// ------------------------------------------------------------------------------------- MMA issuer
__device__ void sh_mma(const ShrinkParams &k, unsigned char *smem, const int *tables, int nruns, const ShWalk &wk,
                       int64_t nunits, uint32_t tmem) {
    const LoraParams &p = k.p;
    const int lane = threadIdx.x & 31;
    const ShBars W = sh_bars(k, smem);
    uint32_t it = 0, uc = 0;
    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
        Unit T;
        int r, part, c0, c1;
        if (!sh_unit(k, tables, nruns, wk, u, false, T, r, part, c0, c1)) continue;
        const int b = uc & 1;
        mbar_wait(&W.acc_empty[b], ((uc >> 1) & 1) ^ 1, p.status, kStatusTimeout);
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, (p.c * r + 15) & ~15);
        const uint32_t d = tmem + (uint32_t)(b * kShAccCols);
        for (int ci = c0; ci < c1; ci += k.chunks, ++it) {
            const int s = it % k.S;
            const int nch = min(k.chunks, c1 - ci);
            mbar_wait(&W.full[s], (it / k.S) & 1, p.status, kStatusTimeout);
            tc_fence_after();
            if (lane == 0) {
                const uint32_t sa = smem_u32(smem + k.o_ring + s * k.stage_bytes);
                // A chunks as the producer laid them out: 3-D boxes of the
                // stage's level, else one tile of a_bytes per chunk
                const int astride = k.use3d && nch == k.chunks ? sh_a_stride(k, sh_a3_level(k, (p.c * r + 15) / 16))
                                                               : k.a_bytes;
                for (int j = 0; j < nch; ++j) {
                    const uint32_t xa = sa + j * 128 * 128;
                    const uint32_t aa = sa + k.a_off + j * astride;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc_mma_bf16(d, smem_desc_kmajor(xa + ks * 32, 128), smem_desc_kmajor(aa + ks * 32, 128), idesc,
                                    ci > c0 || j > 0 || ks > 0);
                }
                tc_commit(&W.empty[s]);
            }
            __syncwarp();
        }
        if (lane == 0) tc_commit(&W.acc_full[b]);
        __syncwarp();
        ++uc;
    }
    // the last stage releases land before the CTA (and its barriers) goes away
    for (uint32_t g = it > (uint32_t)k.S ? it - k.S : 0; g < it; ++g)
        mbar_wait(&W.empty[g % k.S], (g / k.S) & 1, p.status, kStatusTimeout);
}

// ------------------------------------------------------------------------------------- epilogue
// h row of token t: part `part` of the workspace planes, or h itself.
__device__ __forceinline__ void sh_store(const ShrinkParams &k, int part, int t, int col, float v) {
    const LoraParams &p = k.p;
    const int64_t o = (int64_t)part * k.plane + (int64_t)t * p.ldh + col;
    if (p.h_f32) reinterpret_cast<float *>(p.h)[o] = v;
    else reinterpret_cast<__nv_bfloat16 *>(p.h)[o] = __float2bfloat16_rn(v);
}

__device__ void sh_epilogue(const ShrinkParams &k, unsigned char *smem, const int *tables, int nruns, const ShWalk &wk,
                            int64_t nunits, uint32_t tmem) {
    const LoraParams &p = k.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;  // TMEM lanes (tile rows) 32q .. 32q+31
    const int row = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const ShBars W = sh_bars(k, smem);
    const int cR = p.c * p.R;
    uint32_t uc = 0;
    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
        Unit T;
        int r, part, c0, c1;
        if (!sh_unit(k, tables, nruns, wk, u, false, T, r, part, c0, c1)) {
            // h itself (one part): rows of rank-0 tokens are zero
            if (r == 0 && wk.P == 1 && row < T.M) {
                const int t = p.permutation[T.p0 + row];
                if (t >= 0 && t < p.num_tokens)
                    for (int col = 0; col < cR; ++col) sh_store(k, 0, t, col, 0.f);
            }
            continue;
        }
        const int b = uc & 1;
        mbar_wait(&W.tok_full[b], (uc >> 1) & 1, p.status, kStatusTimeout);
        const int trow = row < T.M ? W.tok[b * 128 + row] : -1;
        mbar_wait(&W.acc_full[b], (uc >> 1) & 1, p.status, kStatusTimeout);
        tc_fence_after();
        const int cr = p.c * r;
        const int64_t o = (int64_t)part * k.plane + (int64_t)trow * p.ldh;
        const bool vec = p.h_f32 && (o & 3) == 0;
        for (int cc = 0; cc < cr; cc += 32) {
            __syncwarp();  // tcgen05.ld is warp-wide
            float v[32];
            tmem_ld32(tmem + lane_base + (uint32_t)(b * kShAccCols + cc), v);
            if (trow < 0) continue;
            if (vec && cc + 32 <= cr) {
                float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.h) + o + cc);
#pragma unroll
                for (int e = 0; e < 8; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (cc + e < cr) sh_store(k, part, trow, cc + e, v[e]);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&W.acc_empty[b]);
        if (wk.P == 1 && trow >= 0)  // h itself: columns [c*r, c*R) are zero
            for (int col = cr; col < cR; ++col) sh_store(k, 0, trow, col, 0.f);
        __syncwarp();
        if (lane == 0) mbar_arrive(&W.tok_empty[b]);
        ++uc;
    }
}

__global__ void __launch_bounds__(kShThreads, 1) lora_stream_shrink_kernel(const __grid_constant__ ShrinkParams k) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const ShBars W = sh_bars(k, smem);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < k.S; ++i) {
            mbar_init(&W.full[i], 1);
            mbar_init(&W.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&W.acc_full[i], 1);
            mbar_init(&W.acc_empty[i], 4);
            mbar_init(&W.tok_full[i], 1);
            mbar_init(&W.tok_empty[i], 4);
        }
        fence_mbar_init();
        prefetch_tmap(&k.tmX);
        prefetch_tmap(&k.tmXg);
        for (int i = 0; i < 4; ++i) prefetch_tmap(&k.tmXp[i]);
        prefetch_tmap(&k.tmA);
        prefetch_tmap(&k.tmA32);
        prefetch_tmap(&k.tmA64);
    }
    if (warp == 1) {  // one warp owns the TMEM accumulators of the CTA
        tmem_alloc(W.tmem_slot, 2 * kShAccCols);
        tmem_relinquish();
    }
    tc_fence_before();
    int nruns = 0;
    int *tables = reinterpret_cast<int *>(smem + k.o_run);
    const int ntiles = build_run_table_raw<128, true>(k.p, k.max_segments, k.runcap, tables, &nruns);  // ends with __syncthreads
    tc_fence_after();
    const uint32_t tmem = *W.tmem_slot;
    const ShWalk wk = sh_walk(ntiles, (int)((k.p.K + 63) / 64), k.max_parts, gridDim.x);
    if (k.parts_out && blockIdx.x == 0 && threadIdx.x == 0) *k.parts_out = wk.P;  // for the expand
    const int64_t nunits = (int64_t)ntiles * wk.P;
    if (warp == 0) sh_producer(k, smem, tables, nruns, wk, nunits);
    else if (warp == 1) sh_mma(k, smem, tables, nruns, wk, nunits, tmem);
    else sh_epilogue(k, smem, tables, nruns, wk, nunits, tmem);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * kShAccCols);
    }
}

}  // namespace

const void *lora_kernel_sshrink() { return reinterpret_cast<const void *>(lora_stream_shrink_kernel); }

}  // namespace csgmv
